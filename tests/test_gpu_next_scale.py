"""GPU parity of the next layer's activation scale taken in the GEMM epilogue
(frt_gemm_fp8_next_scale / frt_gemm_bf16_next_scale).

Reading: the scale is that of the layer's own stored bf16 output, so it must
equal, bit for bit, the oracle's per-tensor OCP scale of out[:, :scale_cols]
(amax / 448, NaN ignored, 1 for an all-zero block), and the encode pass with
it (frt_quantize_e4m3 with that static scale) must give the oracle's dynamic
quantize of the same block byte for byte.  The bf16 output itself must equal
the plain GEMM's bit for bit (taking the scale changes nothing it stores);
the plain GEMM is checked against the oracle GEMM by the other GEMM tests.
Shapes cover every launch-plan kind: CTA pairs with 256- and 128-wide tiles
(persistent, split-K through the workspace and inside a cluster), small-M
tiles with a cluster split-K and without, row tails, the GeGLU epilogue, and
a strided next-layer view (scale_cols smaller than the output)."""
import numpy as np
import pytest
import torch

import synth
from bf16_gemm_vla_gb300 import frt, layers
from helpers import bf16_dev
from oracle import e4m3, quantize

pytestmark = pytest.mark.gpu

# (M, K, N, act_cols, scale_cols, geglu)
SHAPES = [
    (768, 2048, 2560, 0, 2048, False),        # pairs, 256 x 128 tiles; the O layer's view
    (768, 2048, 16384, 0, 16384, False),      # pairs, 256 x 256, persistent
    (768, 2048, 32768, 16384, 16384, False),  # merged gate/up, GELU on the gate half
    (768, 16384, 2048, 0, 2048, False),       # pairs, split-K through the workspace
    (300, 1024, 512, 0, 504, False),          # row tail inside a pair tile
    (768, 1024, 4096, 0, 2048, True),         # GeGLU on pairs: out is N / 2 wide
    (50, 1024, 4096, 0, 4096, False),         # small M, cluster split-K
    (50, 1024, 2560, 0, 2048, False),         # small M, strided view
    (50, 4096, 1024, 0, 1024, False),         # small M, deep split
    (17, 512, 256, 256, 200, False),          # small M, GELU on every column
    (50, 1024, 8192, 0, 4096, True),          # small M GeGLU
    (40, 256, 36864, 0, 36864, False),        # small M, more tiles than SMs: no split
    (1, 512, 1024, 0, 1024, False),
]


def _plain_and_inputs(kind, M, K, N, act_cols, geglu, seed):
    lay = synth.layer(np.random.default_rng(seed), M, K, N, act_cols=act_cols, outlier_frac=0.01)
    w = torch.from_numpy(lay["w_f32"]).cuda()
    b = torch.from_numpy(lay["bias"]).cuda()
    pw = layers.prepare_fp8(w, b) if kind == "e4m3" else layers.prepare_bf16(w, b)
    x = bf16_dev(lay["a_bf16"])
    ws = frt.gemm_workspace(M, N, K, kind, x.device)
    ws = False if ws is None else ws
    if kind == "e4m3":
        qa, sa = frt.frt_quantize_e4m3(x, frt.PER_TENSOR, frt.OCP)
        plain = frt.frt_gemm_fp8(qa, sa, pw.packed, pw.w_scale, N, bias=b, act_cols=act_cols,
                                 workspace=ws, geglu=geglu)

        def run(**kw):
            return frt.frt_gemm_fp8_next_scale(qa, sa, pw.packed, pw.w_scale, N, bias=b,
                                               act_cols=act_cols, workspace=ws, geglu=geglu, **kw)
    else:
        plain = frt.frt_gemm_bf16(x, pw.packed, N, bias=b, act_cols=act_cols, workspace=ws,
                                  geglu=geglu)

        def run(**kw):
            return frt.frt_gemm_bf16_next_scale(x, pw.packed, N, bias=b, act_cols=act_cols,
                                                workspace=ws, geglu=geglu, **kw)
    return plain, run


@pytest.mark.parametrize("kind", ["e4m3", "bf16"])
@pytest.mark.parametrize("M,K,N,act_cols,scale_cols,geglu", SHAPES)
def test_next_scale_is_the_oracle_scale_of_the_output(kind, M, K, N, act_cols, scale_cols, geglu):
    plain, run = _plain_and_inputs(kind, M, K, N, act_cols, geglu, seed=M * 31 + N + K)
    hdr = frt.next_scale_workspace("cuda")
    for _ in range(2):  # twice through the same header
        out, s = run(scale_cols=scale_cols, scale_workspace=hdr)
        torch.cuda.synchronize()
        frt.check_device_status()
        assert out.shape == (M, N // 2 if geglu else N)
        assert torch.equal(out, plain)
        x = out[:, :scale_cols].float().cpu().numpy()
        qo, so = quantize.quantize_e4m3(x, quantize.PER_TENSOR, e4m3.OCP)
        assert s.cpu().numpy()[0] == so
        # the encode pass with the taken scale: the dynamic quantize's bytes
        q, s2 = frt.frt_quantize_e4m3(out[:, :scale_cols], frt.PER_TENSOR, frt.OCP,
                                      static_scale=s)
        np.testing.assert_array_equal(q.cpu().numpy(), qo)
        assert s2.cpu().numpy()[0] == so
        h = hdr.view(torch.int32)[:8].cpu().numpy()
        assert h[0] == 0 and h[4] == 0  # arrivals and running maximum back at zero


def test_next_scale_of_zero_output_is_one():
    M, K, N = 64, 256, 512
    pw = layers.prepare_bf16(torch.zeros((K, N), device="cuda"), None)
    x = torch.ones((M, K), dtype=torch.bfloat16, device="cuda")
    out, s = frt.frt_gemm_bf16_next_scale(x, pw.packed, N)
    torch.cuda.synchronize()
    assert float(s.cpu()[0]) == 1.0 and bool((out == 0).all())


def test_next_scale_rejects_bad_arguments():
    M, K, N = 64, 256, 512
    pw = layers.prepare_bf16(torch.zeros((K, N), device="cuda"), None)
    x = torch.ones((M, K), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(frt.FrtError, match="UNSUPPORTED_SHAPE"):
        frt.frt_gemm_bf16_next_scale(x, pw.packed, N, scale_cols=20)  # not a multiple of 8
    with pytest.raises(frt.FrtError, match="INVALID_ARG"):
        frt.frt_gemm_bf16_next_scale(x, pw.packed, N, scale_cols=1024)  # wider than the output
    with pytest.raises(frt.FrtError, match="WORKSPACE_TOO_SMALL"):
        frt.frt_gemm_bf16_next_scale(x, pw.packed, N, scale_workspace=torch.zeros(
            (128,), dtype=torch.uint8, device="cuda"))
