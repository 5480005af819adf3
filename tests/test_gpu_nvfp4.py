"""GPU parity of the NVFP4 path (frt_quantize_nvfp4, frt_gemm_nvfp4) against
the oracle (oracle/nvfp4.py): codes, tiled block scales and the tensor scale
bit for bit; the GEMM within the GEMM tolerance
|gpu - ref| <= 2^-7 |ref| + 1e-5 g_a g_w sum_k |a w| per element, on the
oracle's own quantization of the same inputs."""
import numpy as np
import pytest
import torch

from bf16_gemm_vla_gb300 import frt, layers
from helpers import assert_gemm_close
from oracle import nvfp4

pytestmark = pytest.mark.gpu


def _x(rng, rows, cols, spread=10.0):
    return (rng.standard_normal((rows, cols)) * rng.uniform(1.0 / spread, spread, (rows, 1))
            ).astype(np.float32)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("rows,cols", [(1, 64), (200, 512), (128, 256), (768, 2048), (33, 4096)])
def test_quantize_activations(dtype, rows, cols):
    rng = np.random.default_rng(rows * 7 + cols)
    xd = torch.from_numpy(_x(rng, rows, cols)).cuda().to(dtype)
    q, sf, g = frt.frt_quantize_nvfp4(xd)
    qo, sbo, go = nvfp4.quantize(xd.float().cpu().numpy())
    assert g.cpu().numpy()[0] == go
    np.testing.assert_array_equal(q.cpu().numpy(), nvfp4.pack_nibbles(qo))
    np.testing.assert_array_equal(sf.cpu().numpy(), nvfp4.tile_scales(sbo))


@pytest.mark.parametrize("K,N", [(64, 16), (512, 384), (256, 200), (2048, 2560)])
def test_quantize_weights_down_the_columns(K, N):
    rng = np.random.default_rng(K + N)
    w = (rng.standard_normal((K, N)) * 0.02).astype(np.float32)
    q, sf, g = frt.frt_quantize_nvfp4(torch.from_numpy(w).cuda(), blocks_along_rows=True)
    qo, sbo, go = nvfp4.quantize(w.T.copy())
    assert g.cpu().numpy()[0] == go
    np.testing.assert_array_equal(q.cpu().numpy(), nvfp4.pack_nibbles(qo).T)
    np.testing.assert_array_equal(sf.cpu().numpy(), nvfp4.tile_scales(sbo))


def test_quantize_static_scale_specials_and_workspace_reuse():
    rng = np.random.default_rng(11)
    x = _x(rng, 64, 256)
    x[0, :16] = 0.0                       # an all-zero block: scale 0, codes 0
    x[1, 3] = -1e-30                      # a tiny negative value: -0
    x[2, 5] = np.nan                      # NaN: +0, ignored by the maxima
    x[3, 7] = 1e6                         # a block whose scale saturates at 448
    ws = frt.nvfp4_workspace("cuda")
    for static in (None, 0.004):
        for _ in range(2):  # the workspace is left zero by every call
            st = None if static is None else torch.tensor([static], device="cuda")
            q, sf, g = frt.frt_quantize_nvfp4(torch.from_numpy(x).cuda(), static_scale=st,
                                              workspace=ws)
            qo, sbo, go = nvfp4.quantize(x, g=static)
            assert g.cpu().numpy()[0] == go
            np.testing.assert_array_equal(q.cpu().numpy(), nvfp4.pack_nibbles(qo))
            np.testing.assert_array_equal(sf.cpu().numpy(), nvfp4.tile_scales(sbo))
            assert not ws.any()
    q, sf, g = frt.frt_quantize_nvfp4(torch.zeros((16, 128), device="cuda"))
    assert g.item() == 1.0 and not q.any() and not sf.any()


def _gemm_case(M, N, K, act_cols, bias=True, seed=0, cols=None):
    rng = np.random.default_rng(seed)
    a = _x(rng, M, K, 4.0)
    w = (rng.standard_normal((K, N)) * 0.02 * rng.uniform(0.2, 3, (1, N))).astype(np.float32)
    b = (rng.standard_normal(N) * 0.1).astype(np.float32) if bias else None
    ad = torch.from_numpy(a).cuda().to(torch.bfloat16)
    qa, sfa, ga = frt.frt_quantize_nvfp4(ad)
    pw = layers.prepare_nvfp4(torch.from_numpy(w).cuda(),
                              torch.from_numpy(b).cuda() if bias else None)
    out = frt.frt_gemm_nvfp4(qa, sfa, ga, pw.packed, pw.sf, pw.g, N, bias=pw.bias,
                             act_cols=act_cols)
    torch.cuda.synchronize()
    frt.check_device_status()
    qao, sao, gao = nvfp4.quantize(ad.float().cpu().numpy())
    cols = slice(None) if cols is None else cols
    # (the weight's tensor scale is that of the whole weight; a column sample
    # is quantized with it, so its codes and block scales are the full ones)
    qwo, swo, gwo = nvfp4.quantize(w.T[cols].copy(), g=nvfp4.tensor_scale(w))
    ref, sumabs = nvfp4.gemm(qao, sao, gao, qwo, swo, gwo, None if b is None else b[cols],
                             act_cols=act_cols)
    return out.float().cpu().numpy()[:, cols], ref, sumabs


@pytest.mark.parametrize("M,N,K,act_cols,bias", [
    (128, 128, 256, 0, True),      # one tile, one k-block
    (200, 384, 512, 100, True),    # row tail, GELU on the first 100 columns
    (1, 16, 256, 16, False),       # one row, the narrowest N, no bias
    (300, 272, 1024, 0, True),     # N tail inside a 128-channel tile
    (768, 2560, 2048, 0, True),    # the encoder's QKV shape
    (256, 19456, 256, 9000, True), # more tiles than SMs, the GELU boundary inside a tile
    (300, 25744, 256, 12000, True),  # 256-channel pair tiles with row and channel tails
])
def test_gemm(M, N, K, act_cols, bias):
    y, ref, sumabs = _gemm_case(M, N, K, act_cols, bias, seed=M + N + K)
    assert_gemm_close(y, ref, sumabs, "nvfp4 %dx%dx%d" % (M, N, K))


def test_gemm_encoder_ffn_full_size():
    # the encoder FFN at full size: down 16384 -> 2048 in full, and the merged
    # gate/up 2048 -> 2 x 16384 (GELU on the gate half) on its first 1024
    # output channels (the oracle's decoded weight would take 0.5 GB)
    y, ref, sumabs = _gemm_case(768, 2048, 16384, 0, True, seed=5)
    assert_gemm_close(y, ref, sumabs, "nvfp4 down")
    y, ref, sumabs = _gemm_case(768, 32768, 2048, 16384, True, seed=6, cols=slice(0, 1024))
    assert_gemm_close(y, ref, sumabs, "nvfp4 gate/up")


def test_gemm_rejects_unsupported_shapes():
    qa = torch.zeros((64, 96), dtype=torch.uint8, device="cuda")  # K = 192: not a multiple of 256
    sf = torch.zeros((frt.frt_nvfp4_scale_bytes(128, 256),), dtype=torch.uint8, device="cuda")
    w = torch.zeros((16384,), dtype=torch.uint8, device="cuda")
    with pytest.raises(frt.FrtError, match="UNSUPPORTED_SHAPE"):
        frt.frt_gemm_nvfp4(qa, sf, None, w, sf, None, 128)
