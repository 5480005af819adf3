"""GPU parity of weight packing (bit-exact) and of the FP8 / BF16 GEMMs
(per-element tolerance |gpu - oracle| <= 2^-7 |oracle| + 1e-5 sum|a w|)."""
import numpy as np
import pytest
import torch

import synth
from bf16_gemm_vla_gb300 import frt, layers
from helpers import assert_gemm_close, bf16_dev
from oracle import bf16 as obf16
from oracle import convert, e4m3, gemm, pack, quantize

pytestmark = pytest.mark.gpu


# ---------------------------------------------------------------- pack

@pytest.mark.parametrize("K,N", [(512, 256), (96, 200), (300, 130), (4096, 1024), (32, 16)])
def test_pack_e4m3(K, N):
    g = np.random.default_rng(K * 7 + N)
    w = g.integers(0, 256, (K, N), dtype=np.uint8)
    p = frt.frt_pack_weights(torch.from_numpy(w).cuda(), "e4m3")
    np.testing.assert_array_equal(p.cpu().numpy(), pack.pack(w, "e4m3"))


@pytest.mark.parametrize("K,N", [(512, 256), (96, 200), (80, 136), (1024, 2048)])
def test_pack_bf16_from_fp32_and_bf16(K, N):
    g = np.random.default_rng(K + 3 * N)
    w = np.float32(g.standard_normal((K, N)))
    p = frt.frt_pack_weights(torch.from_numpy(w).cuda(), "bf16")
    np.testing.assert_array_equal(p.cpu().numpy(), pack.pack_fp32_as_bf16(w))
    bits = obf16.f32_to_bf16_bits(w)
    p2 = frt.frt_pack_weights(bf16_dev(bits), "bf16")
    np.testing.assert_array_equal(p2.cpu().numpy(), pack.pack(bits, "bf16"))


def test_pack_strided_source():
    g = np.random.default_rng(1)
    big = g.integers(0, 256, (200, 320), dtype=np.uint8)
    d = torch.from_numpy(big).cuda()[:, :272]
    p = frt.frt_pack_weights(d, "e4m3")
    np.testing.assert_array_equal(p.cpu().numpy(), pack.pack(big[:, :272], "e4m3"))


# ---------------------------------------------------------------- GEMM helpers

def fp8_layer(lay, import_fnuz=False, act_cols=None, bias=True):
    """Runs the FP8 path of one layer on the GPU and the oracle; checks the
    quantized bytes and scales bit-exactly on the way."""
    M, K, N = lay["M"], lay["K"], lay["N"]
    act_cols = lay["act_cols"] if act_cols is None else act_cols
    a_dev = bf16_dev(lay["a_bf16"])
    a_f32 = synth.bf16_bits_as_f32(lay["a_bf16"])
    w_dev = torch.from_numpy(lay["w_f32"]).cuda()
    b_dev = torch.from_numpy(lay["bias"]).cuda() if bias else None
    # activation quantize (OCP per tensor)
    qa, sa = frt.frt_quantize_e4m3(a_dev, frt.PER_TENSOR, frt.OCP)
    qa_o, sa_o = quantize.quantize_e4m3(a_f32, quantize.PER_TENSOR, e4m3.OCP)
    assert sa.cpu().numpy()[0] == sa_o
    np.testing.assert_array_equal(qa.cpu().numpy(), qa_o)
    # weight quantize per channel (optionally FNUZ import, then re-encode)
    fmt, ofmt = (frt.FNUZ, e4m3.FNUZ) if import_fnuz else (frt.OCP, e4m3.OCP)
    qw, sw = frt.frt_quantize_e4m3(w_dev, frt.PER_COL, fmt)
    qw_o, sw_o = quantize.quantize_e4m3(lay["w_f32"], quantize.PER_COL, ofmt)
    np.testing.assert_array_equal(sw.cpu().numpy(), sw_o)
    np.testing.assert_array_equal(qw.cpu().numpy(), qw_o)
    if import_fnuz:
        frt.frt_fnuz_to_ocp(qw.view(-1), out=qw.view(-1))
        qw_o = convert.fnuz_to_ocp(qw_o)
        np.testing.assert_array_equal(qw.cpu().numpy(), qw_o)
    wp = frt.frt_pack_weights(qw, "e4m3")
    torch.cuda.synchronize()  # packed weights are load-time data
    out = frt.frt_gemm_fp8(qa, sa, wp, sw, N, bias=b_dev, act_cols=act_cols)
    frt.check_device_status()
    y, sumabs = gemm.gemm_fp8(qa_o, e4m3.OCP, sa_o, qw_o, e4m3.OCP, sw_o,
                              lay["bias"] if bias else None, act_cols)
    assert_gemm_close(out, y, sumabs, "fp8 M=%d K=%d N=%d" % (M, K, N))
    return out


def bf16_layer(lay, act_cols=None, bias=True, w_scale=None):
    M, K, N = lay["M"], lay["K"], lay["N"]
    act_cols = lay["act_cols"] if act_cols is None else act_cols
    a_dev = bf16_dev(lay["a_bf16"])
    a_f32 = synth.bf16_bits_as_f32(lay["a_bf16"])
    wp = frt.frt_pack_weights(torch.from_numpy(lay["w_f32"]).cuda(), "bf16")
    b_dev = torch.from_numpy(lay["bias"]).cuda() if bias else None
    ws_dev = None if w_scale is None else torch.from_numpy(w_scale).cuda()
    torch.cuda.synchronize()  # packed weights are load-time data
    out = frt.frt_gemm_bf16(a_dev, wp, N, w_scale=ws_dev, bias=b_dev, act_cols=act_cols)
    frt.check_device_status()
    w_bf = obf16.round_to_bf16(lay["w_f32"])
    y, sumabs = gemm.gemm_bf16(a_f32, w_bf, w_scale, lay["bias"] if bias else None, act_cols)
    assert_gemm_close(out, y, sumabs, "bf16 M=%d K=%d N=%d" % (M, K, N))
    return out


def rand_layer(M, K, N, act_cols=0, seed=0, outliers=0.0):
    return synth.layer(np.random.default_rng(seed), M, K, N, act_cols=act_cols,
                       outlier_frac=outliers)


# ---------------------------------------------------------------- tiny config

def test_tiny_config_fp8_with_fnuz_import():
    fp8_layer(synth.tiny(), import_fnuz=True)


def test_tiny_config_bf16():
    bf16_layer(synth.tiny())


def test_integer_gemm_exact():
    # small integers are exact in E4M3 and bf16; with unit scales every
    # output is an integer of magnitude <= 256, exact in bf16
    g = np.random.default_rng(3)
    for M, K, N in ((16, 64, 128), (200, 64, 256), (50, 64, 1024)):
        a = g.integers(-2, 3, (M, K)).astype(np.float32)
        w = g.integers(-2, 3, (K, N)).astype(np.float32)
        exact = a.astype(np.int64) @ w.astype(np.int64)
        one = torch.ones(1, dtype=torch.float32, device="cuda")
        qa, _ = frt.frt_quantize_e4m3(torch.from_numpy(a).cuda(), frt.PER_TENSOR, frt.OCP,
                                      static_scale=one)
        qw, _ = frt.frt_quantize_e4m3(torch.from_numpy(w).cuda(), frt.PER_COL, frt.OCP,
                                      static_scale=torch.ones(N, device="cuda"))
        wp = frt.frt_pack_weights(qw, "e4m3")
        torch.cuda.synchronize()  # packed weights are load-time data
        out = frt.frt_gemm_fp8(qa, one, wp, torch.ones(N, device="cuda"), N)
        np.testing.assert_array_equal(out.float().cpu().numpy(), exact.astype(np.float32))
        wb = frt.frt_pack_weights(torch.from_numpy(w).cuda(), "bf16")
        torch.cuda.synchronize()
        out = frt.frt_gemm_bf16(torch.from_numpy(a).cuda().to(torch.bfloat16), wb, N)
        np.testing.assert_array_equal(out.float().cpu().numpy(), exact.astype(np.float32))
        frt.check_device_status()


# ---------------------------------------------------------------- shapes: tails, modes, splits

SMALL_M = [1, 7, 32, 33, 50, 64, 65, 100, 128]
LARGE_M = [129, 200, 256, 300]


@pytest.mark.parametrize("M", SMALL_M + LARGE_M)
def test_fp8_row_tails(M):
    fp8_layer(rand_layer(M, 1024, 272, seed=M))


@pytest.mark.parametrize("M", SMALL_M + LARGE_M)
def test_bf16_row_tails(M):
    bf16_layer(rand_layer(M, 512, 400, seed=M))


@pytest.mark.parametrize("M,K,N", [(50, 96, 144), (50, 4096, 1024), (16, 8192, 128),
                                   (300, 16384, 256), (768, 2048, 2560), (130, 96, 16),
                                   (64, 2048, 8192), (1, 4096, 4096), (300, 8192, 384),
                                   (520, 1024, 4352), (300, 1152, 256), (768, 1152, 2560)])
def test_fp8_shapes_and_splits(M, K, N):
    fp8_layer(rand_layer(M, K, N, seed=K + N))


@pytest.mark.parametrize("M,K,N", [(50, 112, 144), (50, 4096, 1024), (16, 8192, 128),
                                   (300, 8192, 256), (768, 2048, 2560), (130, 48, 16),
                                   (1, 4096, 4096), (300, 8192, 384), (520, 1024, 4352),
                                   (300, 1088, 256), (768, 1088, 2560)])
def test_bf16_shapes_and_splits(M, K, N):
    bf16_layer(rand_layer(M, K, N, seed=K + N))


def test_gelu_on_leading_columns_only():
    # merged gate/up: GELU on the gate half [0, N/2)
    fp8_layer(rand_layer(50, 1024, 8192, act_cols=4096, seed=1))
    fp8_layer(rand_layer(768, 2048, 4096, act_cols=2048, seed=2))
    bf16_layer(rand_layer(50, 1024, 8192, act_cols=4096, seed=3))
    bf16_layer(rand_layer(256, 512, 1024, act_cols=512, seed=4))
    fp8_layer(rand_layer(40, 256, 160, act_cols=48, seed=5))


def test_no_bias_and_bf16_channel_scale():
    fp8_layer(rand_layer(50, 1024, 512, seed=6), bias=False)
    g = np.random.default_rng(7)
    bf16_layer(rand_layer(50, 1024, 512, seed=7), w_scale=np.float32(g.uniform(0.5, 2, 512)))
    bf16_layer(rand_layer(300, 1024, 512, seed=8), bias=False,
               w_scale=np.float32(g.uniform(0.5, 2, 512)))


def test_strided_activations_and_output():
    lay = rand_layer(50, 1024, 512, seed=9)
    big = bf16_dev(synth.to_bf16_bits(np.random.default_rng(9).standard_normal((50, 1536))))
    a = big[:, :1024]
    a_f32 = big.float().cpu().numpy()[:, :1024]
    wp = frt.frt_pack_weights(torch.from_numpy(lay["w_f32"]).cuda(), "bf16")
    out_big = torch.zeros((50, 640), dtype=torch.bfloat16, device="cuda")
    torch.cuda.synchronize()
    frt.frt_gemm_bf16(a, wp, 512, bias=torch.from_numpy(lay["bias"]).cuda(),
                      out=out_big[:, :512])
    y, sumabs = gemm.gemm_bf16(a_f32, obf16.round_to_bf16(lay["w_f32"]), None, lay["bias"], 0)
    assert_gemm_close(out_big[:, :512], y, sumabs, "strided")
    assert float(out_big[:, 512:].abs().max()) == 0.0  # nothing written past N
    qa, sa = frt.frt_quantize_e4m3(a, frt.PER_TENSOR, frt.OCP)
    pw = layers.prepare_fp8(torch.from_numpy(lay["w_f32"]).cuda())
    big_q = torch.zeros((50, 1152), dtype=torch.uint8, device="cuda")
    big_q[:, :1024] = qa
    out = frt.frt_gemm_fp8(big_q[:, :1024], sa, pw.packed, pw.w_scale, 512)
    ref = frt.frt_gemm_fp8(qa, sa, pw.packed, pw.w_scale, 512)
    assert torch.equal(out, ref)


# ---------------------------------------------------------------- the decoder and encoder configs

@pytest.mark.parametrize("li", range(4))
def test_decoder_config_fp8_and_bf16(li):
    lay = synth.decoder(seed=0)[li]
    fp8_layer(lay)
    bf16_layer(lay)


@pytest.mark.parametrize("li", range(3))
def test_encoder_config_fp8_and_bf16(li):
    lay = synth.encoder(seed=0)[li]
    fp8_layer(lay)
    bf16_layer(lay)


def test_gemm_is_deterministic():
    lay = synth.decoder(seed=0)[3]  # K = 4096: split-K across a cluster
    o1 = fp8_layer(lay)
    o2 = fp8_layer(lay)
    assert torch.equal(o1, o2)


@pytest.mark.parametrize("M", synth.SWEEP_M)
def test_sweep_shapes(M):
    # sweep (i): K = N = 4096 at every M of the sweep, both precisions
    lay = synth.sweep_gemm(M, seed=M)
    fp8_layer(lay)
    bf16_layer(lay)


# ---------------------------------------------------------------- split-K through the workspace

@pytest.mark.parametrize("M,K,N", [(768, 16384, 2048), (300, 16384, 256), (520, 8192, 384)])
def test_split_k_workspace_and_cluster_paths(M, K, N):
    # large-M shapes whose K is split: with a workspace the partial sums meet
    # in global memory, without one inside a cluster; both match the oracle,
    # each is bit-identical from call to call, and the workspace's counters
    # are back at zero after every call (a second input through the same
    # workspace is not mixed with the first)
    nb = frt.frt_gemm_workspace_bytes(M, N, K, "e4m3")
    assert nb > 0
    ws = torch.zeros((nb,), dtype=torch.uint8, device="cuda")
    for seed in (K + N, K + N + 1):
        lay = rand_layer(M, K, N, seed=seed)
        a_dev = bf16_dev(lay["a_bf16"])
        qa, sa = frt.frt_quantize_e4m3(a_dev, frt.PER_TENSOR, frt.OCP)
        pw = layers.prepare_fp8(torch.from_numpy(lay["w_f32"]).cuda(),
                                torch.from_numpy(lay["bias"]).cuda())
        outs = {}
        # a workspace too small for any global split: the cluster path
        tiny = torch.zeros((256,), dtype=torch.uint8, device="cuda")
        for name, w in (("workspace", ws), ("cluster", False), ("too_small", tiny)):
            o1 = frt.frt_gemm_fp8(qa, sa, pw.packed, pw.w_scale, N, bias=pw.bias, workspace=w)
            o2 = frt.frt_gemm_fp8(qa, sa, pw.packed, pw.w_scale, N, bias=pw.bias, workspace=w)
            frt.check_device_status()
            assert torch.equal(o1, o2), name
            outs[name] = o1
        assert int(ws[:256].sum()) == 0
        assert torch.equal(outs["too_small"], outs["cluster"])
        qa_o, sa_o = quantize.quantize_e4m3(synth.bf16_bits_as_f32(lay["a_bf16"]),
                                            quantize.PER_TENSOR, e4m3.OCP)
        qw_o, sw_o = quantize.quantize_e4m3(lay["w_f32"], quantize.PER_COL, e4m3.OCP)
        y, sumabs = gemm.gemm_fp8(qa_o, e4m3.OCP, sa_o, qw_o, e4m3.OCP, sw_o, lay["bias"], 0)
        for name, o in outs.items():
            assert_gemm_close(o, y, sumabs, "%s M=%d K=%d N=%d" % (name, M, K, N))


def test_split_k_workspace_bf16():
    M, K, N = 768, 16384, 2048
    lay = rand_layer(M, K, N, seed=5)
    nb = frt.frt_gemm_workspace_bytes(M, N, K, "bf16")
    assert nb > 0
    ws = torch.zeros((nb,), dtype=torch.uint8, device="cuda")
    a_dev = bf16_dev(lay["a_bf16"])
    wp = frt.frt_pack_weights(torch.from_numpy(lay["w_f32"]).cuda(), "bf16")
    b_dev = torch.from_numpy(lay["bias"]).cuda()
    torch.cuda.synchronize()
    o1 = frt.frt_gemm_bf16(a_dev, wp, N, bias=b_dev, workspace=ws)
    o2 = frt.frt_gemm_bf16(a_dev, wp, N, bias=b_dev, workspace=ws)
    frt.check_device_status()
    assert torch.equal(o1, o2)
    assert int(ws[:256].sum()) == 0
    y, sumabs = gemm.gemm_bf16(synth.bf16_bits_as_f32(lay["a_bf16"]),
                               obf16.round_to_bf16(lay["w_f32"]), None, lay["bias"], 0)
    assert_gemm_close(o1, y, sumabs, "bf16 workspace split")


# ---------------------------------------------------------------- plans

PLAN_SHAPES = [(768, 2048, 2560), (768, 2048, 16384), (768, 16384, 2048), (300, 8192, 384),
               (520, 1024, 4352), (300, 16384, 256), (768, 1152, 2560), (512, 4096, 4096)]


def test_plans_cover_every_pair_kind():
    # the large-M shapes of the parity tests take every CTA-pair plan kind:
    # persistent (no split), K split across a cluster, K split through the
    # workspace; the plan is a pure function of the shape
    kinds = set()
    for M, K, N in PLAN_SHAPES:
        for kind in ("e4m3", "bf16"):
            pl = frt.frt_gemm_describe(M, N, K, kind)
            assert pl == frt.frt_gemm_describe(M, N, K, kind)
            assert pl["kind"] == "pair" and pl["cluster"][0] == 2
            assert pl["grid"][0] % 2 == 0
            if pl["global"]:
                assert pl["cluster"][2] == 1 and pl["grid"][2] == pl["splits"] > 1
            else:
                assert pl["cluster"][2] == pl["splits"]
            kinds.add((pl["global"], pl["splits"] > 1))
    assert kinds == {(0, False), (0, True), (1, True)}
    # without a workspace no plan splits through it
    M, N, K = 768, 2048, 16384
    assert frt.frt_gemm_describe(M, N, K, "e4m3")["global"] == 1
    assert frt.frt_gemm_describe(M, N, K, "e4m3", 0)["global"] == 0
    small = frt.frt_gemm_describe(50, 1024, 4096, "e4m3")
    assert small["kind"] == "swap" and small["cluster"][0] == 1
    with pytest.raises(frt.FrtError):
        frt.frt_gemm_describe(50, 1000, 4096, "e4m3")  # N % 16 != 0


@pytest.mark.parametrize("M,K,N", PLAN_SHAPES)
def test_plan_shapes_fp8_and_bf16(M, K, N):
    lay = rand_layer(M, K, N, seed=M + K + N)
    fp8_layer(lay)
    bf16_layer(lay)


# ---------------------------------------------------------------- fused GeGLU (merged gate/up)

def geglu_oracle(lay, qa_o, sa_o, qw_o, sw_o, kind):
    if kind == "e4m3":
        y, sumabs = gemm.gemm_fp8(qa_o, e4m3.OCP, sa_o, qw_o, e4m3.OCP, sw_o, lay["bias"], 0)
    else:
        y, sumabs = gemm.gemm_bf16(synth.bf16_bits_as_f32(lay["a_bf16"]),
                                   obf16.round_to_bf16(lay["w_f32"]), None, lay["bias"], 0)
    return gemm.geglu(y, sumabs)


@pytest.mark.parametrize("M,K,F", [(300, 1024, 512), (257, 256, 128), (520, 1152, 1280),
                                   (768, 2048, 16384), (50, 1024, 4096), (16, 256, 128),
                                   (128, 4096, 1024), (1, 512, 256), (64, 2048, 640)])
@pytest.mark.parametrize("kind", ["e4m3", "bf16"])
def test_geglu_fused_epilogue(M, K, F, kind):
    # one GEMM over [W_gate, W_up] (2F channels, gate first) whose epilogue
    # writes gelu(gate) * up: F output columns
    lay = rand_layer(M, K, 2 * F, seed=M + K + F)
    a_dev = bf16_dev(lay["a_bf16"])
    b_dev = torch.from_numpy(lay["bias"]).cuda()
    w_dev = torch.from_numpy(lay["w_f32"]).cuda()
    qa_o = sa_o = qw_o = sw_o = None
    if kind == "e4m3":
        qa, sa = frt.frt_quantize_e4m3(a_dev, frt.PER_TENSOR, frt.OCP)
        pw = layers.prepare_fp8(w_dev, b_dev)
        out = frt.frt_gemm_fp8(qa, sa, pw.packed, pw.w_scale, 2 * F, bias=b_dev, geglu=True)
        qa_o, sa_o = quantize.quantize_e4m3(synth.bf16_bits_as_f32(lay["a_bf16"]),
                                            quantize.PER_TENSOR, e4m3.OCP)
        qw_o, sw_o = quantize.quantize_e4m3(lay["w_f32"], quantize.PER_COL, e4m3.OCP)
    else:
        wp = frt.frt_pack_weights(w_dev, "bf16")
        torch.cuda.synchronize()
        out = frt.frt_gemm_bf16(a_dev, wp, 2 * F, bias=b_dev, geglu=True)
    frt.check_device_status()
    assert tuple(out.shape) == (M, F)
    h, prop = geglu_oracle(lay, qa_o, sa_o, qw_o, sw_o, kind)
    assert_gemm_close(out, h, prop, "geglu %s M=%d K=%d F=%d" % (kind, M, K, F))


def test_geglu_rejects_unsupported_shapes():
    a = torch.zeros((300, 256), dtype=torch.bfloat16, device="cuda")
    wp = frt.frt_pack_weights(torch.zeros((256, 384), device="cuda"), "bf16")
    torch.cuda.synchronize()
    with pytest.raises(frt.FrtError):
        frt.frt_gemm_bf16(a, wp, 384, geglu=True)  # N % 256 != 0
