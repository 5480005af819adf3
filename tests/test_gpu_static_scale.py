"""Calibrated (frozen) activation scales: ``Linear.calibrate`` keeps the
largest dynamic per-tensor scale of its calibration inputs, and later calls
only encode with it (one pass over x, no amax).  Checked against the oracle's
static-scale quantize (bit-exact codes) and GEMM (per-element tolerance),
including inputs beyond the calibrated range, which saturate to +-448."""
import numpy as np
import pytest
import torch

import synth
from bf16_gemm_vla_gb300 import frt, layers
from helpers import assert_gemm_close, bf16_dev
from oracle import e4m3, gemm, quantize

pytestmark = pytest.mark.gpu


def _bf16_bits(x):
    return synth.to_bf16_bits(np.asarray(x, dtype=np.float64))


def test_calibrated_scale_then_static_calls():
    M, K, N = 300, 1024, 512
    g = np.random.default_rng(41)
    lay = synth.layer(g, M, K, N, act_cols=N // 2, outlier_frac=0.01)
    w_dev = torch.from_numpy(lay["w_f32"]).cuda()
    b_dev = torch.from_numpy(lay["bias"]).cuda()
    pw = layers.prepare_fp8(w_dev, b_dev)
    dyn = layers.Linear(pw, M, act_cols=N // 2)
    stat = layers.Linear(pw, M, act_cols=N // 2)
    x_cal = [bf16_dev(lay["a_bf16"]), bf16_dev(_bf16_bits(0.25 * g.standard_normal((M, K))))]
    s = stat.calibrate(x_cal)
    # the largest of the inputs' dynamic scales, bit for bit
    _, s0 = quantize.quantize_e4m3(synth.bf16_bits_as_f32(lay["a_bf16"]), quantize.PER_TENSOR,
                                   e4m3.OCP)
    assert np.float32(s) == s0
    # on the calibration input the frozen scale is the dynamic one: same output
    o_dyn = dyn(x_cal[0]).clone()
    o_stat = stat(x_cal[0]).clone()
    assert torch.equal(o_dyn, o_stat)
    qw_o, sw_o = quantize.quantize_e4m3(lay["w_f32"], quantize.PER_COL, e4m3.OCP)
    # new inputs: smaller (codes use less range) and 3x larger (saturation)
    for scale in (0.5, 3.0):
        xf = np.float64(synth.bf16_bits_as_f32(lay["a_bf16"])) * scale
        bits = _bf16_bits(xf)
        xd = bf16_dev(bits)
        out = stat(xd)
        frt.check_device_status()
        x32 = synth.bf16_bits_as_f32(bits)
        qa_o, _ = quantize.quantize_e4m3(x32, quantize.PER_TENSOR, e4m3.OCP,
                                         static_scale=np.float32(s))
        np.testing.assert_array_equal(stat.q.cpu().numpy(), qa_o)
        if scale > 1:
            assert ((stat.q.cpu().numpy() & 0x7F) == 0x7E).any()  # saturated codes
        y, sumabs = gemm.gemm_fp8(qa_o, e4m3.OCP, np.float32(s), qw_o, e4m3.OCP, sw_o,
                                  lay["bias"], N // 2)
        assert_gemm_close(out, y, sumabs, "static scale x%.1f" % scale)


def test_static_scale_step_in_a_graph():
    # after calibration a layer is one encode kernel and one GEMM, and a
    # captured graph of it replays the eager result bit for bit
    M, K, N = 768, 2048, 2560
    lay = synth.layer(np.random.default_rng(5), M, K, N, act_cols=0, outlier_frac=0.01)
    pw = layers.prepare_fp8(torch.from_numpy(lay["w_f32"]).cuda(),
                            torch.from_numpy(lay["bias"]).cuda())
    lin = layers.Linear(pw, M)
    x = bf16_dev(lay["a_bf16"])
    lin.calibrate([x])
    eager = lin(x).clone()
    n0 = frt.frt_launch_count()
    lin(x)
    torch.cuda.synchronize()
    assert frt.frt_launch_count() - n0 == 2  # encode + GEMM
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        lin(x)
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        lin(x)
    lin.out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(lin.out, eager)
