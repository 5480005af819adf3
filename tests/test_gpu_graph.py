"""CUDA-graph capture and replay of the path: a replayed graph gives the
eager result bit for bit, and the synthetic 18+18-layer stack matches the
oracle at its first and last layers."""
import numpy as np
import pytest
import torch

import synth
from bf16_gemm_vla_gb300 import frt, layers
from bf16_gemm_vla_gb300.stack import SyntheticStack
from helpers import assert_gemm_close, bf16_dev
from oracle import bf16 as obf16
from oracle import e4m3, gemm, quantize

pytestmark = pytest.mark.gpu


def test_graph_replay_equals_eager():
    lay = synth.decoder(seed=0)[1]
    w = torch.from_numpy(lay["w_f32"]).cuda()
    b = torch.from_numpy(lay["bias"]).cuda()
    fp8 = layers.Linear(layers.prepare_fp8(w, b), 50, act_cols=lay["N"])
    bf = layers.Linear(layers.prepare_bf16(w, b), 50, act_cols=lay["N"])
    x = torch.zeros((50, lay["K"]), dtype=torch.bfloat16, device="cuda")
    x.copy_(bf16_dev(lay["a_bf16"]))
    e1, e2 = fp8(x).clone(), bf(x).clone()  # eager (also sets kernel attributes)
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fp8(x)
        bf(x)
    torch.cuda.current_stream().wait_stream(s)
    with torch.cuda.graph(g):
        fp8(x)
        bf(x)
    fp8.out.zero_()
    bf.out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(fp8.out, e1) and torch.equal(bf.out, e2)
    # new input data through the same static buffer
    x.copy_(bf16_dev(synth.decoder(seed=5)[1]["a_bf16"]))
    g.replay()
    r1, r2 = fp8.out.clone(), bf.out.clone()
    f1, f2 = fp8(x).clone(), bf(x).clone()
    assert torch.equal(r1, f1) and torch.equal(r2, f2)
    frt.check_device_status()


def _check_layer(st, part, li, name):
    lin = (st.enc if part == "enc" else st.dec)[li][name]
    x = st.inputs_of(part, li, name)
    x_f32 = x.float().cpu().numpy()
    w, b = st.kept[(part, li, name)]
    w, b = w.numpy(), b.numpy()
    if lin.w.kind == "e4m3":
        qa_o, sa_o = quantize.quantize_e4m3(x_f32, quantize.PER_TENSOR, e4m3.OCP)
        np.testing.assert_array_equal(lin.q.cpu().numpy(), qa_o)
        assert lin.a_scale.cpu().numpy()[0] == sa_o
        qw_o, sw_o = quantize.quantize_e4m3(w, quantize.PER_COL, e4m3.OCP)
        np.testing.assert_array_equal(lin.w.w_scale.cpu().numpy(), sw_o)
        y, sumabs = gemm.gemm_fp8(qa_o, e4m3.OCP, sa_o, qw_o, e4m3.OCP, sw_o, b, lin.act_cols)
    else:
        y, sumabs = gemm.gemm_bf16(x_f32, obf16.round_to_bf16(w), None, b, lin.act_cols)
    assert_gemm_close(lin.out, y, sumabs, "%s layer %d %s" % (part, li, name))


def test_stack_graph_matches_oracle_at_first_and_last_layer():
    st = SyntheticStack(n_layers=18, seed=1, keep=(0, 17))
    xe, xd = synth.stack_inputs(seed=1)
    st.x_enc.copy_(bf16_dev(xe))
    st.x_dec.copy_(bf16_dev(xd))
    st.capture()
    st.replay()
    torch.cuda.synchronize()
    frt.check_device_status()
    for part in ("enc", "dec"):
        for li in (0, 17):
            for name in ("qkv", "o", "gate_up", "down"):
                _check_layer(st, part, li, name)
    e_out = st.enc[-1]["down"].out.clone()
    d_out = st.dec[-1]["down"].out.clone()
    st.replay()
    torch.cuda.synchronize()
    assert torch.equal(e_out, st.enc[-1]["down"].out)
    assert torch.equal(d_out, st.dec[-1]["down"].out)
    # one GEMM per layer; every FP8 layer's input is quantized by one launch:
    # the encoder's input by a full quantize (768 x 2048 dense bf16: one
    # grid), every later one by the encode pass with the scale the GEMM
    # before it took
    n = st.launches_per_forward()
    assert n == 18 * 4 + 18 * 4 + 18 * 4
    assert st.launches_per_forward() == n


def test_fused_scale_stack_equals_separate_quantize_stack():
    # the same stack with each FP8 layer's input quantized by a full quantize
    # (amax included): every layer's bf16 output, quantized bytes and scale
    # are equal bit for bit (the scale a GEMM takes is that of its stored
    # output)
    xe, xd = synth.stack_inputs(seed=1)
    outs = []
    for fuse in (True, False):
        st = SyntheticStack(n_layers=18, seed=1, keep=(), fuse_quantize=fuse, parts=("enc",))
        st.x_enc.copy_(bf16_dev(xe))
        st.forward()
        torch.cuda.synchronize()
        frt.check_device_status()
        outs.append([(lay[n].out.clone(), lay[n].q.clone(), lay[n].a_scale.clone())
                     for lay in st.enc for n in ("qkv", "o", "gate_up", "down")])
        del st
    for (o1, q1, s1), (o2, q2, s2) in zip(*outs):
        assert torch.equal(o1, o2) and torch.equal(q1, q2) and torch.equal(s1, s2)
