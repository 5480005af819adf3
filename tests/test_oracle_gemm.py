"""Pins for the oracle's GEMM and epilogue."""
import math

import numpy as np
import pytest
import torch

import synth
from oracle import e4m3, gemm, quantize

# OCP E4M3 bytes of the integers 0..8, typed by hand from the format
# (bias 7: 1 = 0x38, 2 = 0x40, 3 = 1.5 * 2 = 0x44, 4 = 0x48, 5 = 1.25 * 4 = 0x4a,
#  6 = 1.5 * 4 = 0x4c, 7 = 1.75 * 4 = 0x4e, 8 = 0x50); negatives set bit 7.
INT_CODE = {0: 0x00, 1: 0x38, 2: 0x40, 3: 0x44, 4: 0x48, 5: 0x4A, 6: 0x4C, 7: 0x4E, 8: 0x50}


def int_bytes(v):
    return np.vectorize(lambda x: INT_CODE[abs(int(x))] | (0x80 if x < 0 else 0))(v).astype(np.uint8)


@pytest.mark.parametrize("M,K,N", [(3, 5, 4), (16, 64, 32), (7, 96, 9)])
def test_integer_gemm_exact(M, K, N):
    g = np.random.default_rng(M * K * N)
    a = g.integers(-8, 9, (M, K))
    w = g.integers(-8, 9, (K, N))
    exact = [[sum(int(a[m, k]) * int(w[k, n]) for k in range(K)) for n in range(N)]
             for m in range(M)]
    y, sumabs = gemm.gemm_fp8(int_bytes(a), e4m3.OCP, 1.0, int_bytes(w), e4m3.OCP, None)
    np.testing.assert_array_equal(y, np.array(exact, dtype=np.float64))
    np.testing.assert_array_equal(sumabs, np.abs(a) @ np.abs(w))
    # with scales that are powers of two the result scales exactly
    ws = np.float32(2.0 ** np.arange(N) / 8)
    y2, _ = gemm.gemm_fp8(int_bytes(a), e4m3.OCP, 0.25, int_bytes(w), e4m3.OCP, ws)
    np.testing.assert_array_equal(y2, np.array(exact) * 0.25 * ws[None, :])


def test_identity_weight_returns_activations():
    g = np.random.default_rng(3)
    a = synth.bf16_bits_as_f32(synth.to_bf16_bits(g.standard_normal((6, 32))))
    y, _ = gemm.gemm_bf16(a, np.eye(32, dtype=np.float32))
    np.testing.assert_array_equal(y, a.astype(np.float64))


def test_matmul_equals_naive_loop():
    g = np.random.default_rng(4)
    a = g.standard_normal((5, 17))
    w = g.standard_normal((17, 6))
    y, _ = gemm.gemm_values(a, w)
    np.testing.assert_allclose(y, gemm.gemm_naive(a, w), rtol=1e-13, atol=1e-13)


def test_gelu_tanh_closed_forms():
    x = np.array([-6.0, -3.0, -1.0, -0.5, 0.0, 0.5, 1.0, 3.0, 6.0])
    gl = gemm.gelu_tanh(x)
    assert gl[4] == 0.0
    # gelu(x) - gelu(-x) = x for the tanh form (tanh is odd)
    np.testing.assert_allclose(gl[::-1] - gl, -x, rtol=0, atol=1e-15)
    # library cross-check (PyTorch's tanh-approximate GELU, fp64)
    lib = torch.nn.functional.gelu(torch.from_numpy(x), approximate="tanh").numpy()
    np.testing.assert_allclose(gl, lib, rtol=1e-14, atol=1e-15)
    # close to the erf form x * Phi(x): the approximation error is below 1e-3
    erf = x * 0.5 * (1 + np.vectorize(math.erf)(x / math.sqrt(2)))
    assert np.max(np.abs(gl - erf)) < 1e-3


def test_epilogue_hand_case():
    # acc = [1, 2, 4]; * w_scale [1, .5, 2] = [1, 1, 8]; + bias [.5, -1, 0] = [1.5, 0, 8];
    # GELU on the first two columns only: [gelu(1.5), 0, 8]
    a = np.array([[1.0, 2.0]])
    w = np.array([[1.0, 0.0, 2.0], [0.0, 1.0, 1.0]])
    y, sumabs = gemm.gemm_values(a, w, None, np.float32([1, 0.5, 2]), np.float32([0.5, -1, 0]), 2)
    g15 = torch.nn.functional.gelu(torch.tensor(1.5, dtype=torch.float64), approximate="tanh")
    np.testing.assert_allclose(y, [[float(g15), 0.0, 8.0]], rtol=1e-15)
    np.testing.assert_array_equal(sumabs, [[1.0, 1.0, 8.0]])


def test_tiny_fp8_layer_close_to_unquantized():
    # end-to-end sanity of the tiny workload: FNUZ per-column weights
    # re-encoded to OCP, OCP per-tensor activations; the FP8 layer stays
    # within a few percent of the unquantized fp64 layer.
    from oracle import convert

    t = synth.tiny()
    a = synth.bf16_bits_as_f32(t["a_bf16"])
    qa, sa = quantize.quantize_e4m3(a, quantize.PER_TENSOR, e4m3.OCP)
    qz, sw = quantize.quantize_e4m3(t["w_f32"], quantize.PER_COL, e4m3.FNUZ)
    qw = convert.fnuz_to_ocp(qz)
    y, _ = gemm.gemm_fp8(qa, e4m3.OCP, sa, qw, e4m3.OCP, sw, t["bias"], 256)
    ref, _ = gemm.gemm_values(a, t["w_f32"], None, None, t["bias"], 256)
    err = np.abs(y - ref)
    assert np.sqrt(np.mean(err ** 2)) / np.sqrt(np.mean(ref ** 2)) < 0.08


def test_gelu_tanh_prime_against_central_differences():
    # the closed form against (f(v + h) - f(v - h)) / 2h in fp64, and its
    # limits: 0.5 at 0, 1 far right, 0 far left
    v = np.array([-6.0, -2.5, -1.0, -0.3, 0.0, 0.4, 1.0, 1.7, 3.0, 6.0])
    h = 1e-5
    fd = (gemm.gelu_tanh(v + h) - gemm.gelu_tanh(v - h)) / (2 * h)
    np.testing.assert_allclose(gemm.gelu_tanh_prime(v), fd, rtol=1e-8, atol=1e-9)
    assert gemm.gelu_tanh_prime(0.0) == 0.5
    assert abs(gemm.gelu_tanh_prime(20.0) - 1.0) < 1e-12
    assert abs(gemm.gelu_tanh_prime(-20.0)) < 1e-12


def test_geglu_gate_first_and_propagated_magnitude():
    # y = [g0 g1 | u0 u1]: h = [gelu(g0) u0, gelu(g1) u1]; a swapped split
    # (up first) or a missing product would give other values
    y = np.array([[1.0, -2.0, 3.0, 5.0], [0.0, 10.0, 7.0, -0.5]])
    s = np.array([[1.0, 2.0, 3.0, 4.0], [5.0, 6.0, 7.0, 8.0]])
    hh, prop = gemm.geglu(y, s)
    g = lambda v: 0.5 * v * (1.0 + math.tanh(math.sqrt(2.0 / math.pi) * (v + 0.044715 * v ** 3)))  # noqa: E731
    np.testing.assert_allclose(hh, [[g(1.0) * 3.0, g(-2.0) * 5.0], [0.0, g(10.0) * -0.5]],
                               rtol=1e-15, atol=0)
    # gelu(0) = 0: the up magnitude does not count, the gate's does at 0.5 |u|
    assert prop[1, 0] == 0.5 * 7.0 * 5.0
    # far right, gelu(g) = g and gelu'(g) = 1
    assert abs(prop[1, 1] - (0.5 * 6.0 + 10.0 * 8.0)) < 1e-9
