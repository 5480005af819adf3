"""Pins of the decoder-boundary oracle (oracle/norm.py) against hand values,
closed forms and PyTorch's RMS norm."""
import numpy as np
import torch

from oracle import norm


def _style(scale, shift, nxt):
    return np.concatenate([scale, shift, nxt], axis=1)


def test_residual_update_rounds_to_fp32_then_bf16():
    # 1 + 2^-8 is a bf16 tie: to the even neighbour 1.0; 1 + 3 * 2^-9 is
    # nearer 1 + 2^-7; 2 + 2^-6 is exact in bf16
    res = np.array([[1.0, 1.0, 2.0, 0.0, 0.0, 0.0, 0.0, 0.0]])
    out = np.array([[2.0 ** -8, 3 * 2.0 ** -9, 1.0, 0.0, 0.0, 0.0, 0.0, 0.0]])
    gate = np.array([[1.0, 1.0, 2.0 ** -6, 0.0, 0.0, 0.0, 0.0, 0.0]])
    z = np.zeros_like(res)
    r, _, _, _ = norm.gate_residual_ada_norm(res, out, gate, _style(z, z, z), 0.0)
    np.testing.assert_array_equal(r[0, :3], [1.0, 1.0 + 2.0 ** -7, 2.0 + 2.0 ** -6])


def test_constant_row_normalizes_to_one_and_parts_are_in_order():
    H = 16
    res = np.full((2, H), 3.0)
    z = np.zeros((2, H))
    nxt = np.arange(2 * H, dtype=np.float64).reshape(2, H)
    _, y, g, mag = norm.gate_residual_ada_norm(res, z, z, _style(z, z, nxt), 0.0)
    np.testing.assert_array_equal(y, np.ones((2, H)))
    np.testing.assert_array_equal(g, nxt)  # the third part, passed on
    np.testing.assert_array_equal(mag, np.ones((2, H)))
    # scale first (1 + scale multiplies), shift second (adds): a swapped
    # split gives other values
    _, y2, _, _ = norm.gate_residual_ada_norm(res, z, z, _style(z + 1.0, z + 5.0, nxt), 0.0)
    np.testing.assert_array_equal(y2, np.full((2, H), 7.0))


def test_hand_row_and_eps():
    # r = [3, 4, 0 ...] over H = 8: mean(r^2) = 25 / 8
    res = np.zeros((1, 8))
    res[0, :2] = [3.0, 4.0]
    z = np.zeros_like(res)
    _, y, _, _ = norm.gate_residual_ada_norm(res, z, z, _style(z, z, z), 0.0)
    np.testing.assert_allclose(y[0, :2], np.array([3.0, 4.0]) / np.sqrt(25.0 / 8.0), rtol=1e-15)
    # eps adds under the root (an all-zero row stays finite: 0)
    _, y0, _, _ = norm.gate_residual_ada_norm(z, z, z, _style(z, z, z), 1e-6)
    np.testing.assert_array_equal(y0, z)


def test_matches_torch_rms_norm():
    g = np.random.default_rng(3)
    M, H = 5, 64
    res = g.standard_normal((M, H))
    res = torch.from_numpy(res).to(torch.bfloat16).double().numpy()
    z = np.zeros_like(res)
    sc = np.float64(g.standard_normal((M, H)) * 0.1)
    sh = np.float64(g.standard_normal((M, H)) * 0.1)
    r, y, _, _ = norm.gate_residual_ada_norm(res, z, z, _style(sc, sh, z), 1e-6)
    ref = torch.nn.functional.rms_norm(torch.from_numpy(r), (H,), eps=float(np.float32(1e-6)))
    np.testing.assert_allclose(y, ref.numpy() * (1.0 + sc) + sh, rtol=1e-12, atol=1e-14)
