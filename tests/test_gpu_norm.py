"""GPU parity of the BF16 decoder block boundary (gated residual update and
adaptive RMS norm in one kernel) against oracle/norm.py: the updated
residual and the passed-on gate bit for bit, the normalized output within
|gpu - oracle| <= 2^-8 |oracle| + 1e-5 (|r inv (1 + scale)| + |shift|)
(the bf16 store plus the kernel's fp32 sum of squares)."""
import numpy as np
import pytest
import torch

from bf16_gemm_vla_gb300 import frt
from helpers import bf16_dev
from oracle import norm

pytestmark = pytest.mark.gpu


def _bits(g, shape, std):
    return torch.from_numpy(g.standard_normal(shape) * std).to(torch.bfloat16).view(
        torch.int16).numpy().view(np.uint16)


def _f32(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32)


@pytest.mark.parametrize("M,H", [(50, 1024), (10, 1024), (1, 8), (7, 4096), (64, 2048)])
def test_gate_residual_ada_norm(M, H):
    g = np.random.default_rng(M * 31 + H)
    res, out, gate = _bits(g, (M, H), 1.0), _bits(g, (M, H), 1.0), _bits(g, (M, H), 1.0)
    style = np.concatenate([_bits(g, (M, H), 0.1), _bits(g, (M, H), 0.1), _bits(g, (M, H), 1.0)],
                           axis=1)
    res_d = bf16_dev(res)
    normed, nxt = frt.frt_gate_residual_ada_norm_bf16(res_d, bf16_dev(out), bf16_dev(gate),
                                                      bf16_dev(style), eps=1e-6)
    torch.cuda.synchronize()
    r, y, g_o, mag = norm.gate_residual_ada_norm(_f32(res), _f32(out), _f32(gate), _f32(style),
                                                 1e-6)
    np.testing.assert_array_equal(res_d.float().cpu().numpy(), r.astype(np.float32))
    np.testing.assert_array_equal(nxt.float().cpu().numpy(), g_o.astype(np.float32))
    got = normed.float().cpu().numpy().astype(np.float64)
    bound = 2.0 ** -8 * np.abs(y) + 1e-5 * mag
    err = np.abs(got - y)
    assert (err <= bound).all(), (err.max(), np.argmax(err - bound))


def test_gate_residual_ada_norm_edges():
    z = torch.zeros((0, 1024), dtype=torch.bfloat16, device="cuda")
    s = torch.zeros((0, 3072), dtype=torch.bfloat16, device="cuda")
    n, g = frt.frt_gate_residual_ada_norm_bf16(z, z, z, s)
    assert n.shape == (0, 1024) and g.shape == (0, 1024)
    for H in (12, 4104):  # H % 8 != 0; H > 4096
        a = torch.zeros((2, H), dtype=torch.bfloat16, device="cuda")
        st = torch.zeros((2, 3 * H), dtype=torch.bfloat16, device="cuda")
        with pytest.raises(frt.FrtError):
            frt.frt_gate_residual_ada_norm_bf16(a, a, a, st)
