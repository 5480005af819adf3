"""Helpers shared by the GPU parity tests (host side only)."""
import numpy as np
import torch


def within_gemm_tolerance(gpu, ref, sumabs):
    """The GEMM acceptance bar, per element:
    |gpu - ref| <= 2^-7 * |ref| + 1e-5 * s_a * s_w[n] * sum_k |a * w|."""
    gpu = np.asarray(gpu, dtype=np.float64)
    err = np.abs(gpu - ref)
    bound = 2.0 ** -7 * np.abs(ref) + 1e-5 * sumabs
    return err <= bound, err, bound


def assert_gemm_close(gpu_out, ref, sumabs, what=""):
    g = gpu_out.float().cpu().numpy() if isinstance(gpu_out, torch.Tensor) else gpu_out
    ok, err, bound = within_gemm_tolerance(g, ref, sumabs)
    if not ok.all():
        bad = np.argwhere(~ok)
        i = tuple(bad[0])
        raise AssertionError(
            "%s: %d of %d elements outside the tolerance; first at %s: gpu %r ref %r err %.3g "
            "bound %.3g" % (what, len(bad), ok.size, i, float(g[i]), float(ref[i]),
                            float(err[i]), float(bound[i])))


def bf16_dev(bits, device="cuda"):
    """uint16 bf16 bit patterns -> bf16 CUDA tensor (bit copy)."""
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)


def bf16_host_f32(t):
    """bf16 CUDA tensor -> fp32 numpy values (exact)."""
    return t.float().cpu().numpy()
