"""The quantize entry point that allocates nothing, called through the C ABI.

It serves callers that cannot allocate device memory (a running real-time
loop, a plugin handed raw pointers, a graph capture that must not
allocate).  Its scratch is a fixed array inside the library instead of a
caller workspace; its results must equal frt_quantize_e4m3's bit for bit
(the tolerance of every quantize test), call after call.  This file sorts
last so a run stopping at the first failure has run every other test first.
"""
import ctypes

import numpy as np
import pytest
import torch

from bf16_gemm_vla_gb300 import _lib, frt

pytestmark = pytest.mark.gpu


def _noalloc(x, mode, fmt, q, scale):
    lib = _lib.load()
    rows, cols = x.shape
    return lib.frt_quantize_e4m3_noalloc(
        x.data_ptr(), frt._XDT[x.dtype], rows, cols, x.stride(0), frt._MODE[mode],
        frt._FMT[fmt], None, q.data_ptr(), scale.data_ptr(),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("mode,fmt,dtype,shape", [
    (frt.PER_TENSOR, frt.OCP, torch.bfloat16, (50, 1024)),
    (frt.PER_TENSOR, frt.FNUZ, torch.float32, (768, 2048)),
    (frt.PER_COL, frt.OCP, torch.float32, (1024, 256)),
    (frt.PER_COL, frt.FNUZ, torch.bfloat16, (333, 100)),
])
def test_noalloc_matches_workspace_entry_twice(mode, fmt, dtype, shape):
    g = torch.Generator(device="cuda")
    g.manual_seed(shape[0] * 7 + shape[1])
    for call in range(2):  # two calls in a row share the library's scratch array
        x = (torch.randn(shape, generator=g, device="cuda") * (1.0 + 3 * call)).to(dtype)
        q_ref, s_ref = frt.frt_quantize_e4m3(x, mode, fmt)
        q = torch.full(shape, 0x55, dtype=torch.uint8, device="cuda")
        s = torch.full((shape[1] if mode == frt.PER_COL else 1,), -1.0, device="cuda")
        assert _noalloc(x, mode, fmt, q, s) == _lib.FRT_OK
        torch.cuda.synchronize()
        assert torch.equal(q, q_ref), (mode, fmt, call)
        assert torch.equal(s, s_ref), (mode, fmt, call)


def test_noalloc_rejects_shapes_beyond_its_scratch():
    # per column, ceil(rows / 64) * cols partials must fit 262144 floats
    x = torch.zeros((64 * 2, 262144 // 2 + 16), dtype=torch.float32, device="cuda")
    q = torch.empty(x.shape, dtype=torch.uint8, device="cuda")
    s = torch.empty((x.shape[1],), dtype=torch.float32, device="cuda")
    assert _noalloc(x, frt.PER_COL, frt.OCP, q, s) == _lib.FRT_ERR_UNSUPPORTED_SHAPE
    # the largest shape that fits is accepted and matches the workspace entry point
    x = torch.randn((64 * 2, 262144 // 2), device="cuda")
    q = torch.empty(x.shape, dtype=torch.uint8, device="cuda")
    s = torch.empty((x.shape[1],), dtype=torch.float32, device="cuda")
    assert _noalloc(x, frt.PER_COL, frt.OCP, q, s) == _lib.FRT_OK
    q_ref, s_ref = frt.frt_quantize_e4m3(x, frt.PER_COL, frt.OCP)
    torch.cuda.synchronize()
    assert torch.equal(q, q_ref) and torch.equal(s, s_ref)
