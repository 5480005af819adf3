"""The C-ABI library loads, exports every entry point the header declares,
and rejects bad arguments on the host before touching the device (no
compute call is made here: these run without a GPU)."""
import ctypes
import os
import re

import pytest

from bf16_gemm_vla_gb300 import _lib, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "frt.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _lib.load()


def header_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(frt_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_binding(lib):
    names = header_functions()
    assert "frt_gemm_fp8" in names and "frt_quantize_e4m3" in names
    assert sorted(_lib.SIGNATURES) == names


def test_library_exports_every_header_symbol(lib):
    for name in header_functions():
        assert hasattr(lib, name), name
    assert lib.frt_abi_version() == 3
    assert lib.frt_launch_count() >= 0


def test_status_strings(lib):
    for code, name in _lib.STATUS_NAMES.items():
        assert lib.frt_status_string(code).decode() == name
    assert lib.frt_status_string(99).decode() == "FRT_ERR_UNKNOWN"


def test_sizes(lib):
    assert lib.frt_packed_weight_bytes(1024, 4096, _lib.FRT_E4M3_OCP) == 1024 * 4096
    assert lib.frt_packed_weight_bytes(1024, 4096, _lib.FRT_BF16) == 1024 * 4096 * 2
    # padding to 128 channels x 128 bytes
    assert lib.frt_packed_weight_bytes(96, 200, _lib.FRT_E4M3_OCP) == 2 * 1 * 16384
    assert lib.frt_packed_weight_bytes(80, 136, _lib.FRT_BF16) == 2 * 2 * 16384
    assert lib.frt_packed_weight_bytes(64, 64, _lib.FRT_F32) == 0
    assert lib.frt_quantize_workspace_bytes(50, 1024, _lib.FRT_SCALE_PER_TENSOR) == 256 + 4096
    assert lib.frt_quantize_workspace_bytes(4096, 1024, _lib.FRT_SCALE_PER_COL) == 256 + 64 * 1024 * 4
    assert lib.frt_gemm_workspace_bytes(50, 1024, 4096, _lib.FRT_E4M3_OCP) == 0


def test_gemm_describe_rejects_unsupported_problems(lib):
    # checked before any device query: N % 16, K % 32 (FP8) / 16 (BF16),
    # nonpositive sizes and a dtype other than E4M3 OCP or BF16
    buf = ctypes.create_string_buffer(64)
    for args in ((50, 1000, 4096, _lib.FRT_E4M3_OCP), (50, 1024, 4080, _lib.FRT_E4M3_OCP),
                 (50, 1024, 4104, _lib.FRT_BF16), (0, 1024, 4096, _lib.FRT_BF16),
                 (50, 1024, 4096, _lib.FRT_E4M3_FNUZ)):
        assert lib.frt_gemm_describe(*args, 0, buf, len(buf)) == -1


FAKE = 0x10000  # a 64 KiB-aligned address that is never dereferenced: every
                # call below fails its host-side checks before any CUDA call


def test_quantize_rejects_bad_arguments(lib):
    q = lib.frt_quantize_e4m3
    ok_args = [FAKE, _lib.FRT_BF16, 4, 16, 16, _lib.FRT_SCALE_PER_TENSOR, _lib.FRT_E4M3_OCP,
               None, FAKE, FAKE, FAKE, 4096, None]

    def call(**kw):
        a = list(ok_args)
        names = ["x", "dt", "rows", "cols", "ldx", "mode", "fmt", "static", "q", "scale", "ws",
                 "wsb", "stream"]
        for k, v in kw.items():
            a[names.index(k)] = v
        return q(*a)

    assert call(dt=_lib.FRT_E4M3_OCP) == 1
    assert call(fmt=_lib.FRT_BF16) == 1
    assert call(mode=7) == 1
    assert call(rows=-1) == 1
    assert call(ldx=8) == 1
    assert call(x=None) == 1
    assert call(ws=None) == 1
    assert call(x=FAKE + 1) == 3
    assert call(wsb=16) == 4
    assert call(rows=0) == 0  # empty: nothing to do


def test_fnuz_rejects_bad_arguments(lib):
    f = lib.frt_fnuz_to_ocp
    assert f(None, FAKE, 16, None) == 1
    assert f(FAKE, FAKE + 8, 16, None) == 1  # partial overlap
    assert f(None, None, 0, None) == 0


def test_pack_rejects_bad_arguments(lib):
    p = lib.frt_pack_weights
    need = lib.frt_packed_weight_bytes(64, 128, _lib.FRT_E4M3_OCP)
    assert p(FAKE, _lib.FRT_E4M3_OCP, 64, 128, 128, _lib.FRT_BF16, FAKE, need, None) == 1
    assert p(FAKE, _lib.FRT_F32, 64, 128, 100, _lib.FRT_BF16, FAKE, need, None) == 1
    assert p(FAKE, _lib.FRT_E4M3_OCP, 64, 128, 128, _lib.FRT_E4M3_OCP, FAKE, need - 1, None) == 4
    assert p(FAKE, _lib.FRT_E4M3_OCP, 64, 128, 128, _lib.FRT_E4M3_OCP, FAKE + 8, need, None) == 3


def test_gemm_rejects_bad_arguments(lib):
    g = lib.frt_gemm_fp8
    base = dict(a=FAKE, lda=1024, a_scale=FAKE, w=FAKE, w_scale=FAKE, bias=None, M=50, N=1024,
                K=1024, act=0, act_cols=0, out=FAKE, ldo=1024, ws=None, wsb=0, status=None,
                stream=None)
    order = list(base)

    def call(**kw):
        d = dict(base)
        d.update(kw)
        return g(*[d[k] for k in order])

    assert call(a=None) == 1
    assert call(w_scale=None) == 1
    assert call(act=5) == 1
    assert call(act=1, act_cols=2048) == 1
    assert call(M=0) == 1
    assert call(lda=512) == 1
    assert call(N=1000, ldo=1000) == 2
    assert call(K=1000, lda=1000) == 2
    assert call(a=FAKE + 16 * 3 + 8) == 3
    assert call(ldo=1028) == 3
    assert call(lda=1032) == 3  # 1032 bytes is not a multiple of 16
    assert call(lda=1025) == 3
    b = lib.frt_gemm_bf16
    assert b(FAKE, 1024, FAKE, None, None, 50, 1024, 1000, 0, 0, FAKE, 1024, None, 0, None,
             None) == 2
    assert b(FAKE, 1028, FAKE, None, None, 50, 1024, 1024, 0, 0, FAKE, 1024, None, 0, None,
             None) == 3


def test_decoder_boundary_rejects_bad_arguments(lib):
    f = lib.frt_gate_residual_ada_norm_bf16
    code = {name: c for c, name in _lib.STATUS_NAMES.items()}
    ok = [FAKE, FAKE, FAKE, FAKE, 50, 1024, 1e-6, FAKE, FAKE, None]
    assert f(*ok[:4], 0, 1024, 1e-6, *ok[7:]) == code["FRT_OK"]  # M = 0: nothing
    for i, v, want in ((4, -1, "FRT_ERR_INVALID_ARG"), (5, 12, "FRT_ERR_UNSUPPORTED_SHAPE"),
                       (5, 4104, "FRT_ERR_UNSUPPORTED_SHAPE"), (6, -1.0, "FRT_ERR_INVALID_ARG"),
                       (0, None, "FRT_ERR_INVALID_ARG"), (3, FAKE + 8, "FRT_ERR_MISALIGNED")):
        a = list(ok)
        a[i] = v
        assert f(*a) == code[want], (i, v)


def test_nvfp4_sizes(lib):
    # one E4M3 block scale per 16 elements of K, vectors padded to 128
    assert lib.frt_nvfp4_scale_bytes(768, 2048) == 768 * 2048 // 16
    assert lib.frt_nvfp4_scale_bytes(1, 64) == 128 * 4
    assert lib.frt_nvfp4_scale_bytes(200, 512) == 256 * 32
    assert lib.frt_nvfp4_scale_bytes(0, 64) == 0
    assert lib.frt_nvfp4_scale_bytes(16, 96) == 0  # K not a multiple of 64
    assert lib.frt_quantize_nvfp4_workspace_bytes() == 16
    assert lib.frt_gemm_next_scale_workspace_bytes() == 256


def test_nvfp4_quantize_rejects_bad_arguments(lib):
    code = {name: c for c, name in _lib.STATUS_NAMES.items()}
    sfb = lib.frt_nvfp4_scale_bytes(64, 256)
    names = ["x", "dt", "rows", "cols", "ldx", "along", "static", "q", "sf", "sfb", "scale", "ws",
             "wsb", "stream"]
    ok = [FAKE, _lib.FRT_BF16, 64, 256, 256, 0, None, FAKE, FAKE, sfb, FAKE, FAKE, 16, None]

    def call(**kw):
        a = list(ok)
        for k, v in kw.items():
            a[names.index(k)] = v
        return lib.frt_quantize_nvfp4(*a)

    for kw, want in ((dict(x=None), "FRT_ERR_INVALID_ARG"), (dict(sf=None), "FRT_ERR_INVALID_ARG"),
                     (dict(dt=_lib.FRT_E4M3_OCP), "FRT_ERR_INVALID_ARG"),
                     (dict(rows=0), "FRT_ERR_INVALID_ARG"), (dict(ldx=128), "FRT_ERR_INVALID_ARG"),
                     (dict(cols=96, ldx=96), "FRT_ERR_UNSUPPORTED_SHAPE"),
                     (dict(along=1, rows=96), "FRT_ERR_UNSUPPORTED_SHAPE"),  # blocks down 96 rows
                     (dict(sfb=sfb - 1), "FRT_ERR_WORKSPACE_TOO_SMALL"),
                     (dict(ws=None), "FRT_ERR_WORKSPACE_TOO_SMALL"),
                     (dict(wsb=8), "FRT_ERR_WORKSPACE_TOO_SMALL"),
                     (dict(x=FAKE + 8), "FRT_ERR_MISALIGNED"), (dict(q=FAKE + 4), "FRT_ERR_MISALIGNED"),
                     (dict(ldx=260), "FRT_ERR_MISALIGNED")):  # 520-byte rows
        assert call(**kw) == code[want], kw


def test_nvfp4_gemm_rejects_bad_arguments(lib):
    code = {name: c for c, name in _lib.STATUS_NAMES.items()}
    names = ["a", "lda", "a_sf", "a_scale", "w", "w_sf", "w_scale", "bias", "M", "N", "K", "act",
             "act_cols", "out", "ldo", "status", "stream"]
    ok = [FAKE, 128, FAKE, FAKE, FAKE, FAKE, FAKE, None, 64, 256, 256, 0, 0, FAKE, 256, None, None]

    def call(**kw):
        a = list(ok)
        for k, v in kw.items():
            a[names.index(k)] = v
        return lib.frt_gemm_nvfp4(*a)

    for kw, want in ((dict(a=None), "FRT_ERR_INVALID_ARG"), (dict(w_sf=None), "FRT_ERR_INVALID_ARG"),
                     (dict(act=_lib.FRT_ACT_GEGLU), "FRT_ERR_INVALID_ARG"),
                     (dict(act=1, act_cols=512), "FRT_ERR_INVALID_ARG"),
                     (dict(M=0), "FRT_ERR_INVALID_ARG"), (dict(lda=64), "FRT_ERR_INVALID_ARG"),
                     (dict(ldo=128), "FRT_ERR_INVALID_ARG"),
                     (dict(K=192, lda=96), "FRT_ERR_UNSUPPORTED_SHAPE"),
                     (dict(N=200, ldo=200), "FRT_ERR_UNSUPPORTED_SHAPE"),
                     (dict(a=FAKE + 8), "FRT_ERR_MISALIGNED"), (dict(lda=136), "FRT_ERR_MISALIGNED"),
                     (dict(ldo=260), "FRT_ERR_MISALIGNED")):
        assert call(**kw) == code[want], kw


def test_next_scale_gemm_rejects_bad_arguments(lib):
    code = {name: c for c, name in _lib.STATUS_NAMES.items()}
    names = ["a", "lda", "a_scale", "w", "w_scale", "bias", "M", "N", "K", "act", "act_cols", "out",
             "ldo", "scale_cols", "scale", "sws", "swsb", "ws", "wsb", "status", "stream"]
    ok = [FAKE, 1024, FAKE, FAKE, FAKE, None, 50, 1024, 1024, 0, 0, FAKE, 1024, 1024, FAKE, FAKE,
          256, None, 0, None, None]

    def call(**kw):
        a = list(ok)
        for k, v in kw.items():
            a[names.index(k)] = v
        return lib.frt_gemm_fp8_next_scale(*a)

    for kw, want in ((dict(scale=None), "FRT_ERR_INVALID_ARG"), (dict(sws=None), "FRT_ERR_INVALID_ARG"),
                     (dict(scale_cols=0), "FRT_ERR_INVALID_ARG"),
                     (dict(scale_cols=2048), "FRT_ERR_INVALID_ARG"),  # past the output's columns
                     (dict(scale_cols=1020), "FRT_ERR_UNSUPPORTED_SHAPE"),
                     (dict(scale=FAKE + 2), "FRT_ERR_MISALIGNED"),
                     (dict(sws=FAKE + 8), "FRT_ERR_MISALIGNED"),
                     (dict(swsb=128), "FRT_ERR_WORKSPACE_TOO_SMALL")):
        assert call(**kw) == code[want], kw
    # the BF16 variant runs the same checks
    b = lib.frt_gemm_bf16_next_scale
    assert b(FAKE, 1024, FAKE, None, None, 50, 1024, 1024, 0, 0, FAKE, 1024, 1020, FAKE, FAKE, 256,
             None, 0, None, None) == code["FRT_ERR_UNSUPPORTED_SHAPE"]
