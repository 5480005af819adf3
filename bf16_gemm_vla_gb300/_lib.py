"""ctypes view of libfrt.so (the C ABI declared in include/frt.h)."""
import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libfrt.so")

# frt_status
FRT_OK = 0
FRT_ERR_INVALID_ARG = 1
FRT_ERR_UNSUPPORTED_SHAPE = 2
FRT_ERR_MISALIGNED = 3
FRT_ERR_WORKSPACE_TOO_SMALL = 4
FRT_ERR_CUDA = 5
FRT_ERR_TIMEOUT = 6
STATUS_NAMES = {
    0: "FRT_OK", 1: "FRT_ERR_INVALID_ARG", 2: "FRT_ERR_UNSUPPORTED_SHAPE",
    3: "FRT_ERR_MISALIGNED", 4: "FRT_ERR_WORKSPACE_TOO_SMALL", 5: "FRT_ERR_CUDA",
    6: "FRT_ERR_TIMEOUT",
}
# frt_dtype
FRT_F32, FRT_BF16, FRT_E4M3_OCP, FRT_E4M3_FNUZ = 0, 1, 2, 3
# frt_scale_mode
FRT_SCALE_PER_TENSOR, FRT_SCALE_PER_COL = 0, 1
# frt_act
FRT_ACT_NONE, FRT_ACT_GELU_TANH, FRT_ACT_GEGLU = 0, 1, 2

_c_i64 = ctypes.c_int64
_c_sz = ctypes.c_size_t
_c_p = ctypes.c_void_p
_c_int = ctypes.c_int

# name -> (restype, argtypes), in the order of include/frt.h
SIGNATURES = {
    "frt_abi_version": (_c_int, []),
    "frt_launch_count": (ctypes.c_ulonglong, []),
    "frt_status_string": (ctypes.c_char_p, [_c_int]),
    "frt_quantize_workspace_bytes": (_c_sz, [_c_i64, _c_i64, _c_int]),
    "frt_quantize_e4m3": (_c_int, [_c_p, _c_int, _c_i64, _c_i64, _c_i64, _c_int, _c_int, _c_p,
                                   _c_p, _c_p, _c_p, _c_sz, _c_p]),
    "frt_quantize_e4m3_noalloc": (_c_int, [_c_p, _c_int, _c_i64, _c_i64, _c_i64, _c_int, _c_int,
                                           _c_p, _c_p, _c_p, _c_p]),
    "frt_fnuz_to_ocp": (_c_int, [_c_p, _c_p, _c_sz, _c_p]),
    "frt_packed_weight_bytes": (_c_sz, [_c_i64, _c_i64, _c_int]),
    "frt_pack_weights": (_c_int, [_c_p, _c_int, _c_i64, _c_i64, _c_i64, _c_int, _c_p, _c_sz,
                                  _c_p]),
    "frt_gemm_workspace_bytes": (_c_sz, [_c_i64, _c_i64, _c_i64, _c_int]),
    "frt_gemm_describe": (_c_int, [_c_i64, _c_i64, _c_i64, _c_int, _c_sz, ctypes.c_char_p,
                                   _c_sz]),
    "frt_gemm_next_scale_workspace_bytes": (_c_sz, []),
    "frt_gemm_fp8_next_scale": (_c_int, [_c_p, _c_i64, _c_p, _c_p, _c_p, _c_p, _c_i64, _c_i64,
                                         _c_i64, _c_int, _c_i64, _c_p, _c_i64, _c_i64, _c_p, _c_p,
                                         _c_sz, _c_p, _c_sz, _c_p, _c_p]),
    "frt_gemm_bf16_next_scale": (_c_int, [_c_p, _c_i64, _c_p, _c_p, _c_p, _c_i64, _c_i64, _c_i64,
                                          _c_int, _c_i64, _c_p, _c_i64, _c_i64, _c_p, _c_p, _c_sz,
                                          _c_p, _c_sz, _c_p, _c_p]),
    "frt_nvfp4_scale_bytes": (_c_sz, [_c_i64, _c_i64]),
    "frt_quantize_nvfp4_workspace_bytes": (_c_sz, []),
    "frt_quantize_nvfp4": (_c_int, [_c_p, _c_int, _c_i64, _c_i64, _c_i64, _c_int, _c_p, _c_p,
                                    _c_p, _c_sz, _c_p, _c_p, _c_sz, _c_p]),
    "frt_gemm_nvfp4": (_c_int, [_c_p, _c_i64, _c_p, _c_p, _c_p, _c_p, _c_p, _c_p, _c_i64,
                                _c_i64, _c_i64, _c_int, _c_i64, _c_p, _c_i64, _c_p, _c_p]),
    "frt_gate_residual_ada_norm_bf16": (_c_int, [_c_p, _c_p, _c_p, _c_p, _c_i64, _c_i64,
                                                 ctypes.c_float, _c_p, _c_p, _c_p]),
    "frt_gemm_fp8": (_c_int, [_c_p, _c_i64, _c_p, _c_p, _c_p, _c_p, _c_i64, _c_i64, _c_i64,
                              _c_int, _c_i64, _c_p, _c_i64, _c_p, _c_sz, _c_p, _c_p]),
    "frt_gemm_bf16": (_c_int, [_c_p, _c_i64, _c_p, _c_p, _c_p, _c_i64, _c_i64, _c_i64, _c_int,
                               _c_i64, _c_p, _c_i64, _c_p, _c_sz, _c_p, _c_p]),
}

_LIB = None


def load(path=LIB_PATH):
    """Loads libfrt.so and declares every entry point.  Raises if the library
    has not been built: there is no fallback path."""
    global _LIB
    if _LIB is not None:
        return _LIB
    if not os.path.exists(path):
        raise ImportError(
            "libfrt.so is not built (%s); build it with bf16_gemm_vla_gb300.build.build()" % path)
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _LIB = lib
    return lib
