"""GB300-native FP8/BF16 linear layers for latency-bound VLA inference.

The compute path lives in libfrt.so (hand-written sm_103a CUDA kernels behind
the C ABI of include/frt.h).  This package is its thin Python binding plus
the load-time and graph-replay helpers built on it:

  frt     -- one function per C entry point, taking torch tensors
  layers  -- load-time weight preparation and a static-buffer linear layer
  stack   -- the synthetic encoder/decoder stack captured as one CUDA graph
  build   -- compiles libfrt.so in-tree with nvcc for sm_103a
"""
from .frt import (  # noqa: F401
    FNUZ, OCP, PER_COL, PER_TENSOR, FrtError, check_device_status, device_status,
    frt_fnuz_to_ocp, frt_gate_residual_ada_norm_bf16, frt_gemm_bf16, frt_gemm_describe,
    frt_gemm_fp8, frt_gemm_workspace_bytes, frt_launch_count, frt_pack_weights,
    frt_packed_weight_bytes, frt_quantize_e4m3, frt_quantize_e4m3_noalloc,
    frt_quantize_workspace_bytes, gemm_workspace,
)
