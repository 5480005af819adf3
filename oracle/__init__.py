"""Plain CPU oracle for the quantized linear-layer path (test infrastructure).

This package is test infrastructure, not product code.  Only the test suite,
``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may import
it.  It shares no code with the CUDA library: every function here is written
from the format definitions and the method as the source pages describe it,
in fp64 wherever arithmetic is involved, without blocking, fusion or
reordering beyond what the definition states.

Sources (cited by page title and section):
  * "Real-time VLA inference on AMD hardware" (cyberneticphysics.com):
    "Different FP8 representation", "Packing around the instruction",
    "Merging gate and up", "FP8 helps the encoder and hurts the decoder".
  * "Deploying DeepSeek-V4-Flash on AMD MI300X" (lehuy.net): "The FP8
    dialect problem" (FNUZ = finite, NaNs, unsigned zero; same bit layout,
    exponent bias off by one, a byte read in the wrong dialect is 2x off).
  * The OCP 8-bit floating point specification (OFP8) for E4M3.

Modules:
  e4m3      -- decode / encode of E4M3 bytes in the OCP and FNUZ dialects
  bf16      -- fp32 -> bf16 round-to-nearest-even on bit patterns
  quantize  -- amax, scale and encode of a tensor (per tensor / per column)
  convert   -- FNUZ -> OCP re-encoding of bytes
  pack      -- the packed weight layout and its inverse
  gemm      -- fp64 GEMM on decoded values with the scale/bias/GELU epilogue
  nvfp4     -- E2M1 codes with E4M3 block scales: quantize, decode, GEMM
"""
from . import e4m3, bf16, quantize, convert, pack, gemm, nvfp4  # noqa: F401
