"""Oracle: fp32 <-> bf16 on bit patterns (test infrastructure only).

bf16 keeps the top 16 bits of an fp32 (sign, 8 exponent bits, 7 mantissa
bits).  Rounding fp32 to bf16 to nearest-even adds 0x7FFF plus the lowest
kept bit to the fp32 bit pattern and drops the low 16 bits; the carry makes
a tie round to the even neighbour and lets a mantissa overflow step into the
next binade (up to infinity).  NaNs stay NaN (made quiet).
"""
import numpy as np


def f32_to_bf16_bits(x):
    """fp32 array -> uint16 bf16 bit patterns, round-to-nearest-even."""
    x = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    u = x.view(np.uint32).astype(np.uint64)
    keep_lsb = (u >> np.uint64(16)) & np.uint64(1)
    r = (u + np.uint64(0x7FFF) + keep_lsb) >> np.uint64(16)
    nan = np.isnan(x)
    r = np.where(nan, (u >> np.uint64(16)) | np.uint64(0x0040), r)
    return r.astype(np.uint16)


def bf16_bits_to_f32(b):
    """uint16 bf16 bit patterns -> fp32 values (exact)."""
    b = np.ascontiguousarray(np.asarray(b, dtype=np.uint16))
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


def round_to_bf16(x):
    """fp32 values rounded to the nearest bf16, returned as fp32."""
    return bf16_bits_to_f32(f32_to_bf16_bits(x))
