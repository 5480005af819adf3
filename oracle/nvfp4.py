"""Oracle: NVFP4, block-scaled 4-bit floats (test infrastructure only).

The pages name an NVFP4 path beside FP8 for the pi0.5 encoder FFN (the
FlashRT article, section 7.2 in its table of contents, and the
``use_fp4`` / ``fp4_layers`` switches of its ``load_model`` listing) but give
no formula.  The reading taken here is the plain two-level block scaling of
E2M1 values that the NVFP4 name refers to:

  * elements are E2M1: one sign bit, two exponent bits (bias 1) and one
    mantissa bit, i.e. magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6 (exponent field
    0 is subnormal: m * 0.5); no infinity or NaN; -0 exists (code 0x8);
  * each run of 16 consecutive elements along the reduction dimension K
    (a "block") has one scale stored as an OCP E4M3 byte with the sign bit
    clear (unsigned E4M3, largest value 448);
  * each tensor has one fp32 scale g.

For a tensor x (fp32 values, blocks along its last axis), every step an IEEE
fp32 operation rounded to nearest even:
  g     = amax(x) / (6 * 448)        (1 if amax is 0; NaN elements ignored)
  d     = 6 * g
  sb    = E4M3(b / d)                b = max |x| over the block (NaN ignored),
                                     E4M3 round-to-nearest-even, saturating
  e     = dec(sb) * g                the block's dequant multiplier
  q_i   = E2M1(x_i / e)              round-to-nearest-even, saturating at +-6,
                                     sign kept for a value rounding to 0;
                                     0 when e == 0; NaN -> +0
  x_i  ~= dec(q_i) * dec(sb) * g

A GEMM on NVFP4 operands (both blocked along K) computes
  acc[m, n] = sum_k (dec(qa[m,k]) dec(sa[m,k/16])) (dec(qw[n,k]) dec(sw[n,k/16]))
  v         = acc * (ga * gw) + bias[n], then the GELU / bf16 epilogue.

All arithmetic below is fp64 on values that are exact fp32 numbers, with an
explicit rounding to fp32 after each step the definition rounds.
"""
import math

import numpy as np

from . import e4m3

E2M1_MAX = 6.0
BLOCK = 16


def decode_nibble(c):
    """Value of one E2M1 code (low 4 bits of c), fp64.

    sign s = bit 3, exponent field e = bits 2..1, mantissa m = bit 0:
      e == 0 : (-1)^s * m * 0.5                 (subnormal; m = 0 is zero)
      e >= 1 : (-1)^s * (1 + m / 2) * 2^(e - 1)
    """
    c = int(c) & 0xF
    s, e, m = c >> 3, (c >> 1) & 3, c & 1
    mag = m * 0.5 if e == 0 else (1.0 + m / 2.0) * 2.0 ** (e - 1)
    return -mag if s else mag


def decode_table():
    """fp64 array of the 16 code values."""
    return np.array([decode_nibble(c) for c in range(16)], dtype=np.float64)


_MAG_CODE = {0.0: 0, 0.5: 1, 1.0: 2, 1.5: 3, 2.0: 4, 3.0: 5, 4.0: 6, 6.0: 7}
_MAGS = np.array(sorted(_MAG_CODE), dtype=np.float64)


def encode_value(x):
    """E2M1 code of one fp32 value, by the steps of the definition.

    For a magnitude a below 6: the binade of a (or the subnormal range below
    1) has a spacing of quantum = 2^(e - 1) with e = max(floor(log2 a), 0);
    r = rint(a / quantum) * quantum, rint rounding half to even (an even
    multiple of the quantum is an even mantissa).  a >= 6 (infinity
    included) saturates to 6.  The sign is kept, a negative value rounding
    to zero included (code 0x8); NaN encodes as +0.
    """
    x = float(x)
    if math.isnan(x):
        return 0
    sign = 8 if math.copysign(1.0, x) < 0 else 0
    a = abs(x)
    if a >= E2M1_MAX:
        r = E2M1_MAX
    elif a == 0.0:
        r = 0.0
    else:
        e = max(math.floor(math.log2(a)), 0)
        q = 2.0 ** (e - 1)
        r = min(float(np.rint(a / q)) * q, E2M1_MAX)
    return sign | _MAG_CODE[r]


def encode(v):
    """E2M1 codes (uint8, 0..15) of fp32 values v: encode_value applied
    elementwise, written with array operations."""
    v = np.asarray(v, dtype=np.float64)
    nan = np.isnan(v)
    a = np.where(nan, 0.0, np.abs(v))
    with np.errstate(divide="ignore"):
        e = np.maximum(np.floor(np.log2(np.where(a > 0, a, 1.0))), 0.0)
    q = 2.0 ** (e - 1.0)
    with np.errstate(invalid="ignore"):
        r = np.minimum(np.rint(a / q) * q, E2M1_MAX)
    r = np.where(a >= E2M1_MAX, E2M1_MAX, np.where(a == 0.0, 0.0, r))
    code = np.searchsorted(_MAGS, r).astype(np.uint8)
    sign = np.where(np.signbit(v) & ~nan, 8, 0).astype(np.uint8)
    return (sign | code).astype(np.uint8)


def f32(x):
    """Round fp64 values to fp32 (nearest even) and back to fp64."""
    with np.errstate(over="ignore", invalid="ignore"):
        return np.asarray(x, dtype=np.float64).astype(np.float32).astype(np.float64)


def tensor_scale(x):
    """g = amax / (6 * 448) as fp32 (1 if amax is 0; NaN ignored)."""
    a = np.abs(np.asarray(x, dtype=np.float64))
    a = np.where(np.isnan(a), 0.0, a)
    amax = a.max() if a.size else 0.0
    if amax == 0.0:
        return np.float32(1.0)
    return np.float32(f32(amax / (E2M1_MAX * 448.0)))


def quantize(x, g=None):
    """NVFP4 of x [V x K] (fp32 values, K % 16 == 0, blocks along K).

    Returns (q uint8 [V x K] E2M1 codes, one per element; sb uint8
    [V x K / 16] E4M3 block-scale bytes; g fp32).  ``g`` overrides the
    tensor scale (a static scale)."""
    x = np.asarray(x, dtype=np.float32).astype(np.float64)
    V, K = x.shape
    assert K % BLOCK == 0
    g = tensor_scale(x) if g is None else np.float32(g)
    gd = np.float64(g)
    d = f32(6.0 * gd)
    blocks = x.reshape(V, K // BLOCK, BLOCK)
    a = np.abs(blocks)
    a = np.where(np.isnan(a), 0.0, a)
    bmax = a.max(axis=2)
    with np.errstate(divide="ignore", invalid="ignore"):
        sb = e4m3.encode(np.where(d > 0, f32(bmax / d), 0.0).astype(np.float32), e4m3.OCP)
    sbv = e4m3.decode_table(e4m3.OCP)[sb]
    e = f32(sbv * gd)  # [V x K/16]
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = np.where(e[:, :, None] > 0, f32(blocks / e[:, :, None]), 0.0)
    q = encode(ratio).reshape(V, K)
    # a block whose multiplier is 0 (all-zero block, or a block scale that
    # rounds to 0) encodes as +0
    q = np.where(np.repeat(e, BLOCK, axis=1) > 0, q, 0).astype(np.uint8)
    return q, sb.astype(np.uint8), np.float32(g)


def dequantize(q, sb, g):
    """dec(q) * dec(sb) * g in fp64, [V x K]."""
    t = decode_table()[np.asarray(q) & 0xF]
    s = np.repeat(e4m3.decode_table(e4m3.OCP)[np.asarray(sb)], BLOCK, axis=1)
    return t * s * np.float64(g)


def tile_scales(sb):
    """Block scales sb [V x K/16] in the tiled layout the GEMM reads: vectors
    padded with zero scales to a multiple of 128; per group of 128 vectors
    and 4 blocks (64 elements of K) one 512-byte atom of 32 lines x 16 bytes,
    line i holding vectors i, i + 32, i + 64, i + 96 (4 bytes each, blocks in
    order); atoms ordered by vector group, then by K.  Returns a flat uint8
    array."""
    sb = np.asarray(sb, dtype=np.uint8)
    V, nb = sb.shape
    assert nb % 4 == 0
    vp = -(-V // 128) * 128
    pad = np.zeros((vp, nb), dtype=np.uint8)
    pad[:V] = sb
    # [group g][quarter j][line i][chunk c][block t] -> [g][c][i][j][t]
    t = pad.reshape(vp // 128, 4, 32, nb // 4, 4)
    return np.ascontiguousarray(t.transpose(0, 3, 2, 1, 4)).reshape(-1)


def pack_nibbles(q):
    """Two codes per byte along K: element 2j in the low nibble of byte j."""
    q = np.asarray(q, dtype=np.uint8)
    return (q[:, 0::2] & 0xF) | ((q[:, 1::2] & 0xF) << 4)


def unpack_nibbles(p):
    p = np.asarray(p, dtype=np.uint8)
    out = np.empty((p.shape[0], p.shape[1] * 2), dtype=np.uint8)
    out[:, 0::2] = p & 0xF
    out[:, 1::2] = p >> 4
    return out


def gemm(qa, sa, ga, qw, sw, gw, bias=None, act_cols=0):
    """NVFP4 GEMM: qa [M x K], qw [N x K] codes (both blocked along K), sa
    [M x K/16], sw [N x K/16] block-scale bytes, ga, gw tensor scales.
    Returns (v fp64 [M x N] after scale, bias and GELU on the first act_cols
    columns, sumabs = ga gw sum_k |a w| for the tolerance)."""
    from .gemm import gelu_tanh

    a = decode_table()[qa] * np.repeat(e4m3.decode_table(e4m3.OCP)[sa], BLOCK, axis=1)
    w = decode_table()[qw] * np.repeat(e4m3.decode_table(e4m3.OCP)[sw], BLOCK, axis=1)
    acc = a @ w.T
    s = np.float64(ga) * np.float64(gw)
    v = acc * s
    if bias is not None:
        v = v + np.asarray(bias, dtype=np.float64)[None, :]
    if act_cols:
        v[:, :act_cols] = gelu_tanh(v[:, :act_cols])
    return v, np.abs(a) @ np.abs(w).T * abs(s)
