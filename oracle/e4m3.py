"""Oracle: E4M3 bytes in the OCP and FNUZ dialects (test infrastructure only).

Both dialects use one sign bit, four exponent bits and three mantissa bits in
the same positions.  They differ in the exponent bias and in the special
codes:

  * OCP E4M3 (OFP8 specification): bias 7; subnormals at exponent field 0;
    S.1111.111 (0x7F, 0xFF) is NaN; no infinity; +0 and -0 both exist;
    largest finite value 0x7E = 2^8 * 1.75 = 448.
  * FNUZ E4M3 ("finite, NaNs, unsigned zero"): bias 8, i.e. the exponent
    bias is off by one against OCP, so the same byte decodes to half its OCP
    value ("Real-time VLA inference on AMD hardware", section "Different FP8
    representation"; "Deploying DeepSeek-V4-Flash on AMD MI300X", section
    "The FP8 dialect problem").  There is no -0 and no infinity; the byte
    0x80 (the would-be -0) is the only NaN, so 0x7F = 2^7 * 1.875 = 240 is
    the largest finite value.

Encoding is round-to-nearest-even with saturation ("satfinite"): NaN goes to
the dialect's NaN code, any magnitude at or above the largest finite value
(infinity included) goes to the signed largest finite value.  A value that
rounds to zero keeps its sign in OCP (0x80) and becomes 0x00 in FNUZ, which
has no negative zero.

All arithmetic is done in fp64 on values that are exact fp32 numbers, so
every intermediate step below is exact.
"""
import math

import numpy as np

OCP = "ocp"
FNUZ = "fnuz"

# bias, largest finite magnitude, its code, the NaN code
_PARAMS = {
    OCP: dict(bias=7, max=448.0, max_code=0x7E, nan_code=0x7F),
    FNUZ: dict(bias=8, max=240.0, max_code=0x7F, nan_code=0x80),
}


def params(fmt):
    """Bias, largest finite magnitude, its byte and the NaN byte of a dialect."""
    return _PARAMS[fmt]


def is_nan_code(b, fmt):
    """True if byte ``b`` is NaN in the dialect."""
    if fmt == OCP:
        return (b & 0x7F) == 0x7F
    return b == 0x80


def decode_byte(b, fmt):
    """Value of one E4M3 byte, as an fp64 (NaN for the NaN codes).

    sign s = bit 7, exponent field e = bits 6..3, mantissa m = bits 2..0:
      e == 0 : (-1)^s * (m / 8) * 2^(1 - bias)      (subnormal, m = 0 is zero)
      e >= 1 : (-1)^s * (1 + m / 8) * 2^(e - bias)
    """
    b = int(b) & 0xFF
    if is_nan_code(b, fmt):
        return math.nan
    bias = _PARAMS[fmt]["bias"]
    s = b >> 7
    e = (b >> 3) & 0xF
    m = b & 0x7
    if e == 0:
        mag = (m / 8.0) * 2.0 ** (1 - bias)
    else:
        mag = (1.0 + m / 8.0) * 2.0 ** (e - bias)
    return -mag if s else mag


def decode_table(fmt):
    """fp64 array of 256 entries: the value of every byte."""
    return np.array([decode_byte(b, fmt) for b in range(256)], dtype=np.float64)


_TABLES = {}


def decode(q, fmt):
    """Decode an array of bytes to fp64 values."""
    if fmt not in _TABLES:
        _TABLES[fmt] = decode_table(fmt)
    return _TABLES[fmt][np.asarray(q, dtype=np.uint8)]


def _round_half_even(v):
    """Round an fp64 to the nearest integer, ties to even (exact for |v| < 2^52)."""
    f = math.floor(v)
    d = v - f
    if d > 0.5:
        return f + 1
    if d < 0.5:
        return f
    return f if f % 2 == 0 else f + 1


def _code_of_magnitude(r, fmt):
    """Byte (without sign) of an exactly representable nonnegative magnitude."""
    bias = _PARAMS[fmt]["bias"]
    emin = 1 - bias
    if r == 0.0:
        return 0
    if r < 2.0 ** emin:  # subnormal: r = m * 2^(emin - 3)
        m = r / 2.0 ** (emin - 3)
        assert m == int(m) and 0 < m < 8
        return int(m)
    _, ex = math.frexp(r)  # r = f * 2^ex, f in [0.5, 1)
    e = ex - 1
    m = (r / 2.0 ** e - 1.0) * 8.0
    assert m == int(m) and 0 <= m < 8
    return ((e + bias) << 3) | int(m)


def encode_value(x, fmt):
    """E4M3 byte of one fp32 value (given as a Python float), RNE + saturate.

    Steps:
      1. NaN -> the dialect's NaN code.
      2. |x| >= largest finite value (infinity included) -> signed maximum.
      3. Otherwise the exponent of |x|, clamped below at the smallest normal
         exponent, fixes the spacing q = 2^(e - 3) of the codes around |x|;
         r = round_half_even(|x| / q) * q.  |x| / q is a power-of-two
         scaling, so it is exact, and so is r.
      4. Emit the code of r with the sign of x; a negative value that rounds
         to zero is 0x80 (-0) in OCP and 0x00 in FNUZ.
    """
    p = _PARAMS[fmt]
    x = float(x)
    if math.isnan(x):
        return p["nan_code"]
    neg = math.copysign(1.0, x) < 0
    a = abs(x)
    if a >= p["max"]:
        code = p["max_code"]
    else:
        emin = 1 - p["bias"]
        if a == 0.0:
            r = 0.0
        else:
            _, ex = math.frexp(a)
            e = max(ex - 1, emin)
            q = 2.0 ** (e - 3)
            r = _round_half_even(a / q) * q
        if r > p["max"]:
            r = p["max"]
        code = _code_of_magnitude(r, fmt)
    if neg:
        if code == 0:
            return 0x80 if fmt == OCP else 0x00
        return code | 0x80
    return code


def encode(x, fmt):
    """Vectorised E4M3 encode of an array of fp32 values -> uint8 array.

    Same rule as :func:`encode_value`, written for arrays.  For a magnitude a
    below the maximum, with e = max(floor(log2 a), emin) and n = the number
    of spacings 2^(e-3) in a rounded half-to-even, the magnitude code is
    (e - emin) * 8 + n: in the subnormal binade e = emin and the code is n;
    in a normal binade n runs from 8 to 16 and (e - emin) * 8 + n equals
    ((e + bias) << 3) | (n - 8), with n = 16 carrying into the next binade.
    """
    p = _PARAMS[fmt]
    with np.errstate(invalid="ignore", over="ignore"):
        x = np.asarray(x, dtype=np.float32).astype(np.float64)
    nan = np.isnan(x)
    neg = np.signbit(x)
    a = np.abs(np.where(nan, 0.0, x))
    sat = a >= p["max"]
    emin = 1 - p["bias"]
    with np.errstate(invalid="ignore", over="ignore"):
        am = np.where(sat, 0.0, a)
        _, ex = np.frexp(am)
        e = np.maximum(ex.astype(np.int64) - 1, emin)
        n = np.rint(am / np.ldexp(1.0, (e - 3).astype(np.int32)))
        code = (e - emin) * 8 + n.astype(np.int64)
        code = np.where(am == 0.0, 0, code)
        code = np.minimum(code, p["max_code"])
    code = np.where(sat, p["max_code"], code)
    signed = np.where(neg, code | 0x80, code)
    if fmt == OCP:
        out = signed  # -0 stays 0x80
    else:
        out = np.where(neg & (code == 0), 0x00, signed)
    out = np.where(nan, p["nan_code"], out)
    return out.astype(np.uint8)
