"""Oracle: E4M3 quantization of a tensor (test infrastructure only).

FP8 quantization as the method uses it: a scale is taken from the absolute
maximum of the tensor (per tensor for activations, per output channel for
weights), every element is divided by the scale and encoded to E4M3 with
round-to-nearest-even and saturation.  Weights are quantized once at load
("It quantizes and packs the weights", "Real-time VLA inference on AMD
hardware", section "How FlashRT works"); on CDNA3 they are produced in FNUZ
(section "Different FP8 representation").

Readings where the pages are silent:
  * the scale is the dequantization multiplier, x ~= decode(q) * s, with
    s = amax / max_finite (448 OCP, 240 FNUZ) rounded once to fp32;
  * amax == 0 gives s = 1;
  * amax ignores NaN elements (a NaN element still encodes to the NaN code);
  * the element is divided by the scale (IEEE fp32 division, correctly
    rounded), not multiplied by a reciprocal;
  * per-column mode takes one scale for each column c of a [rows x cols]
    tensor, the max over its rows (the output channel n of W[K x N]).

fp64 division rounded once to fp32 equals the correctly rounded fp32
division, because 53 >= 2 * 24 + 2.
"""
import numpy as np

from . import e4m3

PER_TENSOR = "per_tensor"
PER_COL = "per_col"


def amax(x, mode):
    """Max |x| over the tensor (per tensor) or over rows for each column, fp64.

    NaN elements are ignored (fmax reduction); an all-NaN reduction gives 0.
    """
    a = np.abs(np.asarray(x, dtype=np.float64))
    a = np.where(np.isnan(a), 0.0, a)
    if mode == PER_TENSOR:
        return np.float64(a.max()) if a.size else np.float64(0.0)
    return a.max(axis=0) if a.shape[0] else np.zeros(a.shape[1])


def scale_from_amax(am, fmt):
    """fp32 scale amax / max_finite, correctly rounded; 1 where amax == 0."""
    am = np.asarray(am, dtype=np.float64)
    with np.errstate(over="ignore"):
        s = (am / e4m3.params(fmt)["max"]).astype(np.float32)
    return np.where(am == 0.0, np.float32(1.0), s).astype(np.float32)


def divide_f32(x, s):
    """Correctly rounded fp32 quotient x / s (fp64 division, one rounding)."""
    with np.errstate(over="ignore", invalid="ignore", divide="ignore"):
        return (np.asarray(x, dtype=np.float64) / np.asarray(s, dtype=np.float64)).astype(
            np.float32
        )


def quantize_e4m3(x, mode, fmt, static_scale=None):
    """Quantize x (fp32 values, 2-D [rows x cols]) to E4M3 bytes.

    Returns (q uint8 [rows x cols], scale fp32: shape () per tensor or
    (cols,) per column).  With ``static_scale`` the amax step is skipped and
    the given scale is used as is.
    """
    x = np.asarray(x, dtype=np.float32)
    if static_scale is None:
        s = scale_from_amax(amax(x, mode), fmt)
    else:
        s = np.asarray(static_scale, dtype=np.float32)
    if mode == PER_TENSOR:
        s = np.float32(s.reshape(()))
        y = divide_f32(x, s)
    else:
        s = s.reshape(-1)
        y = divide_f32(x, s[None, :])
    return e4m3.encode(y, fmt), s
