"""Oracle: the BF16 decoder block boundary (test infrastructure only).

"Real-time VLA inference on AMD hardware", section "Fusing the BF16 decoder
boundary": between decoder blocks the graph updates the residual stream,
residual = BF16(residual + output x gate), and then takes an adaptive RMS
norm of it, normalized, next_gate = adaptive_rms_norm(residual, style).  The
page gives no formula for the norm; the plainest reading, taken here, reads
the style row as three H-wide parts [scale | shift | next gate] and

    normalized = rms_norm(r) * (1 + scale) + shift,
    rms_norm(r) = r / sqrt(mean(r^2) + eps),

with the next block's gate passed on unchanged.  The residual update is
computed the way the kernel's fp32 arithmetic defines it: the exact value of
residual + output * gate (bf16 operands, exact in fp64), rounded once to fp32
and then to bf16.  The norm is evaluated in fp64 and not rounded; the kernel's
bf16 store and fp32 sums are covered by the comparison tolerance.
"""
import numpy as np

from . import bf16


def gate_residual_ada_norm(residual, output, gate, style, eps):
    """residual, output, gate [M x H] and style [M x 3H] as fp32 arrays of
    bf16 values.  Returns (r, normalized, next_gate, mag): r [M x H] the
    updated residual (fp32 values of bf16), normalized [M x H] fp64,
    next_gate [M x H] and mag = |r * inv * (1 + scale)| + |shift|, the
    magnitude the tolerance of normalized is measured against."""
    residual = np.asarray(residual, dtype=np.float64)
    output = np.asarray(output, dtype=np.float64)
    gate = np.asarray(gate, dtype=np.float64)
    style = np.asarray(style, dtype=np.float64)
    H = residual.shape[1]
    upd = (residual + output * gate).astype(np.float32)  # one rounding to fp32
    r = bf16.round_to_bf16(upd).astype(np.float64)       # then to bf16
    scale, shift, nxt = style[:, :H], style[:, H:2 * H], style[:, 2 * H:]
    inv = 1.0 / np.sqrt(np.mean(r * r, axis=1, keepdims=True) + float(np.float32(eps)))
    t = r * inv * (1.0 + scale)
    return r, t + shift, nxt, np.abs(t) + np.abs(shift)
