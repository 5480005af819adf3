"""Oracle: the quantized linear layer, fp64 (test infrastructure only).

Computes Y = act(s_a * s_w[n] * sum_k a[m,k] * w[k,n] + b[n]) on the
decoded values in fp64, with

  * a, w the E4M3 bytes decoded (FP8 path) or the bf16 values (BF16 path);
  * s_a the per-tensor activation scale (1 on the BF16 path), s_w[n] the
    per-output-channel weight scale (1 when absent), b[n] the fp32 bias
    (0 when absent) -- the bias is applied in the GEMM epilogue ("Real-time
    VLA inference on AMD hardware", section "Merging gate and up");
  * act the tanh-approximate GELU, 0.5 v (1 + tanh(sqrt(2/pi) (v + 0.044715
    v^3))), on the output columns n < act_cols and the identity on the rest.
    A merged gate/up weight [W_gate, W_up] (concatenated along N, same
    section) applies GELU to the gate columns [0, N/2) only.

Epilogue order (a reading; the pages do not fix it): scale, then bias, then
GELU.  The result stays fp64; the final bf16 store is the kernel's rounding,
covered by the comparison tolerance.

The product sum uses numpy's fp64 matmul (BLAS dgemm) as a library primitive;
``gemm_naive`` is the plain triple loop for tiny shapes.  ``geglu`` is the
fused GeGLU of a merged gate/up layer, applied to the layer's output without
activation.
"""
import math

import numpy as np

from . import e4m3

SQRT_2_OVER_PI = math.sqrt(2.0 / math.pi)


def gelu_tanh(v):
    """tanh-approximate GELU in fp64."""
    v = np.asarray(v, dtype=np.float64)
    return 0.5 * v * (1.0 + np.tanh(SQRT_2_OVER_PI * (v + 0.044715 * v * v * v)))


def epilogue(acc, col_scale, bias, act_cols):
    """v = acc * col_scale[n] + bias[n]; GELU on columns n < act_cols."""
    v = np.asarray(acc, dtype=np.float64) * np.asarray(col_scale, dtype=np.float64)[None, :]
    if bias is not None:
        v = v + np.asarray(bias, dtype=np.float64)[None, :]
    if act_cols:
        v[:, :act_cols] = gelu_tanh(v[:, :act_cols])
    return v


def _col_scale(N, a_scale, w_scale):
    s = np.full(N, 1.0 if a_scale is None else float(np.float32(a_scale)), dtype=np.float64)
    if w_scale is not None:
        s = s * np.asarray(w_scale, dtype=np.float32).astype(np.float64)
    return s


def gemm_values(a, w, a_scale=None, w_scale=None, bias=None, act_cols=0):
    """The layer on already decoded fp64 operands a [M x K], w [K x N].

    Returns (y [M x N] fp64, sumabs [M x N] fp64) where sumabs is
    s_a * s_w[n] * sum_k |a[m,k] * w[k,n]|, the magnitude the tolerance of a
    floating-point sum is measured against.
    """
    a = np.asarray(a, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    N = w.shape[1]
    cs = _col_scale(N, a_scale, w_scale)
    acc = a @ w
    y = epilogue(acc, cs, bias, act_cols)
    sumabs = (np.abs(a) @ np.abs(w)) * np.abs(cs)[None, :]
    return y, sumabs


def gemm_fp8(qa, a_fmt, a_scale, qw, w_fmt, w_scale, bias=None, act_cols=0):
    """FP8 layer: E4M3 activation bytes qa [M x K] (per-tensor scale) times
    E4M3 weight bytes qw [K x N] (per-column scales)."""
    return gemm_values(e4m3.decode(qa, a_fmt), e4m3.decode(qw, w_fmt), a_scale, w_scale,
                       bias, act_cols)


def gemm_bf16(a_f32, w_f32, w_scale=None, bias=None, act_cols=0):
    """BF16 layer on bf16 values given as fp32 arrays (exact)."""
    return gemm_values(a_f32, w_f32, None, w_scale, bias, act_cols)


def gelu_tanh_prime(v):
    """Derivative of the tanh-approximate GELU, in closed form (fp64):
    0.5 (1 + t) + 0.5 v (1 - t^2) sqrt(2/pi) (1 + 3 * 0.044715 v^2) with
    t = tanh(sqrt(2/pi) (v + 0.044715 v^3))."""
    v = np.asarray(v, dtype=np.float64)
    t = np.tanh(SQRT_2_OVER_PI * (v + 0.044715 * v * v * v))
    return 0.5 * (1.0 + t) + 0.5 * v * (1.0 - t * t) * SQRT_2_OVER_PI * (
        1.0 + 3.0 * 0.044715 * v * v)


def geglu(y, sumabs):
    """GeGLU of a merged gate/up layer ("Real-time VLA inference on AMD
    hardware", section "Merging gate and up": one GEMM over [W_gate, W_up],
    the gate's channels first): with y [M x N] the layer's output before any
    activation (fp64) and F = N / 2,

        h[m, j] = gelu_tanh(y[m, j]) * y[m, F + j],   0 <= j < F.

    Returns (h [M x F], prop [M x F]): prop carries the magnitudes the
    layer's sums are measured against through the product to first order,
    |gelu_tanh'(g)| |u| sumabs_gate + |gelu_tanh(g)| sumabs_up, the
    magnitude h's tolerance is measured against.
    """
    y = np.asarray(y, dtype=np.float64)
    F = y.shape[1] // 2
    g, u = y[:, :F], y[:, F:]
    h = gelu_tanh(g) * u
    prop = (np.abs(gelu_tanh_prime(g)) * np.abs(u) * sumabs[:, :F] +
            np.abs(gelu_tanh(g)) * sumabs[:, F:])
    return h, prop


def gemm_naive(a, w):
    """sum_k a[m,k] * w[k,n] by the plain triple loop (tiny shapes only)."""
    a = np.asarray(a, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    M, K = a.shape
    N = w.shape[1]
    out = np.zeros((M, N), dtype=np.float64)
    for m in range(M):
        for n in range(N):
            s = 0.0
            for k in range(K):
                s += a[m, k] * w[k, n]
            out[m, n] = s
    return out
