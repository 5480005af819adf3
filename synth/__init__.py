"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle checks.

This module only draws random numbers and casts them to the input dtypes
(fp32, or bf16 through PyTorch's CPU cast); it holds none of the method's
arithmetic.  Every generator is deterministic in its seed; the draw order is
stated in each docstring so the streams can be reproduced.

bf16 arrays are returned as uint16 bit patterns (NumPy has no bf16 type).

Workloads (shapes and distributions of a pi0.5-style small-batch VLA
forward pass, "Real-time VLA inference on AMD hardware", section "FP8 helps
the encoder and hurts the decoder": an encoder GEMM with hundreds of rows and
an action-decoder GEMM with a few dozen rows):

  * tiny     -- A bf16 [16 x 512] ~ N(0,1), W fp32 [512 x 256] ~ N(0, 0.02),
                bias fp32 [256] ~ N(0, 0.1); seed 0.
  * decoder  -- M = 50, hidden 1024: (K, N) = (1024, 2048), (1024, 4096)
                gate with GELU, (1024, 4096) up, (4096, 1024) down.
  * encoder  -- M = 768: (2048, 2560), (2048, 16384), (16384, 2048); the
                activations carry 1% outlier entries scaled by 50.
  * stack    -- 18 encoder layers (M = 768, hidden 2048) and 18 decoder
                layers (M = 50, hidden 1024), seed 1.
  * sweeps   -- M in {1 ... 1024} at K = N = 4096; a uniform byte stream;
                Student-t (nu = 3) bf16 values.
"""
import numpy as np
import torch

DECODER_LAYERS = (  # (name, K, N, act)
    ("qkv", 1024, 2048, False),
    ("gate", 1024, 4096, True),
    ("up", 1024, 4096, False),
    ("down", 4096, 1024, False),
)
ENCODER_LAYERS = (
    ("qkv", 2048, 2560, False),
    ("gate_up", 2048, 16384, False),
    ("down", 16384, 2048, False),
)
SWEEP_M = (1, 2, 4, 8, 16, 32, 50, 64, 128, 256, 512, 768, 1024)

# stack: per layer (name, K, N, act_cols) -- merged gate/up with GELU on the gate half
STACK_ENCODER = (
    ("qkv", 2048, 2560, 0),
    ("o", 2048, 2048, 0),
    ("gate_up", 2048, 2 * 16384, 16384),
    ("down", 16384, 2048, 0),
)
STACK_DECODER = (
    ("qkv", 1024, 2560, 0),
    ("o", 2048, 1024, 0),
    ("gate_up", 1024, 2 * 4096, 4096),
    ("down", 4096, 1024, 0),
)


def rng(seed):
    return np.random.default_rng(seed)


def to_bf16_bits(x):
    """fp32/fp64 array -> bf16 bit patterns (uint16) via PyTorch's CPU cast."""
    t = torch.from_numpy(np.ascontiguousarray(np.asarray(x, dtype=np.float32)))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()


def bf16_bits_as_f32(b):
    """bf16 bit patterns -> fp32 values via PyTorch's CPU cast."""
    t = torch.from_numpy(np.ascontiguousarray(np.asarray(b, dtype=np.uint16)).view(np.int16))
    return t.view(torch.bfloat16).to(torch.float32).numpy()


def normal_f32(g, shape, std):
    return (g.standard_normal(shape) * std).astype(np.float32)


def activations(g, M, K, outlier_frac=0.0, outlier_mult=50.0):
    """A ~ N(0,1) as bf16 bits; optionally a fraction of entries (chosen by a
    uniform draw < outlier_frac, drawn after the normals) multiplied."""
    a = g.standard_normal((M, K))
    if outlier_frac:
        mask = g.random((M, K)) < outlier_frac
        a = np.where(mask, a * outlier_mult, a)
    return to_bf16_bits(a)


def layer(g, M, K, N, act_cols=0, outlier_frac=0.0, w_std=0.02, b_std=0.1):
    """One linear layer's inputs.  Draw order: A (then its outlier mask),
    W [K x N] ~ N(0, w_std), bias [N] ~ N(0, b_std)."""
    a = activations(g, M, K, outlier_frac)
    w = normal_f32(g, (K, N), w_std)
    b = normal_f32(g, (N,), b_std)
    return dict(M=M, K=K, N=N, act_cols=act_cols, a_bf16=a, w_f32=w, bias=b)


def tiny(seed=0):
    """A bf16 [16 x 512] ~ N(0,1); W fp32 [512 x 256] ~ N(0, 0.02); bias
    fp32 [256] ~ N(0, 0.1); GELU on every column."""
    g = rng(seed)
    return layer(g, 16, 512, 256, act_cols=256)


def decoder(seed=0, M=50):
    """Decoder-shaped layers at M rows, drawn in DECODER_LAYERS order."""
    g = rng(seed)
    return [dict(layer(g, M, K, N, act_cols=N if act else 0), name=name)
            for name, K, N, act in DECODER_LAYERS]


def encoder(seed=0, M=768):
    """Encoder-shaped layers at M rows with 1% x50 activation outliers."""
    g = rng(seed)
    return [dict(layer(g, M, K, N, act_cols=N if act else 0, outlier_frac=0.01), name=name)
            for name, K, N, act in ENCODER_LAYERS]


def stack_weights(seed=1, layers=18):
    """Weights and biases of the synthetic stack, encoder layers first, then
    decoder layers; per layer W [K x N] ~ N(0, 0.02) then bias ~ N(0, 0.1)."""
    g = rng(seed)
    out = {"encoder": [], "decoder": []}
    for part, spec in (("encoder", STACK_ENCODER), ("decoder", STACK_DECODER)):
        for _ in range(layers):
            out[part].append([dict(name=n, K=K, N=N, act_cols=ac,
                                   w_f32=normal_f32(g, (K, N), 0.02),
                                   bias=normal_f32(g, (N,), 0.1))
                              for n, K, N, ac in spec])
    return out


def stack_inputs(seed=1):
    """The stack's two input activations: encoder [768 x 2048] then decoder
    [50 x 1024], both ~ N(0,1) bf16 (drawn from seed + 1000)."""
    g = rng(seed + 1000)
    return activations(g, 768, 2048), activations(g, 50, 1024)


def sweep_gemm(M, seed=0, K=4096, N=4096):
    """Sweep (i) layer at M rows, K = N = 4096."""
    return layer(rng(seed), M, K, N)


def uniform_bytes(n, seed=2):
    """n uniform random bytes (every value, 0x80 and subnormal codes included)."""
    return rng(seed).integers(0, 256, size=n, dtype=np.uint8)


def student_t_bf16(n, seed=3, nu=3):
    """n bf16 values from a Student-t distribution with nu degrees of freedom."""
    return to_bf16_bits(rng(seed).standard_t(nu, size=n))
