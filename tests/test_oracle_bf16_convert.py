"""Pins for the oracle's bf16 rounding and FNUZ -> OCP re-encoding."""
import math
import os

import numpy as np
import torch

from oracle import bf16, convert, e4m3

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "fnuz_to_ocp_cases.txt")


def test_bf16_rne_matches_torch():
    # library cross-check: PyTorch's CPU float32 -> bfloat16 cast is RNE
    g = np.random.default_rng(5)
    x = np.concatenate([
        g.standard_normal(50000).astype(np.float32),
        np.float32(2.0 ** g.uniform(-140, 127, 20000)),
        np.array([0.0, -0.0, np.inf, -np.inf, 3.4e38, 1e-45, -1e-40], dtype=np.float32),
    ])
    # exact ties: low 16 bits = 0x8000, with the kept LSB both even and odd
    u = (g.integers(0, 2 ** 15, 4000, dtype=np.uint32) << 16) | 0x8000
    x = np.concatenate([x, u.view(np.float32), (u | 0x80000000).view(np.float32)])
    ours = bf16.f32_to_bf16_bits(x)
    lib = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    fin = ~np.isnan(x)
    np.testing.assert_array_equal(ours[fin], lib[fin])
    assert np.isnan(bf16.bf16_bits_to_f32(bf16.f32_to_bf16_bits(np.float32([np.nan])))).all()


def test_bf16_tie_cases_by_hand():
    # 1 + 2^-8 is halfway between 1.0 and 1 + 2^-7: ties to 1.0 (even)
    # 1 + 3 * 2^-8 is halfway between 1 + 2^-7 and 1 + 2^-6: ties to 1 + 2^-6
    x = np.float32([1 + 2 ** -8, 1 + 3 * 2 ** -8, 1 + 2 ** -8 + 2 ** -20])
    np.testing.assert_array_equal(bf16.round_to_bf16(x),
                                  np.float32([1.0, 1 + 2 ** -6, 1 + 2 ** -7]))


def rule_fnuz_to_ocp(b):
    """Rule-based derivation, independent of the codec: FNUZ bias 8 vs OCP
    bias 7.  Exponent field e >= 2 -> same sign and mantissa, field e - 1.
    Field 0 or 1: value v * 2^-10 with v = (e << 3) | m in 0..15, which is
    v / 2 OCP subnormal quanta: round half to even, keep the sign."""
    if b == 0x80:
        return 0x7F
    s = b & 0x80
    e = (b >> 3) & 0xF
    if e >= 2:
        return b - 0x08
    v = b & 0x0F
    r = v // 2
    if v % 2 == 1 and r % 2 == 1:
        r += 1
    return s | r


def test_fnuz_to_ocp_against_rules():
    table = convert.fnuz_to_ocp_table()
    for b in range(256):
        assert table[b] == rule_fnuz_to_ocp(b), hex(b)


def test_fnuz_to_ocp_golden_cases():
    table = convert.fnuz_to_ocp_table()
    n = 0
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            a, b = line.split()[:2]
            assert table[int(a, 16)] == int(b, 16), line
            n += 1
    assert n == 20


def test_fnuz_to_ocp_value_preserving_where_representable():
    table = convert.fnuz_to_ocp_table()
    inexact = []
    for b in range(256):
        z = e4m3.decode_byte(b, e4m3.FNUZ)
        o = e4m3.decode_byte(int(table[b]), e4m3.OCP)
        if math.isnan(z):
            assert math.isnan(o)
        elif z != o:
            inexact.append(b)
    # 8 magnitudes (fields 0/1 with odd mantissa), each with two signs
    mags = sorted({b & 0x7F for b in inexact})
    assert mags == [0x01, 0x03, 0x05, 0x07, 0x09, 0x0B, 0x0D, 0x0F]
    assert len(inexact) == 16


def test_fnuz_to_ocp_array():
    data = np.arange(256, dtype=np.uint8).repeat(3)
    np.testing.assert_array_equal(convert.fnuz_to_ocp(data),
                                  np.array([rule_fnuz_to_ocp(b) for b in data], dtype=np.uint8))
