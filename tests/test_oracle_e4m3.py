"""Pins for the oracle's E4M3 codec, checked against what the format
definitions and the pages fix, not against the oracle itself.

* hand-typed byte values (tests/golden/e4m3_values.txt);
* the 2x relation between the dialects ("Real-time VLA inference on AMD
  hardware", section "Different FP8 representation");
* FNUZ has no -0 and no infinity ("Deploying DeepSeek-V4-Flash on AMD
  MI300X", section "The FP8 dialect problem");
* encode against a brute-force nearest-code search, ties to the even code;
* a library cross-check against PyTorch's float8 dtypes.
"""
import math
import os

import numpy as np
import pytest
import torch

from oracle import e4m3

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "e4m3_values.txt")


def _parse(v):
    if v == "nan":
        return math.nan
    if v == "-0":
        return -0.0
    return float(v)


def golden_rows():
    rows = []
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            b, o, z = line.split()
            rows.append((int(b, 16), _parse(o), _parse(z)))
    return rows


def same(a, b):
    if math.isnan(b):
        return math.isnan(a)
    return a == b and math.copysign(1, a) == math.copysign(1, b)


@pytest.mark.parametrize("b,ocp,fnuz", golden_rows())
def test_golden_values(b, ocp, fnuz):
    assert same(e4m3.decode_byte(b, e4m3.OCP), ocp)
    assert same(e4m3.decode_byte(b, e4m3.FNUZ), fnuz)


def test_fnuz_is_half_of_ocp():
    checked = 0
    for b in range(256):
        o = e4m3.decode_byte(b, e4m3.OCP)
        z = e4m3.decode_byte(b, e4m3.FNUZ)
        if math.isnan(o) or math.isnan(z) or o == 0 or z == 0:
            continue
        assert z == o / 2, hex(b)
        checked += 1
    # all bytes but 0x00, 0x80 and the OCP NaNs 0x7f / 0xff
    assert checked == 252


def test_special_codes():
    ocp = e4m3.decode_table(e4m3.OCP)
    fnuz = e4m3.decode_table(e4m3.FNUZ)
    assert [b for b in range(256) if math.isnan(ocp[b])] == [0x7F, 0xFF]
    assert [b for b in range(256) if math.isnan(fnuz[b])] == [0x80]
    assert np.nanmax(ocp) == 448.0 and np.nanmin(ocp) == -448.0
    assert np.nanmax(fnuz) == 240.0 and np.nanmin(fnuz) == -240.0
    assert not np.isinf(ocp).any() and not np.isinf(fnuz).any()
    # FNUZ: unsigned zero -- exactly one byte is zero and none is -0
    zeros = [b for b in range(256) if fnuz[b] == 0]
    assert zeros == [0x00]
    # OCP keeps both zeros
    assert [b for b in range(256) if ocp[b] == 0] == [0x00, 0x80]
    assert math.copysign(1, ocp[0x80]) < 0
    # 127 distinct positive finite values in FNUZ, 126 in OCP
    assert len({v for v in fnuz if v > 0}) == 127
    assert len({v for v in ocp if v > 0}) == 126


def test_decode_matches_torch_float8():
    # library cross-check: PyTorch's float8_e4m3fn is OCP E4M3, float8_e4m3fnuz is FNUZ
    allb = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    for fmt, dt in ((e4m3.OCP, torch.float8_e4m3fn), (e4m3.FNUZ, torch.float8_e4m3fnuz)):
        lib = allb.view(dt).to(torch.float64).numpy()
        ours = e4m3.decode_table(fmt)
        np.testing.assert_array_equal(np.isnan(lib), np.isnan(ours))
        m = ~np.isnan(ours)
        np.testing.assert_array_equal(lib[m], ours[m])
        np.testing.assert_array_equal(np.signbit(lib[m]), np.signbit(ours[m]))


def brute_force_encode(x, fmt):
    """Definition of RNE-with-saturation by exhaustive search: the finite
    code nearest to x, the even code (mantissa bit 0 clear) on a tie; NaN to
    the NaN code; |x| >= max to the signed maximum."""
    p = e4m3.params(fmt)
    if math.isnan(x):
        return p["nan_code"]
    neg = math.copysign(1.0, x) < 0
    a = abs(x)
    if a >= p["max"]:
        return p["max_code"] | (0x80 if neg else 0)
    best = None
    for c in range(0x80):  # nonnegative codes
        v = e4m3.decode_byte(c, fmt)
        if math.isnan(v):
            continue
        d = abs(v - a)
        if best is None or d < best[0] or (d == best[0] and c % 2 == 0):
            best = (d, c)
    c = best[1]
    if neg:
        if c == 0:
            return 0x80 if fmt == e4m3.OCP else 0x00
        return c | 0x80
    return c


def probe_values():
    """Code values, midpoints between adjacent codes, and their fp32
    neighbours; a log-uniform random spread; specials."""
    vals = set()
    for fmt in (e4m3.OCP, e4m3.FNUZ):
        t = e4m3.decode_table(fmt)
        pos = np.unique(t[(t >= 0) & ~np.isnan(t)])
        mids = (pos[1:] + pos[:-1]) / 2
        for v in np.concatenate([pos, mids, [pos[-1] * 1.03, pos[-1] + 8, pos[-1] + 16]]):
            f = np.float32(v)
            vals.update([float(f), float(np.nextafter(f, np.float32(np.inf))),
                         float(np.nextafter(f, np.float32(0)))])
    g = np.random.default_rng(123)
    vals.update(np.float32(2.0 ** g.uniform(-14, 10, 3000)).astype(float).tolist())
    vals.update([0.0, 1e-45, 1e-30, 2.0 ** -10, 2.0 ** -11, 447.99, 448.0, 464.0, 500.0,
                 239.99, 240.0, 248.0, 1e30, math.inf])
    out = sorted(vals)
    out += [-v for v in out] + [math.nan]
    return out


@pytest.mark.parametrize("fmt", [e4m3.OCP, e4m3.FNUZ])
def test_encode_matches_brute_force(fmt):
    xs = probe_values()
    vec = e4m3.encode(np.array(xs, dtype=np.float32), fmt)
    for x, v in zip(xs, vec):
        bf = brute_force_encode(x, fmt)
        assert e4m3.encode_value(x, fmt) == bf, (x, fmt)
        assert int(v) == bf, (x, fmt)


@pytest.mark.parametrize("fmt", [e4m3.OCP, e4m3.FNUZ])
def test_encode_decode_roundtrip(fmt):
    for b in range(256):
        if e4m3.is_nan_code(b, fmt):
            continue
        v = e4m3.decode_byte(b, fmt)
        assert e4m3.encode_value(v, fmt) == b, hex(b)
    arr = np.array([b for b in range(256) if not e4m3.is_nan_code(b, fmt)], dtype=np.uint8)
    np.testing.assert_array_equal(e4m3.encode(e4m3.decode(arr, fmt).astype(np.float32), fmt), arr)


def test_midpoints_round_to_even_code():
    # 1.0625 lies between 1.0 (0x38, even) and 1.125 (0x39): goes to 0x38;
    # 1.1875 lies between 0x39 and 1.25 (0x3a): goes to 0x3a.
    assert e4m3.encode_value(1.0625, e4m3.OCP) == 0x38
    assert e4m3.encode_value(1.1875, e4m3.OCP) == 0x3A
    # OCP subnormal tie: 1.5 * 2^-9 -> 2 * 2^-9 (0x02); 0.5 * 2^-9 -> 0
    assert e4m3.encode_value(1.5 * 2 ** -9, e4m3.OCP) == 0x02
    assert e4m3.encode_value(0.5 * 2 ** -9, e4m3.OCP) == 0x00
    assert e4m3.encode_value(-0.5 * 2 ** -9, e4m3.OCP) == 0x80
    assert e4m3.encode_value(-0.5 * 2 ** -10, e4m3.FNUZ) == 0x00
    # the tie between the top two OCP codes 416 (0x7d) and 448 (0x7e) -> 448
    assert e4m3.encode_value(432.0, e4m3.OCP) == 0x7E
    assert e4m3.encode_value(-432.0, e4m3.OCP) == 0xFE
    # saturation, infinity and NaN
    assert e4m3.encode_value(1e9, e4m3.OCP) == 0x7E
    assert e4m3.encode_value(-math.inf, e4m3.FNUZ) == 0xFF
    assert e4m3.encode_value(math.nan, e4m3.OCP) == 0x7F
    assert e4m3.encode_value(math.nan, e4m3.FNUZ) == 0x80


@pytest.mark.parametrize("fmt,dt", [(e4m3.OCP, torch.float8_e4m3fn),
                                    (e4m3.FNUZ, torch.float8_e4m3fnuz)])
def test_encode_matches_torch_cast_in_range(fmt, dt):
    # library cross-check inside the finite range (PyTorch does not saturate)
    g = np.random.default_rng(7)
    mx = e4m3.params(fmt)["max"]
    x = np.float32(g.uniform(-mx, mx, 20000) * 2.0 ** g.integers(-16, 1, 20000))
    lib = torch.from_numpy(x).to(dt).view(torch.uint8).numpy()
    np.testing.assert_array_equal(e4m3.encode(x, fmt), lib)
