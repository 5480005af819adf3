"""Pins of the NVFP4 oracle (oracle/nvfp4.py) against what the format
definitions and the mathematics fix: the hand-typed E2M1 code table, a
brute-force nearest-code search with ties to the even code, round trips,
hand-computed block scales and codes, the block-maximum invariant, exact
scaling by powers of two, and integer-exact GEMMs against Python loops."""
import math
import os

import numpy as np
import pytest

from oracle import e4m3, nvfp4

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "e2m1_values.txt")


def _golden():
    out = {}
    with open(GOLDEN) as f:
        for line in f:
            line = line.split("#", 1)[0].split()
            if not line:
                continue
            code, val = int(line[0], 16), line[1]
            out[code] = -0.0 if val == "-0" else float(val)
    return out


def test_decode_matches_hand_table():
    g = _golden()
    assert sorted(g) == list(range(16))
    t = nvfp4.decode_table()
    for c, v in g.items():
        assert t[c] == v and math.copysign(1.0, t[c]) == math.copysign(1.0, v), c


def _nearest_even(x):
    """Brute force: the code whose value is nearest to x; on a tie the one
    with mantissa bit 0 (the even code); |x| >= 6 -> +-6; sign kept."""
    if math.isnan(x):
        return 0
    t = nvfp4.decode_table()
    sign = 8 if math.copysign(1.0, x) < 0 else 0
    a = min(abs(x), 6.0)
    best = None
    for c in range(8):
        d = abs(t[c] - a)
        if best is None or d < best[0] or (d == best[0] and (c & 1) == 0):
            best = (d, c)
    return sign | best[1]


def _probes():
    t = nvfp4.decode_table()[:8]
    mids = (t[1:] + t[:-1]) / 2
    vals = np.concatenate([t, mids, [6.5, 7.0, 100.0, 1e-30, 0.1, 0.2, 0.3]])
    f = vals.astype(np.float32)
    up = np.nextafter(f, np.float32(np.inf))
    dn = np.nextafter(f, np.float32(-np.inf))
    rnd = np.random.default_rng(5).uniform(-8, 8, 4000).astype(np.float32)
    allv = np.concatenate([f, up, dn, -f, -up, -dn, rnd]).astype(np.float64)
    return np.concatenate([allv, [np.inf, -np.inf, np.nan, -0.0]])


def test_encode_is_nearest_with_ties_to_even():
    p = _probes()
    got = nvfp4.encode(p)
    for x, c in zip(p, got):
        assert c == _nearest_even(x), (x, c)
        assert c == nvfp4.encode_value(x), x


def test_encode_decode_round_trip():
    t = nvfp4.decode_table()
    np.testing.assert_array_equal(nvfp4.encode(t), np.arange(16))


def test_hand_block():
    # one block holding every magnitude of the format, positive and negative:
    # amax 6 -> g = 6 / 2688, d = 6 g, the block scale E4M3(6 / d) = 448
    # (0x7e), e = 448 g ~ 1, so every value encodes to its own code
    x = np.array([[6, 4, 3, 2, 1.5, 1, 0.5, 0, -6, -4, -3, -2, -1.5, -1, -0.5, -0.0]],
                 dtype=np.float32)
    q, sb, g = nvfp4.quantize(x)
    assert g == np.float32(6.0 / 2688.0)
    assert sb.tolist() == [[0x7E]]
    assert q.tolist() == [[7, 6, 5, 4, 3, 2, 1, 0, 15, 14, 13, 12, 11, 10, 9, 8]]


def test_hand_two_blocks_and_zero_block():
    # block 0 max 6 (scale 448), block 1 max 0.375 = 6 / 16 (scale 28 =
    # 1.75 * 2^4 -> E4M3 byte 0.1011.110 = 0x5e), block 2 all zero (scale 0)
    x = np.zeros((1, 48), dtype=np.float32)
    x[0, 3] = 6.0
    x[0, 20] = -0.375
    x[0, 21] = 0.09375  # 0.375 / 4: value 1.5 after the block's e = 0.0625
    q, sb, g = nvfp4.quantize(x)
    assert sb.tolist() == [[0x7E, 0x5E, 0x00]]
    assert e4m3.decode_byte(0x5E, e4m3.OCP) == 28.0
    assert q[0, 3] == 7 and q[0, 20] == 15 and q[0, 21] == 3
    assert (q[0, 32:] == 0).all()
    # an all-zero tensor: g = 1, scales and codes 0
    q, sb, g = nvfp4.quantize(np.zeros((2, 32), dtype=np.float32))
    assert g == 1.0 and not sb.any() and not q.any()


def test_block_maximum_encodes_to_six():
    # the block's largest magnitude lands within the E4M3 scale rounding of
    # 6, whose nearest E2M1 value is 6
    rng = np.random.default_rng(3)
    x = (rng.standard_normal((32, 256)) * rng.uniform(0.01, 100, (32, 1))).astype(np.float32)
    q, sb, g = nvfp4.quantize(x)
    blocks = np.abs(x).reshape(32, 16, 16)
    arg = blocks.argmax(axis=2)
    qb = q.reshape(32, 16, 16)
    for i in range(32):
        for j in range(16):
            if sb[i, j] >= 0x08:  # a normal block scale
                assert qb[i, j, arg[i, j]] & 7 == 7


def test_power_of_two_scaling_moves_only_the_tensor_scale():
    rng = np.random.default_rng(4)
    x = (rng.standard_normal((8, 64)) * rng.uniform(0.1, 10, (8, 1))).astype(np.float32)
    q0, s0, g0 = nvfp4.quantize(x)
    for k in (-8, -1, 3, 9):
        q, s, g = nvfp4.quantize((x * np.float32(2.0 ** k)).astype(np.float32))
        np.testing.assert_array_equal(q, q0)
        np.testing.assert_array_equal(s, s0)
        assert g == np.float32(g0 * 2.0 ** k)


def test_nibble_packing():
    q = np.arange(32, dtype=np.uint8).reshape(1, 32) & 0xF
    p = nvfp4.pack_nibbles(q)
    assert p[0, 0] == 0x10 and p[0, 1] == 0x32  # element 0 low, element 1 high
    np.testing.assert_array_equal(nvfp4.unpack_nibbles(p), q)


def test_gemm_integer_exact():
    # unit block scales (E4M3 0x38 = 1) and unit tensor scales: values are
    # multiples of 0.5 up to 6, so 4 * acc is an exact integer sum
    rng = np.random.default_rng(7)
    M, N, K = 5, 7, 64
    qa = rng.integers(0, 16, (M, K)).astype(np.uint8)
    qw = rng.integers(0, 16, (N, K)).astype(np.uint8)
    sa = np.full((M, K // 16), 0x38, dtype=np.uint8)
    sw = np.full((N, K // 16), 0x38, dtype=np.uint8)
    bias = np.arange(N, dtype=np.float32)
    v, _ = nvfp4.gemm(qa, sa, 1.0, qw, sw, 1.0, bias)
    twice = {c: int(round(2 * nvfp4.decode_nibble(c))) for c in range(16)}
    for m in range(M):
        for n in range(N):
            s4 = sum(twice[int(qa[m, k])] * twice[int(qw[n, k])] for k in range(K))
            assert v[m, n] == s4 / 4 + n


def test_gemm_block_scales_and_tensor_scales_apply_per_block():
    # power-of-two block scales differ per block and per row/column: the
    # result equals a triple loop over k with each element's own scale
    rng = np.random.default_rng(8)
    M, N, K = 3, 4, 48
    qa = rng.integers(0, 16, (M, K)).astype(np.uint8)
    qw = rng.integers(0, 16, (N, K)).astype(np.uint8)
    sa = rng.choice([0x30, 0x38, 0x40, 0x48], (M, K // 16)).astype(np.uint8)  # 0.5, 1, 2, 4
    sw = rng.choice([0x28, 0x38, 0x50], (N, K // 16)).astype(np.uint8)        # 0.25, 1, 8
    v, _ = nvfp4.gemm(qa, sa, 0.5, qw, sw, 4.0)
    dec = nvfp4.decode_nibble
    sc = lambda b: e4m3.decode_byte(b, e4m3.OCP)  # noqa: E731
    for m in range(M):
        for n in range(N):
            acc = sum(dec(qa[m, k]) * sc(sa[m, k // 16]) * dec(qw[n, k]) * sc(sw[n, k // 16])
                      for k in range(K))
            assert v[m, n] == acc * 2.0
