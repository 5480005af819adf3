"""Pins for the oracle's quantize and pack."""
import numpy as np
import pytest

from oracle import bf16, e4m3, pack, quantize


@pytest.mark.parametrize("fmt", [e4m3.OCP, e4m3.FNUZ])
def test_amax_element_maps_to_max_code(fmt):
    g = np.random.default_rng(0)
    x = np.float32(g.standard_normal((37, 53)))
    q, s = quantize.quantize_e4m3(x, quantize.PER_TENSOR, fmt)
    i = np.unravel_index(np.argmax(np.abs(x)), x.shape)
    mx = e4m3.params(fmt)["max_code"]
    assert q[i] & 0x7F == mx
    assert s == np.float32(np.abs(x).max() / e4m3.params(fmt)["max"])
    # per column: the largest |x| of every column reaches the maximum code
    q, s = quantize.quantize_e4m3(x, quantize.PER_COL, fmt)
    rows = np.argmax(np.abs(x), axis=0)
    assert ((q[rows, np.arange(x.shape[1])] & 0x7F) == mx).all()
    assert s.shape == (53,)


def test_quantize_hand_ties():
    # amax 448 -> s = 1 exactly, so x / s = x: ties decide by the even code
    x = np.float32([[448.0, 1.0625, 1.1875, -1.0625, 0.5 * 2 ** -9, 3.0]])
    q, s = quantize.quantize_e4m3(x, quantize.PER_TENSOR, e4m3.OCP)
    assert s == 1.0
    assert q.tolist() == [[0x7E, 0x38, 0x3A, 0xB8, 0x00, 0x44]]
    # amax 896 -> s = 2; 2.125 / 2 = 1.0625 ties to 1.0
    x = np.float32([[896.0, 2.125]])
    q, s = quantize.quantize_e4m3(x, quantize.PER_TENSOR, e4m3.OCP)
    assert s == 2.0 and q.tolist() == [[0x7E, 0x38]]


def test_quantize_monotone_and_accurate():
    g = np.random.default_rng(1)
    x = np.sort(np.float32(g.standard_t(3, 20000))).reshape(1, -1)
    for fmt in (e4m3.OCP, e4m3.FNUZ):
        q, s = quantize.quantize_e4m3(x, quantize.PER_TENSOR, fmt)
        deq = e4m3.decode(q, fmt) * float(s)
        assert (np.diff(deq[0]) >= 0).all()
        # relative error of a normal E4M3 value is at most 2^-4 (3 mantissa bits)
        norm = np.abs(x / s) >= 2.0 ** (1 - e4m3.params(fmt)["bias"])
        rel = np.abs(deq - x) / np.abs(x)
        assert (rel[norm] <= 2.0 ** -4).all()


def test_quantize_zero_nan_inf_static():
    z = np.zeros((3, 4), dtype=np.float32)
    q, s = quantize.quantize_e4m3(z, quantize.PER_TENSOR, e4m3.OCP)
    assert s == 1.0 and (q == 0).all()
    q, s = quantize.quantize_e4m3(z, quantize.PER_COL, e4m3.FNUZ)
    assert (s == 1.0).all() and (q == 0).all()
    x = np.float32([[1.0, np.nan, -2.0]])
    q, s = quantize.quantize_e4m3(x, quantize.PER_TENSOR, e4m3.OCP)
    assert s == np.float32(2.0 / 448.0)  # NaN ignored by amax
    assert q[0, 1] == 0x7F and q[0, 2] == 0xFE
    q, s = quantize.quantize_e4m3(np.float32([[1.0, 5.0]]), quantize.PER_TENSOR, e4m3.OCP,
                                  static_scale=np.float32(0.001))
    assert s == np.float32(0.001) and q.tolist() == [[0x7E, 0x7E]]  # 1000, 5000 saturate


def test_quantize_divides_not_reciprocal():
    # a case where x * (1/s) and x / s round differently in fp32
    g = np.random.default_rng(2)
    found = False
    for _ in range(2000):
        s = np.float32(g.uniform(0.001, 1.0))
        x = np.float32(g.uniform(-400, 400) * s)
        div = np.float32(np.float64(x) / np.float64(s))
        mul = np.float32(x * np.float32(np.float32(1.0) / s))
        if div != mul:
            found = True
            assert quantize.divide_f32(x, s) == div
    assert found


# ------------------------------------------------------------------ pack

def packed_offset(k, n, K, kind):
    """Byte offset of the first byte of W[k, n], from the layout's definition
    stated scalar-wise: tile (n // 128, kb) of 16 KiB, row n % 128 of 128
    bytes, 16-byte chunk (j // 16) XOR (row % 8), byte j % 16 in it."""
    es = pack.esize_of(kind)
    KB = -(-(K * es) // 128)
    kbyte = k * es
    nb, r = divmod(n, 128)
    kb, j = divmod(kbyte, 128)
    return ((nb * KB + kb) * 128 + r) * 128 + ((j // 16) ^ (r % 8)) * 16 + (j % 16)


@pytest.mark.parametrize("K,N", [(64, 128), (512, 256), (96, 200), (300, 130), (32, 16)])
def test_pack_e4m3_layout(K, N):
    g = np.random.default_rng(K * N)
    w = g.integers(0, 256, (K, N), dtype=np.uint8)
    p = pack.pack(w, "e4m3")
    assert p.size == pack.packed_bytes(K, N, "e4m3")
    assert p.size == -(-N // 128) * 128 * (-(-K // 128)) * 128
    for k, n in zip(g.integers(0, K, 500), g.integers(0, N, 500)):
        assert p[packed_offset(k, n, K, "e4m3")] == w[k, n]
    np.testing.assert_array_equal(pack.unpack(p, K, N, "e4m3"), w)
    # padding bytes are zero: the number of nonzero bytes equals that of w
    assert np.count_nonzero(p) == np.count_nonzero(w)


@pytest.mark.parametrize("K,N", [(64, 128), (512, 256), (80, 136)])
def test_pack_bf16_layout(K, N):
    g = np.random.default_rng(K + N)
    w = np.float32(g.standard_normal((K, N)))
    bits = bf16.f32_to_bf16_bits(w)
    p = pack.pack_fp32_as_bf16(w)
    assert p.size == pack.packed_bytes(K, N, "bf16")
    for k, n in zip(g.integers(0, K, 500), g.integers(0, N, 500)):
        o = packed_offset(k, n, K, "bf16")
        assert int(p[o]) | (int(p[o + 1]) << 8) == bits[k, n]  # little-endian bf16
    np.testing.assert_array_equal(pack.unpack(p, K, N, "bf16"), bits)
