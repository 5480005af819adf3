"""GPU parity of the cast kernels (FNUZ -> OCP and E4M3 quantize) against
the oracle: bit-exact on every byte and every scale."""
import math

import numpy as np
import pytest
import torch

import synth
from bf16_gemm_vla_gb300 import frt
from helpers import bf16_dev
from oracle import convert, e4m3, quantize

pytestmark = pytest.mark.gpu


# ---------------------------------------------------------------- FNUZ -> OCP

@pytest.mark.parametrize("offset,length", [(0, 4096), (0, 4099), (1, 4096), (3, 17), (16, 1),
                                           (5, 100003)])
def test_fnuz_to_ocp_all_bytes(offset, length):
    g = np.random.default_rng(length)
    host = np.concatenate([np.tile(np.arange(256, dtype=np.uint8), 8),
                           g.integers(0, 256, length + 64, dtype=np.uint8)])
    dev = torch.from_numpy(host).cuda()
    x = dev[offset:offset + length]
    out = frt.frt_fnuz_to_ocp(x)
    np.testing.assert_array_equal(out.cpu().numpy(),
                                  convert.fnuz_to_ocp(host[offset:offset + length]))


def test_fnuz_to_ocp_in_place():
    host = np.tile(np.arange(256, dtype=np.uint8), 33)
    dev = torch.from_numpy(host).cuda()
    frt.frt_fnuz_to_ocp(dev, out=dev)
    np.testing.assert_array_equal(dev.cpu().numpy(), convert.fnuz_to_ocp(host))


def test_fnuz_to_ocp_1gib_stream():
    # sweep (ii): 1 GiB of uniform random bytes (every value, 0x80 and the
    # subnormal codes included), seed 2; compared in full
    n = 1 << 30
    host = synth.uniform_bytes(n, seed=2)
    dev = torch.from_numpy(host).cuda()
    out = frt.frt_fnuz_to_ocp(dev)
    ref = convert.fnuz_to_ocp(host)
    assert np.array_equal(out.cpu().numpy(), ref)


# ---------------------------------------------------------------- quantize

def _dev_input(x_f32, dtype):
    if dtype == torch.bfloat16:
        bits = synth.to_bf16_bits(x_f32)
        return bf16_dev(bits), synth.bf16_bits_as_f32(bits)
    return torch.from_numpy(np.ascontiguousarray(x_f32, dtype=np.float32)).cuda(), \
        np.asarray(x_f32, dtype=np.float32)


FMTS = [(frt.OCP, e4m3.OCP), (frt.FNUZ, e4m3.FNUZ)]


@pytest.mark.parametrize("fmt,ofmt", FMTS)
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("rows,cols", [(16, 512), (50, 1024), (7, 40), (3, 13), (768, 2048),
                                       (1, 1)])
def test_quantize_per_tensor(fmt, ofmt, dtype, rows, cols):
    g = np.random.default_rng(rows * 1000 + cols)
    x = g.standard_normal((rows, cols))
    if rows * cols > 100:
        x[g.random((rows, cols)) < 0.01] *= 50.0
    xd, xh = _dev_input(x, dtype)
    q, s = frt.frt_quantize_e4m3(xd, frt.PER_TENSOR, fmt)
    qo, so = quantize.quantize_e4m3(xh, quantize.PER_TENSOR, ofmt)
    assert s.cpu().numpy()[0] == so
    np.testing.assert_array_equal(q.cpu().numpy(), qo)


@pytest.mark.parametrize("fmt,ofmt", FMTS)
def test_quantize_strided_rows(fmt, ofmt):
    g = np.random.default_rng(11)
    big = g.standard_normal((50, 2560))
    xd, xh = _dev_input(big, torch.bfloat16)
    for cols in (2048, 1000, 13):
        q, s = frt.frt_quantize_e4m3(xd[:, :cols], frt.PER_TENSOR, fmt)
        qo, so = quantize.quantize_e4m3(xh[:, :cols], quantize.PER_TENSOR, ofmt)
        assert s.cpu().numpy()[0] == so
        np.testing.assert_array_equal(q.cpu().numpy(), qo)


@pytest.mark.parametrize("fmt,ofmt", FMTS)
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("K,N", [(512, 256), (1024, 4096), (300, 130), (65, 7), (4096, 1024)])
def test_quantize_per_col(fmt, ofmt, dtype, K, N):
    g = np.random.default_rng(K + N)
    w = g.standard_normal((K, N)) * 0.02
    wd, wh = _dev_input(w, dtype)
    q, s = frt.frt_quantize_e4m3(wd, frt.PER_COL, fmt)
    qo, so = quantize.quantize_e4m3(wh, quantize.PER_COL, ofmt)
    np.testing.assert_array_equal(s.cpu().numpy(), so)
    np.testing.assert_array_equal(q.cpu().numpy(), qo)


@pytest.mark.parametrize("fmt,ofmt", FMTS)
def test_encode_every_bf16_pattern(fmt, ofmt):
    # static scale 1: q = E4M3(x) for all 65536 bf16 bit patterns (NaN, inf,
    # subnormals, both zeros included)
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16).reshape(256, 256)
    one = torch.ones(1, dtype=torch.float32, device="cuda")
    q, _ = frt.frt_quantize_e4m3(bf16_dev(bits), frt.PER_TENSOR, fmt, static_scale=one)
    ref = e4m3.encode(synth.bf16_bits_as_f32(bits), ofmt)
    np.testing.assert_array_equal(q.cpu().numpy(), ref)


def _fp32_probes():
    vals = []
    for fmt in (e4m3.OCP, e4m3.FNUZ):
        t = e4m3.decode_table(fmt)
        pos = np.unique(t[(t >= 0) & ~np.isnan(t)])
        mids = (pos[1:] + pos[:-1]) / 2
        for v in np.concatenate([pos, mids]):
            f = np.float32(v)
            vals += [f, np.nextafter(f, np.float32(np.inf)), np.nextafter(f, np.float32(0))]
    g = np.random.default_rng(99)
    vals += list(np.float32(2.0 ** g.uniform(-30, 12, 60000)))
    vals += [np.float32(v) for v in (0.0, 1e-45, 1e-39, 240.0, 448.0, 1e38, math.inf, math.nan)]
    v = np.array(vals, dtype=np.float32)
    v = np.concatenate([v, -v])
    pad = (-len(v)) % 8
    return np.concatenate([v, np.zeros(pad, dtype=np.float32)]).reshape(-1, 8)


@pytest.mark.parametrize("fmt,ofmt", FMTS)
def test_encode_fp32_probes_and_division(fmt, ofmt):
    x = _fp32_probes()
    xd = torch.from_numpy(x).cuda()
    one = torch.ones(1, dtype=torch.float32, device="cuda")
    q, _ = frt.frt_quantize_e4m3(xd, frt.PER_TENSOR, fmt, static_scale=one)
    np.testing.assert_array_equal(q.cpu().numpy(), e4m3.encode(x, ofmt))
    # arbitrary static scales: the quotient is an IEEE fp32 division
    g = np.random.default_rng(5)
    for s in np.float32(g.uniform(1e-3, 3.0, 4)):
        sd = torch.tensor([s], dtype=torch.float32, device="cuda")
        xs = np.float32(x[:, :] * np.float32(g.uniform(0.5, 2.0)))
        q, so = frt.frt_quantize_e4m3(torch.from_numpy(xs).cuda(), frt.PER_TENSOR, fmt,
                                      static_scale=sd)
        qo, _ = quantize.quantize_e4m3(xs, quantize.PER_TENSOR, ofmt, static_scale=s)
        np.testing.assert_array_equal(q.cpu().numpy(), qo)
        assert so.cpu().numpy()[0] == s


def test_quantize_edge_cases():
    z = torch.zeros((5, 24), dtype=torch.bfloat16, device="cuda")
    q, s = frt.frt_quantize_e4m3(z, frt.PER_TENSOR, frt.OCP)
    assert s.item() == 1.0 and int(q.sum()) == 0
    q, s = frt.frt_quantize_e4m3(z.float(), frt.PER_COL, frt.FNUZ)
    assert bool((s == 1.0).all()) and int(q.sum()) == 0
    x = np.float32([[1.0, np.nan, -2.0, np.inf, -np.inf, -0.0, 0.0, 3.0]])
    for fmt, ofmt in FMTS:
        q, s = frt.frt_quantize_e4m3(torch.from_numpy(x).cuda(), frt.PER_TENSOR, fmt)
        qo, so = quantize.quantize_e4m3(x, quantize.PER_TENSOR, ofmt)
        assert s.cpu().numpy()[0] == so
        np.testing.assert_array_equal(q.cpu().numpy(), qo)
    empty = torch.zeros((0, 16), dtype=torch.bfloat16, device="cuda")
    q, s = frt.frt_quantize_e4m3(empty, frt.PER_TENSOR, frt.OCP)
    assert q.shape == (0, 16)


def test_quantize_student_t_full_size():
    # sweep (iii): 256 Mi bf16 from Student-t (nu = 3), per-tensor OCP.  The
    # scale is checked exactly, and every one of the 256 Mi bytes: the
    # oracle's quantize with that scale is an elementwise function of the
    # bf16 input, so it is evaluated once on each of the 65536 bf16 bit
    # patterns and looked up by each element's bits.
    n = 256 << 20
    bits = synth.student_t_bf16(n, seed=3)
    xd = bf16_dev(bits.reshape(-1, 4096))
    q, s = frt.frt_quantize_e4m3(xd, frt.PER_TENSOR, frt.OCP)
    xh = synth.bf16_bits_as_f32(bits)
    so = quantize.scale_from_amax(quantize.amax(xh, quantize.PER_TENSOR), e4m3.OCP)
    del xh
    assert s.cpu().numpy()[0] == so
    patterns = synth.bf16_bits_as_f32(np.arange(1 << 16, dtype=np.uint16)).reshape(1, -1)
    table, _ = quantize.quantize_e4m3(patterns, quantize.PER_TENSOR, e4m3.OCP, static_scale=so)
    np.testing.assert_array_equal(q.view(-1).cpu().numpy(), table.reshape(-1)[bits])


@pytest.mark.parametrize("fmt,ofmt", FMTS)
def test_quotients_near_rounding_midpoints(fmt, ofmt):
    # x is built so that x / s lands within +-12 fp32 steps of every midpoint
    # between adjacent E4M3 codes, for many scales: the region where a
    # quotient computed by a reciprocal could round differently from the
    # IEEE quotient.  Bytes must equal the oracle's (IEEE fp32 division).
    t = e4m3.decode_table(ofmt)
    pos = np.unique(t[(t > 0) & ~np.isnan(t)])
    mids = np.float32((pos[1:] + pos[:-1]) / 2)
    steps = np.arange(-12, 13, dtype=np.int64)
    g = np.random.default_rng(17)
    for s in np.float32(np.concatenate([g.uniform(1e-3, 4.0, 6), [1.0, 0.5, 3.0 / 448]])):
        target = (mids.view(np.int32)[:, None] + steps[None, :]).astype(np.int32).view(np.float32)
        x = np.float32(target.astype(np.float64) * np.float64(s)).reshape(-1)
        x = np.concatenate([x, -x])
        x = np.concatenate([x, np.zeros((-len(x)) % 8, dtype=np.float32)]).reshape(-1, 8)
        sd = torch.tensor([s], dtype=torch.float32, device="cuda")
        for dt in (torch.float32,):
            q, _ = frt.frt_quantize_e4m3(torch.from_numpy(x).cuda().to(dt), frt.PER_TENSOR, fmt,
                                         static_scale=sd)
            qo, _ = quantize.quantize_e4m3(x, quantize.PER_TENSOR, ofmt, static_scale=s)
            np.testing.assert_array_equal(q.cpu().numpy(), qo)
        # the same values as one column of a per-column quantize
        xc = np.ascontiguousarray(x.reshape(-1, 1))
        q, _ = frt.frt_quantize_e4m3(torch.from_numpy(xc).cuda(), frt.PER_COL, fmt,
                                     static_scale=torch.tensor([s], device="cuda"))
        qo, _ = quantize.quantize_e4m3(xc, quantize.PER_COL, ofmt, static_scale=np.float32([s]))
        np.testing.assert_array_equal(q.cpu().numpy(), qo)


def test_quantize_workspace_reused_across_shapes():
    # one zero-filled workspace through a sequence of per-tensor shapes whose
    # one-grid launches have different CTA counts (and a strided view, which
    # takes the two-kernel path): every result is the oracle's and the
    # header is ready for the next call (arrivals and status at zero, the
    # next call's running maximum cleared); the inputs' maxima go down as
    # well as up, so a maximum left over from a call would show in a later
    # scale
    nb = frt.frt_quantize_workspace_bytes(768, 16384, frt.PER_TENSOR)
    ws = torch.zeros((nb // 4,), dtype=torch.float32, device="cuda")
    g = np.random.default_rng(21)
    big = g.standard_normal((64, 1032))
    for rows, cols in [(768, 16384), (3, 16), (50, 1024), (768, 2048), (1, 8), (768, 16384),
                       ("strided", 0), (200, 4096)]:
        if rows == "strided":
            xd, xh = _dev_input(big, torch.bfloat16)
            xd, xh = xd[:, :1024], xh[:, :1024]
        else:
            x = g.standard_normal((rows, cols))
            x[g.random((rows, cols)) < 0.01] *= 50.0
            xd, xh = _dev_input(x, torch.bfloat16)
        q, s = frt.frt_quantize_e4m3(xd, frt.PER_TENSOR, frt.OCP, workspace=ws)
        qo, so = quantize.quantize_e4m3(xh, quantize.PER_TENSOR, e4m3.OCP)
        assert s.cpu().numpy()[0] == so
        np.testing.assert_array_equal(q.cpu().numpy(), qo)
        hdr = ws[:8].view(torch.int32).cpu().numpy()
        assert hdr[0] == 0 and hdr[1] == 0 and hdr[4 + (hdr[2] & 1)] == 0


@pytest.mark.parametrize("extra_row", [0, 1])
def test_quantize_one_grid_capacity_boundary(extra_row):
    # the largest dense bf16 tensor held in the SMs' shared memory (208 KiB
    # per SM) and one row more (two-kernel path): both bit-exact
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    cols = 8192
    rows = sms * 212992 // (2 * cols) + extra_row
    bits = synth.student_t_bf16(rows * cols, seed=4).reshape(rows, cols)
    q, s = frt.frt_quantize_e4m3(bf16_dev(bits), frt.PER_TENSOR, frt.OCP)
    xh = synth.bf16_bits_as_f32(bits)
    qo, so = quantize.quantize_e4m3(xh, quantize.PER_TENSOR, e4m3.OCP)
    assert s.cpu().numpy()[0] == so
    np.testing.assert_array_equal(q.cpu().numpy(), qo)


@pytest.mark.parametrize("rows,cols", [(16, 256), (768, 16384)])
@pytest.mark.parametrize("case", ["nan", "inf", "subnormal_max"])
def test_quantize_bf16_amax_specials(rows, cols, case):
    # per-tensor amax over bf16 input (the one-grid paths, registers and
    # shared memory): NaNs are ignored, an infinite |x| is the maximum, and
    # a maximum among bf16 subnormals is exact; bytes and scale match the
    # oracle bit for bit
    g = np.random.default_rng(rows + len(case))
    x = g.standard_normal((rows, cols)) * (1e-39 if case == "subnormal_max" else 1.0)
    idx = g.integers(0, rows * cols, 64)
    if case == "nan":
        x.reshape(-1)[idx] = np.nan
        x.reshape(-1)[idx[:8]] = -np.nan
        x.reshape(-1)[idx[8:16]] = -0.0
    elif case == "inf":
        x.reshape(-1)[idx[:4]] = -np.inf
    else:
        x.reshape(-1)[idx[:4]] = np.nan
    xd, xh = _dev_input(x, torch.bfloat16)
    q, s = frt.frt_quantize_e4m3(xd, frt.PER_TENSOR, frt.OCP)
    qo, so = quantize.quantize_e4m3(xh, quantize.PER_TENSOR, e4m3.OCP)
    np.testing.assert_array_equal(s.cpu().numpy(), np.float32([so]))
    np.testing.assert_array_equal(q.cpu().numpy(), qo)
