"""The bounded-wait give-up path, made to run out from the host with no GPU
fault.

The one-grid per-tensor quantize meets at a grid barrier in its workspace
header: each CTA arrives on a count and waits until the count is complete
(or the last CTA to arrive has published the scale).  Here the header's
arrival word is pre-set far from zero, so the count never completes and no
CTA sees itself as the last arrival: every CTA waits until its one-second
limit, gives up and returns.  The call must then be visibly invalid (NaN
scale, NaN codes, the give-up record 0x201 in header word 1), the device must
stay usable, and after the header is zero-filled again the next call must be
bit-exact with the oracle.
"""
import math

import numpy as np
import pytest
import torch

import synth
from bf16_gemm_vla_gb300 import frt
from helpers import bf16_dev
from oracle import e4m3, quantize

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("rows,cols", [(768, 2048), (768, 16384)])
def test_quantize_barrier_gives_up_then_recovers(rows, cols):
    # 768 x 2048 bf16 sits in registers, 768 x 16384 in shared memory: both
    # one-grid kernels
    bits = synth.activations(np.random.default_rng(31), rows, cols, outlier_frac=0.01)
    xd = bf16_dev(bits)
    nb = frt.frt_quantize_workspace_bytes(rows, cols, frt.PER_TENSOR)
    ws = torch.zeros((nb // 4,), dtype=torch.int32, device="cuda")
    ws[0] = -(1 << 16)  # arrivals = 0xffff0000: the count never reaches the grid size
    q, s = frt.frt_quantize_e4m3(xd, frt.PER_TENSOR, frt.OCP, workspace=ws)
    torch.cuda.synchronize()
    assert math.isnan(float(s.cpu()[0]))
    assert int(ws[1].cpu()) == 0x201
    assert bool((q == 0x7F).all())  # every element encoded with a NaN scale
    # the device is still usable; a zero-filled header makes the next call valid
    ws[:64].zero_()
    q, s = frt.frt_quantize_e4m3(xd, frt.PER_TENSOR, frt.OCP, workspace=ws)
    qo, so = quantize.quantize_e4m3(synth.bf16_bits_as_f32(bits), quantize.PER_TENSOR, e4m3.OCP)
    assert s.cpu().numpy()[0] == so
    np.testing.assert_array_equal(q.cpu().numpy(), qo)
    hdr = ws[:8].cpu().numpy()
    # arrivals and status back at zero, and the next call's running maximum
    # (word 4 or 5 by the generation's parity) cleared
    assert hdr[0] == 0 and hdr[1] == 0 and hdr[4 + (hdr[2] & 1)] == 0
