"""Shared pytest configuration.

Marker ``gpu``: the test launches CUDA kernels through the C-ABI library and
needs a GB300 (sm_103a).  Everything else runs on the CPU.
"""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 GPU and the built CUDA library")


def within_gemm_tolerance(gpu, ref, sumabs):
    """The GEMM acceptance bar, per element:
    |gpu - ref| <= 2^-7 * |ref| + 1e-5 * sum_k |a*w| (scaled)."""
    import numpy as np

    gpu = np.asarray(gpu, dtype=np.float64)
    err = np.abs(gpu - ref)
    bound = 2.0 ** -7 * np.abs(ref) + 1e-5 * sumabs
    return err <= bound, err, bound
