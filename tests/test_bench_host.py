"""Host-side logic of bench.py, on the CPU: the whole-job aggregation over
ranks (world_size 2, gloo) and the argument defaults.  The path has no
exchange step, so N GPUs run N replicas; the job's value is the units of
all ranks over the slowest rank's time."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        units = [100.0, 300.0][rank]
        secs = [2.0, 5.0][rank]
        value, slowest = bench.aggregate(units, secs, world)
        assert bench.dist_env() == (rank, rank, world)
        bench.barrier(world)
        out[rank] = (value, slowest)
    finally:
        dist.destroy_process_group()


def test_aggregate_over_two_gloo_ranks():
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(2, port, out), nprocs=2, join=True)
        res = dict(out)
    # (100 + 300) units over the slowest rank's 5 s, the same on both ranks
    assert res[0] == pytest.approx((80.0, 5.0))
    assert res[1] == pytest.approx((80.0, 5.0))


def test_single_rank_aggregate_and_defaults(monkeypatch):
    assert bench.aggregate(10.0, 4.0, 1) == (2.5, 4.0)
    a = bench.parse_args([])
    assert (a.gpus, a.impl, a.warmup >= 3, a.steps > 0) == (1, "ours", True, True)
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    # the reference arm runs on rank 0 only; other ranks exit 0 without work
    assert bench.run_reference(bench.parse_args(["--impl", "reference"])) == 0


def test_peaks_fall_back_without_measurements(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    peaks, kind = bench.load_peaks()
    assert kind == "fallback" and peaks["hbm_gbs"] == 6800.0


def test_profiled_traffic_keyed_to_gemm_code_not_comments(tmp_path, monkeypatch):
    # the recorded ncu DRAM figures apply while the GEMM sources' code is the
    # captured one: a comment edit keeps them, a code edit drops them (null)
    csrc = tmp_path / "bf16_gemm_vla_gb300" / "csrc"
    csrc.mkdir(parents=True)
    prof = tmp_path / "profiles"
    prof.mkdir()
    for f in ("frt_gemm.cu", "frt_device.cuh"):
        (csrc / f).write_text("int x = 1;  // a comment\n\n// another\nint y = 2;\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h = bench.gemm_source_hash()
    (prof / "gemm_fp8_dram_traffic.txt").write_text(
        "# header\nsource %s\n768 2048 16384 100\n768 16384 2048 300\n" % h)
    shapes = [(768, 2048, 16384), (768, 16384, 2048)]
    assert bench.profiled_traffic(shapes) == 200.0
    (csrc / "frt_gemm.cu").write_text("int x = 1;  // the comment, reworded\nint y = 2;\n")
    assert bench.gemm_source_hash() == h and bench.profiled_traffic(shapes) == 200.0
    (csrc / "frt_gemm.cu").write_text("int x = 3;\nint y = 2;\n")
    assert bench.gemm_source_hash() != h and bench.profiled_traffic(shapes) is None
    assert bench.profiled_traffic([(1, 2, 3)]) is None  # a shape without a figure
