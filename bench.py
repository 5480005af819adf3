#!/usr/bin/env python
"""Benchmark of the quantized linear-layer path on GB300; prints one JSON line.

Headline step (value, unit TFLOP/s): the encoder-shaped FP8 layer set at
M = 768 -- (K, N) = (2048, 2560), (2048, 16384), (16384, 2048) -- each layer
a per-tensor dynamic E4M3 quantize of its bf16 activations (amax + encode)
followed by the FP8 tcgen05 GEMM with per-channel weight scales and bias,
all three replayed as one CUDA graph.  value = FP8 GEMM FLOPs of the step x
steps / device time of the timed region.  R rotating sets of weights,
activations and outputs (together larger than 4x L2) are cycled so no step
finds its operands in L2.

Also measured in the same run (``components``): the decoder-shaped GEMMs at
M = 50, FP8 and BF16, as weight-stream GB/s per layer (weight bytes / kernel
time, rotating weight copies > 4x L2); the encoder BF16 GEMMs; quantize GB/s
on 256 Mi Student-t bf16 values; FNUZ -> OCP GB/s on a 1 GiB byte stream;
and the 18+18-layer synthetic stack's replay latency.

--impl reference times the CPU oracle on the host cores instead (the
reference arm of the comparison), on bounded samples of the same workload.

Multi-GPU: replicas only (the path has no exchange step); under torchrun
every rank runs the same step on its own GPU, and value = work of all ranks /
the slowest rank's time.
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import synth  # noqa: E402

METRIC = "FP8 GEMM TFLOP/s (M=768) & weight-stream GB/s (M=50) vs roofline; quantize GB/s"
M_ENC = 768
M_DEC = 50
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
FP8_OVER_BF16 = 2.0  # nominal dense ratio, 4.5 / 2.25 PFLOP/s
ENC_WORKLOAD = ("encoder-shaped FP8 layers, M=768, (K,N)=(2048,2560),(2048,16384),(16384,2048): "
                "per-tensor dynamic OCP E4M3 activation quantize + FP8 GEMM with per-channel "
                "weight scales and bias, one CUDA graph per step")


def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=2000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=("ours", "reference"), default="ours")
    p.add_argument("--no-components", action="store_true",
                   help="time the headline step only")
    p.add_argument("--no-sweep", action="store_true",
                   help="skip the M sweep at K=N=4096 (run by default with the components)")
    p.add_argument("--rotate", type=int, default=0,
                   help="rotating buffer sets for the headline step (0: enough for 4x L2)")
    return p.parse_args(argv)


# ---------------------------------------------------------------- multi-rank plumbing

def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0")),
            int(os.environ.get("WORLD_SIZE", "1")))


def init_dist(world):
    if world > 1 and not torch.distributed.is_initialized():
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        torch.distributed.init_process_group(backend)


def barrier(world):
    if world > 1:
        torch.distributed.barrier()


def reduce_max(x, world, device=None):
    """Max of a float over ranks (the slowest rank's time)."""
    if world == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def reduce_sum(x, world, device=None):
    if world == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.SUM)
    return float(t.item())


def aggregate(units_per_rank, seconds_per_rank, world, device=None):
    """Whole-job throughput: units of all ranks / the slowest rank's time."""
    units = reduce_sum(units_per_rank, world, device)
    secs = reduce_max(seconds_per_rank, world, device)
    return units / secs, secs


# ---------------------------------------------------------------- peaks and clocks

def gemm_source_hash():
    """Hash of the GEMM sources' code: line comments and blank lines are left
    out, so that editing a comment does not invalidate the recorded ncu
    figures (the sources hold no '//' inside string literals)."""
    import hashlib

    h = hashlib.sha256()
    for f in ("bf16_gemm_vla_gb300/csrc/frt_gemm.cu", "bf16_gemm_vla_gb300/csrc/frt_device.cuh"):
        with open(os.path.join(ROOT, f), encoding="utf-8") as fh:
            for line in fh:
                code = line.split("//", 1)[0].rstrip()
                if code:
                    h.update(code.encode() + b"\n")
    return h.hexdigest()[:16]


def profiled_traffic(shapes):
    """Mean DRAM bytes per launch over `shapes` [(M, K, N)] from the committed ncu
    figures, or None when the GEMM sources changed since they were taken."""
    path = os.path.join(ROOT, "profiles", "gemm_fp8_dram_traffic.txt")
    if not os.path.exists(path):
        return None
    src, table = None, {}
    with open(path) as f:
        for line in f:
            parts = line.split()
            if not parts or parts[0].startswith("#"):
                continue
            if parts[0] == "source":
                src = parts[1]
            elif len(parts) == 4:
                table[tuple(int(x) for x in parts[:3])] = float(parts[3])
    if src != gemm_source_hash() or not all(tuple(s) in table for s in shapes):
        return None
    return sum(table[tuple(s)] for s in shapes) / len(shapes)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def fp8_peak_burst(peaks):
    """Dense FP8 peak for kernels timed in sub-second bursts: the BF16 burst
    figure x the nominal FP8/BF16 dense ratio."""
    return peaks["bf16_tflops"] * FP8_OVER_BF16


def measure_fp8_peak(device, n=8192, reps=10):
    """cuBLAS FP8 (E4M3 x E4M3 -> bf16) throughput on this GPU in this run,
    torch._scaled_mm on n x n x n, best of `reps` (the same protocol as the
    BF16 burst figure).  A denominator only: no step of the path uses it.
    Returns TFLOP/s, or None where torch offers no FP8 matmul."""
    try:
        a = torch.randn((n, n), device=device).to(torch.float8_e4m3fn)
        b = torch.randn((n, n), device=device).to(torch.float8_e4m3fn).t()  # column-major
        one = torch.ones((), dtype=torch.float32, device=device)
        mm = lambda: torch._scaled_mm(a, b, scale_a=one, scale_b=one,  # noqa: E731
                                      out_dtype=torch.bfloat16)
        for _ in range(3):
            mm()
        best = None
        for _ in range(reps):
            secs = device_time(lambda i: mm(), 1)
            best = secs if best is None or secs < best else best
        del a, b
        torch.cuda.empty_cache()
        return 2.0 * n ** 3 / best / 1e12
    except (RuntimeError, AttributeError, TypeError):
        return None


class ClockSampler:
    """nvidia-smi samples (every 100 ms) while the benchmark runs; the
    summary keeps the samples taken inside timed regions."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.windows = []
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def window(self, t0, t1):
        self.windows.append((t0, t1))

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                    ts += float("0." + parts[0].split(".")[1]) if "." in parts[0] else 0.0
                    rows.append((ts, float(parts[1]), float(parts[2]), parts[5:9]))
                except (ValueError, IndexError):
                    continue
        os.unlink(self.path)
        inside = [r for r in rows if any(a - 0.15 <= r[0] <= b + 0.15 for a, b in self.windows)]
        use = inside if inside else rows
        if not use:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in use for i, v in enumerate(r[3]) if v == "Active"})
        return {"sm_mhz": statistics.median(r[1] for r in use),
                "sm_max_mhz": max(r[2] for r in use), "reasons": reasons,
                "samples": len(use), "in_timed_regions": bool(inside)}


# ---------------------------------------------------------------- timing helpers

def device_time(fn, reps, stream=None):
    """Seconds of device time of reps calls of fn (CUDA events on the
    launching stream, synchronised on both sides)."""
    s = stream or torch.cuda.current_stream()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(s)
    for i in range(reps):
        fn(i)
    e1.record(s)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / 1e3


def capture(fn):
    """CUDA graph of fn() (after one eager warm-up on a side stream)."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    return g


def launches_of(fn):
    """Kernels of this library that one call of fn() launches (its launch
    counter around the call)."""
    from bf16_gemm_vla_gb300 import frt

    n0 = frt.frt_launch_count()
    fn()
    torch.cuda.synchronize()
    return frt.frt_launch_count() - n0


def l2_bytes():
    return int(getattr(torch.cuda.get_device_properties(torch.cuda.current_device()),
                       "L2_cache_size", 128 << 20))


def bf16_to_dev(bits, device):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)


# ---------------------------------------------------------------- headline step

class EncoderFP8Set:
    """One set of encoder-layer weights, inputs and outputs (static buffers)."""

    def __init__(self, src, device):
        from bf16_gemm_vla_gb300 import layers

        self.layers = []
        self.inputs = []
        for lay in src:
            if isinstance(lay, dict):
                w = torch.from_numpy(lay["w_f32"]).to(device)
                b = torch.from_numpy(lay["bias"]).to(device)
                pw = layers.prepare_fp8(w, b)
                x = bf16_to_dev(lay["a_bf16"], device)
            else:  # (Linear, input) of another set: copy to fresh buffers
                lin0, x0 = lay
                p = lin0.w
                pw = layers.PackedWeight(p.packed.clone(), p.K, p.N, p.kind, p.w_scale.clone(),
                                         p.bias.clone())
                x = x0.clone()
            self.layers.append(layers.Linear(pw, M_ENC, act_cols=0, device=device))
            self.inputs.append(x)

    def forward(self):
        for lin, x in zip(self.layers, self.inputs):
            lin(x)

    def flops(self):
        return sum(2.0 * M_ENC * lin.w.K * lin.w.N for lin in self.layers)

    def nbytes(self):
        n = 0
        for lin, x in zip(self.layers, self.inputs):
            n += lin.w.packed.numel() + x.numel() * 2 + lin.out.numel() * 2 + lin.q.numel()
        return n


def kernel_durations(sets, iters):
    """Per-layer device durations of the quantize (amax + encode) and of the
    GEMM, from events around each launch; the GPU is held busy first so the
    whole sequence is queued before it runs back to back."""
    from bf16_gemm_vla_gb300 import frt

    nl = len(sets[0].layers)
    ev = [[[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(nl)]
          for _ in range(iters)]
    torch.cuda.synchronize()
    torch.cuda._sleep(400_000_000)  # ~0.2 s at 2 GHz: longer than the enqueue below
    for it in range(iters):
        st = sets[it % len(sets)]
        for li, (lin, x) in enumerate(zip(st.layers, st.inputs)):
            ev[it][li][0].record()
            frt.frt_quantize_e4m3(x, frt.PER_TENSOR, frt.OCP, q=lin.q, scale=lin.a_scale,
                                  workspace=lin.ws)
            ev[it][li][1].record()
            frt.frt_gemm_fp8(lin.q, lin.a_scale, lin.w.packed, lin.w.w_scale, lin.w.N,
                             bias=lin.w.bias, out=lin.out, workspace=lin.gws)
            ev[it][li][2].record()
    torch.cuda.synchronize()
    quant = [[ev[it][li][0].elapsed_time(ev[it][li][1]) / 1e3 for it in range(iters)]
             for li in range(nl)]
    gemm = [[ev[it][li][1].elapsed_time(ev[it][li][2]) / 1e3 for it in range(iters)]
            for li in range(nl)]
    return quant, gemm


def back_to_back_durations(sets, reps):
    """Per-layer device durations of the quantize (amax + encode) and of the
    GEMM in steady state: each is the mean over launches of that one kernel
    back to back on rotating inputs larger than 4x L2 (the GEMM over the
    sets' weights and activations, the quantize over the sets' activations
    and copies of them), captured in one CUDA graph and timed with events
    around the replays."""
    from bf16_gemm_vla_gb300 import frt

    # each graph cycles the sets `cycles` times (at least 32 launches), so the
    # gap between two graph replays is spread over many launches
    cycles = max(1, -(-32 // len(sets)))
    quant, gemm = [], []
    for li in range(len(sets[0].layers)):
        def run_gemms(li=li):
            for _ in range(cycles):
                for st in sets:
                    lin = st.layers[li]
                    frt.frt_gemm_fp8(lin.q, lin.a_scale, lin.w.packed, lin.w.w_scale, lin.w.N,
                                     bias=lin.w.bias, out=lin.out, workspace=lin.gws)

        # the quantize reads only the activations: copies of them so that its
        # rotation too is larger than 4x L2
        xs = [st.inputs[li] for st in sets]
        per_x = xs[0].numel() * xs[0].element_size()
        extra = max(0, -(-4 * l2_bytes() // per_x) - len(xs))
        xs = xs + [xs[i % len(sets)].clone() for i in range(extra)]
        qcycles = max(1, -(-32 // len(xs)))

        def run_quants(li=li, xs=xs):
            for _ in range(qcycles):
                for i, x in enumerate(xs):
                    lin = sets[i % len(sets)].layers[li]
                    frt.frt_quantize_e4m3(x, frt.PER_TENSOR, frt.OCP, q=lin.q, scale=lin.a_scale,
                                          workspace=lin.ws)

        for fn, dst, n in ((run_quants, quant, qcycles * len(xs)),
                           (run_gemms, gemm, cycles * len(sets))):
            g = capture(fn)
            g.replay()
            secs = device_time(lambda i: g.replay(), reps)
            dst.append(secs / (reps * n))
            del g
        del xs
    return quant, gemm


def run_headline(args, device, world, sampler, peaks, peak_kind):
    from bf16_gemm_vla_gb300 import frt

    src = synth.encoder(seed=0, M=M_ENC)
    set0 = EncoderFP8Set(src, device)
    per_set = set0.nbytes()
    R = args.rotate or max(2, -(-4 * l2_bytes() // per_set))
    sets = [set0] + [EncoderFP8Set(list(zip(set0.layers, set0.inputs)), device)
                     for _ in range(R - 1)]
    torch.cuda.synchronize()  # weight copies complete before the GEMMs read them
    launches_per_step = launches_of(set0.forward)  # what one replay of a step graph runs
    graphs = [capture(s.forward) for s in sets]
    flops = set0.flops()
    for i in range(args.warmup):
        graphs[i % R].replay()
    barrier(world)
    t0 = time.time()
    secs = device_time(lambda i: graphs[i % R].replay(), args.steps)
    sampler.window(t0, time.time())
    barrier(world)
    frt.check_device_status()
    value, secs_max = aggregate(flops * args.steps, secs, world, device)

    # the same step over a longer window (50 warm-up replays, then 100 timed
    # one by one with an event after each): the median step
    long_ev = [torch.cuda.Event(enable_timing=True) for _ in range(101)]
    for i in range(50):
        graphs[i % R].replay()
    torch.cuda.synchronize()
    t0 = time.time()
    long_ev[0].record()
    for i in range(100):
        graphs[i % R].replay()
        long_ev[i + 1].record()
    torch.cuda.synchronize()
    sampler.window(t0, time.time())
    per_step = [long_ev[i].elapsed_time(long_ev[i + 1]) / 1e3 for i in range(100)]
    med = statistics.median(per_step)
    long_window = {"warmup": 50, "steps": 100, "median_ms_per_step": med * 1e3,
                   "median_tflops": flops / med / 1e12,
                   "p10_ms": sorted(per_step)[10] * 1e3, "p90_ms": sorted(per_step)[90] * 1e3,
                   "timing": "CUDA event after every replay, median over the 100 steps"}

    # per-kernel durations for the roofline: steady state (back to back);
    # event-separated launches (the quantize then the GEMM of each layer,
    # with an event between every two kernels) for reference
    iters = min(100, max(10, args.steps // 10))
    t0 = time.time()
    quant_b2b, gemm_b2b = back_to_back_durations(sets, max(5, min(50, args.steps // 20)))
    quant, gemm = kernel_durations(sets, iters)
    sampler.window(t0, time.time())
    layers_out = []
    tot_flops = 0.0
    tot_time = 0.0
    for li, lin in enumerate(set0.layers):
        g = gemm_b2b[li]
        f = 2.0 * M_ENC * lin.w.K * lin.w.N
        tot_flops += f
        tot_time += g
        layers_out.append({"K": lin.w.K, "N": lin.w.N, "gemm_us": g * 1e6,
                           "gemm_tflops": f / g / 1e12, "quantize_us": quant_b2b[li] * 1e6,
                           "gemm_us_event_separated": statistics.mean(gemm[li]) * 1e6,
                           "quantize_us_event_separated": statistics.mean(quant[li]) * 1e6})
    # the kernels are timed in bursts well under a second at full clock: the
    # burst peak is the denominator (the sustained figure was measured over
    # seconds under the power cap, at a lower clock)
    fp8_peak = fp8_peak_burst(peaks)
    # the dominant kernel: the GEMM instantiation (tile width) with the
    # largest share of the step's GEMM time, over its launches in one step
    plans = [frt.frt_gemm_describe(M_ENC, lin.w.N, lin.w.K, "e4m3") for lin in set0.layers]
    groups = {}
    for li, pl in enumerate(plans):
        groups.setdefault((pl["kind"], pl["bn"]), []).append(li)
    (kind, bn), dom = max(groups.items(), key=lambda kv: sum(gemm_b2b[i] for i in kv[1]))
    dom_flops = sum(2.0 * M_ENC * set0.layers[i].w.K * set0.layers[i].w.N for i in dom)
    dom_time = sum(gemm_b2b[i] for i in dom)
    achieved = dom_flops / dom_time / 1e12
    traffic = profiled_traffic([(M_ENC, set0.layers[i].w.K, set0.layers[i].w.N) for i in dom])
    roofline = {"bound": "tensor", "achieved": achieved, "peak": fp8_peak, "unit": "TFLOP/s",
                "frac": achieved / fp8_peak, "traffic": traffic,
                "traffic_unit": "bytes per launch (mean over the kernel's launches in a step, "
                                "ncu)",
                "kernel": "gemm_tc_kernel<fp8, %s, %d> (layers %s: %.0f%% of the step's GEMM "
                          "time)" % (kind, bn, ", ".join("%dx%d" % (set0.layers[i].w.K,
                                                                    set0.layers[i].w.N)
                                                        for i in dom),
                                     100.0 * dom_time / tot_time),
                "timing": "mean device time per launch, each layer's GEMM launched back to back "
                          "on %d rotating sets (larger than L2), cycled to at least 32 launches "
                          "per CUDA graph, CUDA events around the replays on the launching "
                          "stream" % R,
                "peak_source": "%s bf16 burst (%.1f TFLOP/s) x %.0f (nominal FP8/BF16 dense "
                               "ratio), of %s" % (peak_kind, peaks["bf16_tflops"], FP8_OVER_BF16,
                                                  peak_kind),
                "per_launch_flops": dom_flops / len(dom),
                "all_gemms": {"achieved": tot_flops / tot_time / 1e12,
                              "frac": tot_flops / tot_time / 1e12 / fp8_peak,
                              "launches_per_step": len(set0.layers)}}

    # end to end through the public API: every step copies its inputs from
    # pinned host memory, replays its graph and reads its outputs back to
    # pinned host memory.  Steps are pipelined over three streams (inputs
    # up, graph, outputs down) with the R buffer sets in rotation: a set is
    # refilled only after its previous step's graph has read it, and
    # recomputed only after that step's outputs have been read.
    h_in = [torch.empty(x.shape, dtype=x.dtype, pin_memory=True) for x in set0.inputs]
    for h, x in zip(h_in, set0.inputs):
        h.copy_(x)
    h_out = [[torch.empty(l.out.shape, dtype=l.out.dtype, pin_memory=True) for l in st.layers]
             for st in sets]
    h2d = sum(h.numel() * h.element_size() for h in h_in)
    d2h = sum(h.numel() * h.element_size() for h in h_out[0])
    up, run, down = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: torch.cuda.Event()  # noqa: E731
    computed = [ev() for _ in range(R)]  # graph of the set's last step done
    read_back = [ev() for _ in range(R)]  # outputs of the set's last step read
    used = [False] * R

    def e2e_step(i):
        r = i % R
        st = sets[r]
        filled = ev()
        with torch.cuda.stream(up):
            if used[r]:
                up.wait_event(computed[r])
            for h, x in zip(h_in, st.inputs):
                x.copy_(h, non_blocking=True)
            filled.record(up)
        with torch.cuda.stream(run):
            run.wait_event(filled)
            if used[r]:
                run.wait_event(read_back[r])
            graphs[r].replay()
            computed[r].record(run)
        with torch.cuda.stream(down):
            down.wait_event(computed[r])
            for h, lin in zip(h_out[r], st.layers):
                h.copy_(lin.out, non_blocking=True)
            read_back[r].record(down)
        used[r] = True

    def e2e_run(n):
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(up)
        run.wait_event(e0)
        down.wait_event(e0)
        for i in range(n):
            e2e_step(i)
        for s_ in (up, run):
            down.wait_stream(s_)
        e1.record(down)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / 1e3

    e2e_steps = max(10, min(args.steps, 500))
    e2e_run(min(max(args.warmup, R), 2 * R))
    barrier(world)
    t0 = time.time()
    e2e_secs = e2e_run(e2e_steps)
    sampler.window(t0, time.time())
    e2e_value, _ = aggregate(flops * e2e_steps, e2e_secs, world, device)
    # every step's outputs reached the host: the last step's equal the device's
    r_last = (e2e_steps - 1) % R
    for h, lin in zip(h_out[r_last], sets[r_last].layers):
        if not torch.equal(h, lin.out.cpu()):
            raise RuntimeError("end-to-end outputs differ from the device's")

    cfg = {"workload": ENC_WORKLOAD, "M": M_ENC,
           "layers": [[lin.w.K, lin.w.N] for lin in set0.layers],
           "weights": "N(0,0.02) fp32 -> per-channel OCP E4M3; A ~ N(0,1) bf16 with 1% x50 "
                      "outliers; bias N(0,0.1); seed 0",
           "l2": "inputs larger than L2: %d rotating sets of weights+activations+outputs, "
                 "%.0f MB in total (L2 %.0f MB)" % (R, R * per_set / 1e6, l2_bytes() / 1e6),
           "parallelism": "replicas" if world > 1 else "single GPU"}
    return {
        "value": value / 1e12, "secs": secs_max, "flops_per_step": flops, "config": cfg,
        "roofline": roofline, "layers": layers_out,
        "e2e": {"value": e2e_value / 1e12, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                "pipelining": "inputs up, graph and outputs down on three streams, %d buffer "
                              "sets in rotation" % R},
        "launches_per_step": launches_per_step, "long_window": long_window,
    }


# ---------------------------------------------------------------- components

def gemm_stream_rate(lay, kind, device, sampler, reps=3, geglu=False):
    """Per-launch device time of one layer's GEMM, over rotating weight copies
    (total > 4x L2) captured back to back in one graph.  geglu: the layer is a
    merged gate/up and the GEMM writes gelu(gate) * up (N / 2 columns)."""
    from bf16_gemm_vla_gb300 import frt, layers

    w = torch.from_numpy(lay["w_f32"]).to(device)
    b = torch.from_numpy(lay["bias"]).to(device)
    x = bf16_to_dev(lay["a_bf16"], device)
    pw = layers.prepare_fp8(w, b) if kind == "e4m3" else layers.prepare_bf16(w, b)
    wbytes = pw.packed.numel()
    copies = max(4, -(-4 * l2_bytes() // wbytes))
    copies = min(copies, 256)
    packs = [pw.packed] + [pw.packed.clone() for _ in range(copies - 1)]
    torch.cuda.synchronize()  # weight copies complete before the GEMMs read them
    lin = layers.Linear(pw, lay["M"], act_cols=lay["act_cols"], device=device)
    if kind == "e4m3":
        frt.frt_quantize_e4m3(x, frt.PER_TENSOR, frt.OCP, q=lin.q, scale=lin.a_scale,
                              workspace=lin.ws)
    out = lin.out[:, :pw.N // 2] if geglu else lin.out
    act_cols = 0 if geglu else lay["act_cols"]

    def run_all():
        for p in packs:
            if kind == "e4m3":
                frt.frt_gemm_fp8(lin.q, lin.a_scale, p, pw.w_scale, pw.N, bias=b,
                                 act_cols=act_cols, out=out, workspace=lin.gws, geglu=geglu)
            else:
                frt.frt_gemm_bf16(x, p, pw.N, bias=b, act_cols=act_cols, out=out,
                                  workspace=lin.gws, geglu=geglu)

    g = capture(run_all)
    g.replay()
    t0 = time.time()
    secs = device_time(lambda i: g.replay(), reps)
    sampler.window(t0, time.time())
    per = secs / (reps * copies)
    flops = 2.0 * lay["M"] * lay["K"] * lay["N"]
    del packs, g
    return {"K": lay["K"], "N": lay["N"], "us": per * 1e6, "weight_bytes": wbytes,
            "weight_gbs": wbytes / per / 1e9, "tflops": flops / per / 1e12, "copies": copies}


def run_components(args, device, sampler, peaks):
    from bf16_gemm_vla_gb300 import frt
    from bf16_gemm_vla_gb300.stack import SyntheticStack

    out = {}
    hbm = peaks["hbm_gbs"]
    fp8_peak = fp8_peak_burst(peaks)
    bf16_peak = peaks["bf16_tflops"]
    # decoder-shaped GEMMs, weight-stream GB/s (each layer's GEMM back to
    # back over its own rotating weight copies)
    dec = synth.decoder(seed=0, M=M_DEC)
    for kind in ("e4m3", "bf16"):
        rows = [gemm_stream_rate(lay, kind, device, sampler) for lay in dec]
        for r in rows:
            r["frac_of_hbm"] = r["weight_gbs"] / hbm
        tb = sum(r["weight_bytes"] for r in rows)
        tt = sum(r["us"] for r in rows) / 1e6
        out["decoder_m50_" + ("fp8" if kind == "e4m3" else "bf16")] = {
            "layers": rows, "weight_gbs": tb / tt / 1e9, "frac_of_hbm": tb / tt / 1e9 / hbm}
    # the decoder as a dependent chain: 18 layers of qkv -> o -> gate/up ->
    # down at M = 50 (each GEMM reads the previous one's output), one graph
    out.update(decoder_chains(device, sampler, hbm))
    # encoder-shaped BF16 GEMMs
    enc = synth.encoder(seed=0, M=M_ENC)
    rows = [gemm_stream_rate(lay, "bf16", device, sampler, reps=2) for lay in enc]
    for r in rows:
        r["frac_of_bf16_peak"] = r["tflops"] / bf16_peak
    tf = sum(2.0 * M_ENC * r["K"] * r["N"] for r in rows)
    tt = sum(r["us"] for r in rows) / 1e6
    out["encoder_m768_bf16"] = {"layers": rows, "tflops": tf / tt / 1e12,
                                "frac_of_bf16_peak": tf / tt / 1e12 / bf16_peak}
    del enc
    # the merged encoder gate/up (2048 -> 2 x 16384, the stack's FFN) at M=768:
    # one GEMM writing both halves (GELU on the gate half) against the same
    # GEMM with the GeGLU fused (gelu(gate) * up, half the output)
    gu = synth.layer(np.random.default_rng(7), M_ENC, 2048, 2 * 16384, act_cols=16384,
                     outlier_frac=0.01)
    fl = 2.0 * M_ENC * 2048 * 2 * 16384
    both = {"unfused": gemm_stream_rate(gu, "e4m3", device, sampler, reps=2),
            "fused_geglu": gemm_stream_rate(gu, "e4m3", device, sampler, reps=2, geglu=True)}
    for v in both.values():
        v["frac_of_fp8_peak"] = fl / (v["us"] * 1e-6) / 1e12 / fp8_peak
    out["encoder_gate_up_fp8_m768"] = both
    del gu
    # the decoder's merged gate/up (1024 -> 2 x 4096) at M=50, BF16 and FP8
    gu = synth.layer(np.random.default_rng(8), M_DEC, 1024, 2 * 4096, act_cols=4096)
    for kind in ("bf16", "e4m3"):
        out["decoder_gate_up_m50_" + ("fp8" if kind == "e4m3" else "bf16")] = {
            "unfused": gemm_stream_rate(gu, kind, device, sampler),
            "fused_geglu": gemm_stream_rate(gu, kind, device, sampler, geglu=True)}
    del gu
    # the BF16 decoder block boundary at M=50, hidden 1024 (gated residual
    # update + adaptive RMS norm in one launch), back to back over 64 sets
    H = 1024
    gen = torch.Generator(device=device)
    gen.manual_seed(9)
    bsets = [[(torch.randn((M_DEC, w), generator=gen, device=device) * sd).to(torch.bfloat16)
              for w, sd in ((H, 1.0), (H, 1.0), (H, 1.0), (3 * H, 0.1))] for _ in range(64)]
    bouts = [(torch.empty((M_DEC, H), dtype=torch.bfloat16, device=device),
              torch.empty((M_DEC, H), dtype=torch.bfloat16, device=device)) for _ in bsets]

    def boundary_all():
        for (res, o, gt, sty), (nrm, nxt) in zip(bsets, bouts):
            frt.frt_gate_residual_ada_norm_bf16(res, o, gt, sty, normalized=nrm, next_gate=nxt)

    gb = capture(boundary_all)
    gb.replay()
    t0 = time.time()
    secs = device_time(lambda i: gb.replay(), 20) / (20 * len(bsets))
    sampler.window(t0, time.time())
    nbytes = M_DEC * H * 2 * (2 + 1 + 1 + 3 + 1 + 1)  # residual r/w, output, gate, style, 2 outputs
    out["decoder_boundary_m50_h1024"] = {"us": secs * 1e6, "bytes": nbytes,
                                         "gbs": nbytes / secs / 1e9,
                                         "note": "latency-bound: 0.9 MB per call, L2-resident"}
    del gb, bsets, bouts
    # the encoder FP8 step with each layer's activation scale calibrated once
    # (on that layer's input) and frozen: the quantize is one encode pass
    set0 = EncoderFP8Set(synth.encoder(seed=0, M=M_ENC), device)
    R = max(2, -(-4 * l2_bytes() // set0.nbytes()))
    sets = [set0] + [EncoderFP8Set(list(zip(set0.layers, set0.inputs)), device)
                     for _ in range(R - 1)]
    scales = [[lin.calibrate([x]) for lin, x in zip(st_.layers, st_.inputs)] for st_ in sets]
    graphs = [capture(st_.forward) for st_ in sets]
    for i in range(3):
        graphs[i % R].replay()
    steps = max(20, min(args.steps, 500))
    t0 = time.time()
    secs = device_time(lambda i: graphs[i % R].replay(), steps) / steps
    sampler.window(t0, time.time())
    frt.check_device_status()
    qus = []
    for li in range(len(set0.layers)):
        # the sets' activations and copies of them: more than 4x L2
        xs = [st_.inputs[li] for st_ in sets]
        per_x = xs[0].numel() * xs[0].element_size()
        xs = xs + [xs[i % R].clone() for i in range(max(0, -(-4 * l2_bytes() // per_x) - R))]

        def qrun(li=li, xs=xs):
            for i, x in enumerate(xs):
                lin = sets[i % R].layers[li]
                frt.frt_quantize_e4m3(x, frt.PER_TENSOR, frt.OCP,
                                      static_scale=lin.a_scale, q=lin.q, scale=lin.s_out)
        g = capture(qrun)
        g.replay()
        qus.append(device_time(lambda i: g.replay(), 20) / (20 * len(xs)) * 1e6)
        del g, xs
    out["encoder_m768_fp8_static_scale"] = {
        "tflops": set0.flops() / secs / 1e12, "ms_per_step": secs * 1e3,
        "launches_per_step": launches_of(set0.forward), "scales": scales[0],
        "quantize_us": qus,
        "quantize_gbs_3B_per_elem": [3.0 * M_ENC * lin.w.K / (u * 1e-6) / 1e9
                                     for lin, u in zip(set0.layers, qus)]}
    del sets, graphs, set0
    torch.cuda.empty_cache()
    # quantize, 256 Mi Student-t bf16 (two passes: 2 B + 2 B read, 1 B written)
    n = 256 << 20
    x = bf16_to_dev(synth.student_t_bf16(n, seed=3).reshape(-1, 4096), device)
    q = torch.empty(x.shape, dtype=torch.uint8, device=device)
    s = torch.empty(1, dtype=torch.float32, device=device)
    ws = torch.zeros(frt.frt_quantize_workspace_bytes(x.shape[0], x.shape[1]) // 4,
                     dtype=torch.float32, device=device)

    def quant(i):
        frt.frt_quantize_e4m3(x, frt.PER_TENSOR, frt.OCP, q=q, scale=s, workspace=ws)

    quant(0)
    t0 = time.time()
    secs = device_time(quant, 10) / 10
    sampler.window(t0, time.time())
    out["quantize_256Mi_bf16"] = {"us": secs * 1e6, "gbs_5B_per_elem": 5.0 * n / secs / 1e9,
                                  "gbs_3B_per_elem": 3.0 * n / secs / 1e9,
                                  "frac_of_hbm": 5.0 * n / secs / 1e9 / hbm}
    del x, q
    # FNUZ -> OCP over 1 GiB
    nb = 1 << 30
    src = torch.from_numpy(synth.uniform_bytes(nb, seed=2)).to(device)
    dst = torch.empty_like(src)
    frt.frt_fnuz_to_ocp(src, out=dst)
    t0 = time.time()
    secs = device_time(lambda i: frt.frt_fnuz_to_ocp(src, out=dst), 10) / 10
    sampler.window(t0, time.time())
    out["fnuz_to_ocp_1GiB"] = {"us": secs * 1e6, "gbs": 2.0 * nb / secs / 1e9,
                               "frac_of_hbm": 2.0 * nb / secs / 1e9 / hbm}
    del src, dst
    torch.cuda.empty_cache()
    # the synthetic 18+18-layer stack, one CUDA graph per replay
    st = SyntheticStack(n_layers=18, seed=1, device=device, keep=())
    xe, xd = synth.stack_inputs(seed=1)
    st.x_enc.copy_(bf16_to_dev(xe, device))
    st.x_dec.copy_(bf16_to_dev(xd, device))
    st.capture()
    st.replay()
    t0 = time.time()
    secs = device_time(lambda i: st.replay(), 10) / 10
    sampler.window(t0, time.time())
    frt.check_device_status()
    out["stack_18enc_fp8_18dec_bf16"] = {"ms_per_replay": secs * 1e3,
                                         "launches_per_replay": launches_of(st.forward),
                                         "weight_bytes": st.weight_bytes(),
                                         "kernels": stack_kernel_table(st, sampler, peaks,
                                                                       secs)}
    del st
    torch.cuda.empty_cache()
    out["nvfp4_encoder_ffn_m768"] = nvfp4_ffn(device, sampler, peaks)
    if not args.no_sweep:
        out["sweep_k4096_n4096"] = run_sweep(device, sampler, peaks)
    return out


FP4_OVER_BF16 = 6.0  # nominal dense ratio, 13.5 / 2.25 PFLOP/s


def nvfp4_ffn(device, sampler, peaks):
    """The encoder FFN on NVFP4 operands at M = 768: the merged gate/up
    2048 -> 2 x 16384 (GELU on the gate half) and down 16384 -> 2048, each
    GEMM back to back over rotating weight copies (> 4x L2), and the NVFP4
    activation quantize (amax + encode) of each input.  The fraction is of
    the dense FP4 peak taken as the measured BF16 burst x 6 (nominal ratio;
    no FP4 measurement)."""
    from bf16_gemm_vla_gb300 import frt, layers

    fp4_peak = peaks["bf16_tflops"] * FP4_OVER_BF16
    g = torch.Generator(device=device)
    g.manual_seed(12)
    rows = []
    for K, N, act in ((2048, 2 * 16384, 16384), (16384, 2048, 0)):
        w = torch.randn((K, N), generator=g, device=device) * 0.02
        b = torch.randn((N,), generator=g, device=device) * 0.1
        pw = layers.prepare_nvfp4(w, b)
        del w
        wbytes = pw.packed.numel() + pw.sf.numel()
        copies = min(64, max(4, -(-4 * l2_bytes() // wbytes)))
        ws = [(pw.packed, pw.sf)] + [(pw.packed.clone(), pw.sf.clone()) for _ in range(copies - 1)]
        x = torch.randn((M_ENC, K), generator=g, device=device).to(torch.bfloat16)
        qa, sfa, ga = frt.frt_quantize_nvfp4(x)
        out = torch.empty((M_ENC, N), dtype=torch.bfloat16, device=device)
        torch.cuda.synchronize()

        def run_gemm():
            for pk, sf in ws:
                frt.frt_gemm_nvfp4(qa, sfa, ga, pk, sf, pw.g, N, bias=b, act_cols=act, out=out)

        gr = capture(run_gemm)
        gr.replay()
        t0 = time.time()
        per = device_time(lambda i: gr.replay(), 5) / (5 * copies)
        sampler.window(t0, time.time())
        nws = frt.nvfp4_workspace(device)
        # the activation quantize over copies of x larger than 4x L2
        xs = [x] + [x.clone() for _ in range(max(0, -(-4 * l2_bytes() // (x.numel() * 2)) - 1))]

        def run_quant():
            for xc in xs:
                frt.frt_quantize_nvfp4(xc, q=qa, sf=sfa, scale=ga, workspace=nws)

        gq = capture(run_quant)
        gq.replay()
        qper = device_time(lambda i: gq.replay(), 5) / (5 * len(xs))
        frt.check_device_status()
        tf = 2.0 * M_ENC * N * K / per / 1e12
        rows.append({"K": K, "N": N, "act_cols": act, "us": per * 1e6, "tflops": tf,
                     "frac_of_fp4_peak": tf / fp4_peak, "weight_bytes": wbytes,
                     "quantize_us": qper * 1e6, "copies": copies})
        del ws, gr, gq, pw, xs
        torch.cuda.empty_cache()
    return {"layers": rows, "fp4_peak": fp4_peak,
            "peak_source": "measured bf16 burst x %.0f (nominal FP4/BF16 dense ratio)"
                           % FP4_OVER_BF16,
            "kernel": "gemm_nvfp4_pair_kernel (256-row tiles on CTA pairs, 256 or 128 channels "
                      "wide; tcgen05 kind::mxf4nvf4 with E4M3 block scales per 16)"}


def run_sweep(device, sampler, peaks):
    """Sweep (i): M in {1 ... 1024} at K = N = 4096, FP8 against BF16, each
    GEMM back to back over rotating weight copies (> 4x L2).  Both bounds
    are reported at every M (weight GB/s of HBM, TFLOP/s of the dtype's dense
    peak); the crossover is the smallest M from which the FP8 GEMM stays
    faster than the BF16 one."""
    hbm = peaks["hbm_gbs"]
    rows = []
    for M in synth.SWEEP_M:
        lay = synth.sweep_gemm(M, seed=M)
        a = gemm_stream_rate(lay, "e4m3", device, sampler, reps=2)
        b = gemm_stream_rate(lay, "bf16", device, sampler, reps=2)
        rows.append({"M": M, "fp8_us": a["us"], "bf16_us": b["us"],
                     "fp8_tflops": a["tflops"], "bf16_tflops": b["tflops"],
                     "fp8_frac_of_fp8_peak": a["tflops"] / fp8_peak_burst(peaks),
                     "bf16_frac_of_bf16_peak": b["tflops"] / peaks["bf16_tflops"],
                     "fp8_weight_gbs": a["weight_gbs"], "bf16_weight_gbs": b["weight_gbs"],
                     "fp8_weight_frac_of_hbm": a["weight_gbs"] / hbm,
                     "bf16_weight_frac_of_hbm": b["weight_gbs"] / hbm,
                     "fp8_faster": a["us"] < b["us"]})
    crossover = None
    for i in range(len(rows)):
        if all(r["fp8_faster"] for r in rows[i:]):
            crossover = rows[i]["M"]
            break
    small = [r for r in rows if r["M"] <= 64]
    return {"rows": rows, "fp8_faster_from_M": crossover,
            "min_weight_frac_of_hbm_M_le_64": {
                "fp8": min(r["fp8_weight_frac_of_hbm"] for r in small),
                "bf16": min(r["bf16_weight_frac_of_hbm"] for r in small)}}


def decoder_chains(device, sampler, hbm):
    """The decoder's 18 layers as one dependent chain at M = 50 (qkv 1024 ->
    2560, o 2048 -> 1024, merged gate/up 1024 -> 2 x 4096 with GELU on the
    gate half, down 4096 -> 1024; each GEMM reads the previous one's output),
    BF16 and FP8 (the FP8 chain quantizes each GEMM's input per tensor),
    replayed as one CUDA graph: weight bytes / replay time."""
    from bf16_gemm_vla_gb300 import frt
    from bf16_gemm_vla_gb300.stack import SyntheticStack

    out = {}
    xd = synth.stack_inputs(seed=1)[1]
    for kind in ("bf16", "e4m3"):
        st = SyntheticStack(n_layers=18, seed=1, device=device, dec_kind=kind, keep=(),
                            parts=("dec",))
        st.x_dec.copy_(bf16_to_dev(xd, device))
        st.capture()
        st.replay()
        t0 = time.time()
        secs = device_time(lambda i: st.replay(), 20) / 20
        sampler.window(t0, time.time())
        frt.check_device_status()
        wb = st.weight_bytes()
        n_launch = launches_of(st.forward)
        out["decoder_chain_m50_" + ("fp8" if kind == "e4m3" else "bf16")] = {
            "layers": 18, "us_per_replay": secs * 1e6, "weight_bytes": wb,
            "weight_gbs": wb / secs / 1e9, "frac_of_hbm": wb / secs / 1e9 / hbm,
            "launches_per_replay": n_launch, "us_per_launch": secs * 1e6 / n_launch,
            "l2": "weights %.0f MB per replay (L2 %.0f MB)" % (wb / 1e6, l2_bytes() / 1e6)}
        del st
        torch.cuda.empty_cache()
    return out


def stack_kernel_table(st, sampler, peaks, replay_secs):
    """Per-kernel figures of one stack replay: for each distinct launch
    (chain, layer name, quantize or GEMM) the mean device time per launch,
    from a CUDA graph of that launch over all 18 layers' own buffers
    (weights, inputs, outputs) back to back, and its fraction of the bound
    that applies: dense FP8/BF16 peak for the M = 768 GEMMs, HBM on weight
    bytes for the M = 50 GEMMs, HBM at 3 B per element for the quantize."""
    from bf16_gemm_vla_gb300 import frt

    hbm = peaks["hbm_gbs"]
    groups = {}
    for part, li, name, op, lin, call in st.op_list():
        groups.setdefault((part, name, op), []).append((lin, call))
    rows = []
    total = 0.0
    for (part, name, op), items in groups.items():
        def run(items=items):
            for _, c in items:
                c()

        g = capture(run)
        g.replay()
        t0 = time.time()
        per = device_time(lambda i: g.replay(), 10) / (10 * len(items))
        sampler.window(t0, time.time())
        del g
        lin = items[0][0]
        M, K, N = lin.M, lin.w.K, lin.w.N
        row = {"chain": part, "layer": name, "op": op, "M": M, "K": K, "N": N,
               "launches": len(items), "us": per * 1e6}
        if op in ("quantize", "encode"):
            row["kernel"] = ("quantize (per tensor, dynamic)" if op == "quantize" else
                             "quantize encode pass (per tensor, scale taken by the GEMM before)")
            row["gbs_3B_per_elem"] = 3.0 * M * K / per / 1e9
            row["bound"] = "hbm"
            row["frac"] = row["gbs_3B_per_elem"] / hbm
        else:
            pl = frt.frt_gemm_describe(M, N, K, lin.w.kind)
            row["kernel"] = "gemm_tc_kernel<%s, %s, %d>%s" % (
                "fp8" if lin.w.kind == "e4m3" else "bf16", pl["kind"], pl["bn"],
                " taking the next layer's scale" if op == "gemm+scale" else "")
            row["tflops"] = 2.0 * M * N * K / per / 1e12
            row["weight_gbs"] = lin.w.packed.numel() / per / 1e9
            if M > 128:
                row["bound"] = "tensor"
                row["frac"] = row["tflops"] / (fp8_peak_burst(peaks) if lin.w.kind == "e4m3"
                                               else peaks["bf16_tflops"])
            else:
                row["bound"] = "hbm (weights)"
                row["frac"] = row["weight_gbs"] / hbm
        total += per * len(items)
        rows.append(row)
    return {"rows": rows, "sum_of_kernel_us": total * 1e6, "replay_us": replay_secs * 1e6,
            "timing": "mean per launch over the 18 layers' launches of that kind back to back "
                      "in one CUDA graph (events around 10 replays); the sum runs the kinds "
                      "separately, so it differs from the replay by the overlap between "
                      "neighbouring kernels"}


# ---------------------------------------------------------------- CPU oracle (baseline / reference arm)

def oracle_sample_step(src, rows, cols):
    """One sample of the headline step on the CPU oracle: per encoder layer,
    quantize `rows` activation rows, then the FP8 layer on the first `cols`
    output channels (weights quantized at load).  Returns FLOPs done."""
    from oracle import e4m3, gemm, quantize

    flops = 0.0
    for lay in src:
        a = synth.bf16_bits_as_f32(lay["a_bf16"][:rows])
        qa, sa = quantize.quantize_e4m3(a, quantize.PER_TENSOR, e4m3.OCP)
        qw, sw = lay["_oracle_w"]
        gemm.gemm_fp8(qa, e4m3.OCP, sa, qw[:, :cols], e4m3.OCP, sw[:cols], lay["bias"][:cols], 0)
        flops += 2.0 * rows * lay["K"] * cols
    return flops


def oracle_setup(cols):
    from oracle import e4m3, quantize

    src = synth.encoder(seed=0, M=M_ENC)
    for lay in src:
        lay["_oracle_w"] = quantize.quantize_e4m3(lay["w_f32"][:, :cols], quantize.PER_COL,
                                                  e4m3.OCP)
    return src


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count()


def cpu_baseline(budget_s=12.0, rows=16, cols=256):
    src = oracle_setup(cols)
    oracle_sample_step(src, rows, cols)  # warm
    flops = 0.0
    t0 = time.perf_counter()
    n = 0
    while time.perf_counter() - t0 < budget_s:
        flops += oracle_sample_step(src, rows, cols)
        n += 1
    secs = time.perf_counter() - t0
    return {"value": flops / secs / 1e12, "unit": "TFLOP/s", "cores": cpu_cores(), "kind": "oracle",
            "sample": "%d steps of %d activation rows x the first %d output channels of each "
                      "encoder layer (quantize + fp64 GEMM + epilogue), %.1f s" % (n, rows, cols, secs)}


def run_reference(args):
    rank, _, world = dist_env()
    if rank != 0:
        return 0
    rows = 16
    cols = 256
    src = oracle_setup(cols)
    t0 = time.perf_counter()
    oracle_sample_step(src, rows, cols)
    one = time.perf_counter() - t0
    budget = 150.0 / max(1, args.steps + args.warmup)
    while one > budget and cols > 16:
        cols //= 2
        one /= 2
    src = oracle_setup(cols)
    for _ in range(args.warmup):
        oracle_sample_step(src, rows, cols)
    t0 = time.perf_counter()
    flops = 0.0
    for _ in range(args.steps):
        flops += oracle_sample_step(src, rows, cols)
    secs = time.perf_counter() - t0
    value = flops / secs / 1e12
    sample = ("%d activation rows x the first %d output channels of each encoder layer per step "
              "(quantize + fp64 GEMM + epilogue)" % (rows, cols))
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": secs / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": ENC_WORKLOAD + " (CPU oracle, bounded sample)", "M": M_ENC,
                       "sample": sample},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cpu_cores(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


# ---------------------------------------------------------------- main

def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        return run_reference(args)
    rank, local_rank, world = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device (GB300); the library has no CPU path")
    torch.cuda.set_device(local_rank)
    device = torch.device("cuda", local_rank)
    init_dist(world)
    from bf16_gemm_vla_gb300 import build

    if rank == 0:
        build.build()
    barrier(world)
    peaks, peak_kind = load_peaks()
    sampler = ClockSampler(local_rank)
    sampler.start()
    try:
        head = run_headline(args, device, world, sampler, peaks, peak_kind)
        comps = None if args.no_components else run_components(args, device, sampler, peaks)
        t0 = time.time()
        fp8_measured = measure_fp8_peak(device)
        sampler.window(t0, time.time())
    finally:
        clocks = sampler.stop()
    roof = head["roofline"]
    roof["measured_fp8_peak"] = fp8_measured
    roof["frac_of_measured_fp8_peak"] = (roof["achieved"] / fp8_measured
                                         if fp8_measured else None)
    cpu = cpu_baseline() if (rank == 0 and world == 1) else None
    if rank == 0:
        line = {
            "metric": METRIC, "value": head["value"], "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": head["secs"] / args.steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "e4m3", "data": "synthetic",
            "config": head["config"], "roofline": head["roofline"], "cpu_baseline": cpu,
            "e2e": head["e2e"],
            "gpu_launches": head["launches_per_step"] * args.steps,
            "clocks": clocks, "layers": head["layers"], "components": comps,
            "peaks": {"source": peak_kind, "hbm_gbs": peaks["hbm_gbs"],
                      "bf16_tflops": peaks["bf16_tflops"],
                      "bf16_tflops_sustained": peaks["bf16_tflops_sustained"],
                      "fp8_tflops_burst": fp8_peak_burst(peaks),
                      "fp8_tflops_measured_this_run": fp8_measured,
                      "fp8_measured_how": "torch._scaled_mm (cuBLAS) E4M3 8192^3 -> bf16, best "
                                          "of 10, CUDA events"},
            "long_window": head["long_window"],
        }
        print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
