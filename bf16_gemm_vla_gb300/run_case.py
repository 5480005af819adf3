"""Runs one layer of the path a few times, for profiling (e.g. under ncu).

    python -m bf16_gemm_vla_gb300.run_case --kind fp8 --M 50 --K 1024 --N 4096 --reps 3
    python -m bf16_gemm_vla_gb300.run_case --kind nvfp4 --M 768 --K 2048 --N 16384 --reps 3
    python -m bf16_gemm_vla_gb300.run_case --op quantize --M 768 --K 16384 --reps 3
    python -m bf16_gemm_vla_gb300.run_case --op nvfp4_quantize --M 768 --K 16384 --reps 3

Synthetic inputs are drawn on the device (seeded): activations N(0,1) bf16,
weights N(0,0.02), bias N(0,0.1).  The FP8 path quantizes the activations
per tensor and the weights per output channel (load time, before the timed
launches), then launches the GEMM `reps` times; --with-quantize repeats the
activation quantize before each GEMM.  Prints the mean device time per
launch (CUDA events) unless --quiet.
"""
import argparse

import torch

from . import frt, layers


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--kind", choices=("fp8", "bf16", "nvfp4"), default="fp8")
    ap.add_argument("--M", type=int, default=50)
    ap.add_argument("--K", type=int, default=1024)
    ap.add_argument("--N", type=int, default=4096)
    ap.add_argument("--act-cols", type=int, default=0)
    ap.add_argument("--reps", type=int, default=3)
    ap.add_argument("--with-quantize", action="store_true")
    ap.add_argument("--quiet", action="store_true")
    ap.add_argument("--op", choices=("gemm", "quantize", "nvfp4_quantize"), default="gemm")
    ap.add_argument("--static-scale", action="store_true")
    a = ap.parse_args(argv)
    dev = torch.device("cuda")
    if a.op == "quantize":
        return quantize_case(a, dev)
    if a.op == "nvfp4_quantize":
        g = torch.Generator(device=dev)
        g.manual_seed(0)
        x = torch.randn((a.M, a.K), generator=g, device=dev).to(torch.bfloat16)
        q, sf, s = frt.frt_quantize_nvfp4(x)
        ws = frt.nvfp4_workspace(dev)
        return _time(a, lambda: frt.frt_quantize_nvfp4(x, q=q, sf=sf, scale=s, workspace=ws),
                     "nvfp4 quantize %d x %d" % (a.M, a.K))
    g = torch.Generator(device=dev)
    g.manual_seed(0)
    x = torch.randn((a.M, a.K), generator=g, device=dev).to(torch.bfloat16)
    w = torch.randn((a.K, a.N), generator=g, device=dev) * 0.02
    b = torch.randn((a.N,), generator=g, device=dev) * 0.1
    if a.kind == "nvfp4":
        return nvfp4_case(a, x, w, b)
    pw = layers.prepare_fp8(w, b) if a.kind == "fp8" else layers.prepare_bf16(w, b)
    lin = layers.Linear(pw, a.M, act_cols=a.act_cols)
    if a.kind == "fp8":
        frt.frt_quantize_e4m3(x, frt.PER_TENSOR, frt.OCP, q=lin.q, scale=lin.a_scale,
                              workspace=lin.ws)

    def once():
        if a.kind == "fp8":
            if a.with_quantize:
                return lin(x)
            return frt.frt_gemm_fp8(lin.q, lin.a_scale, pw.packed, pw.w_scale, pw.N, bias=b,
                                    act_cols=a.act_cols, out=lin.out, workspace=lin.gws)
        return lin(x)

    once()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(a.reps):
        once()
    e1.record()
    torch.cuda.synchronize()
    frt.check_device_status()
    if not a.quiet:
        print("%s M=%d K=%d N=%d: %.2f us per launch" % (a.kind, a.M, a.K, a.N,
                                                          e0.elapsed_time(e1) * 1e3 / a.reps))


def _time(a, once, what):
    once()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(a.reps):
        once()
    e1.record()
    torch.cuda.synchronize()
    frt.check_device_status()
    if not a.quiet:
        print("%s: %.2f us per launch" % (what, e0.elapsed_time(e1) * 1e3 / a.reps))


def nvfp4_case(a, x, w, b):
    pw = layers.prepare_nvfp4(w, b)
    qa, sfa, ga = frt.frt_quantize_nvfp4(x)
    out = torch.empty((a.M, a.N), dtype=torch.bfloat16, device=x.device)
    _time(a, lambda: frt.frt_gemm_nvfp4(qa, sfa, ga, pw.packed, pw.sf, pw.g, a.N, bias=pw.bias,
                                        act_cols=a.act_cols, out=out),
          "nvfp4 M=%d K=%d N=%d" % (a.M, a.K, a.N))


def quantize_case(a, dev):
    g = torch.Generator(device=dev)
    g.manual_seed(0)
    x = torch.randn((a.M, a.K), generator=g, device=dev).to(torch.bfloat16)
    q = torch.empty((a.M, a.K), dtype=torch.uint8, device=dev)
    s = torch.empty((1,), dtype=torch.float32, device=dev)
    ws = torch.zeros((4096,), dtype=torch.float32, device=dev)  # header zero-filled once
    cal = torch.empty((1,), dtype=torch.float32, device=dev)
    frt.frt_quantize_e4m3(x, q=q, scale=cal, workspace=ws)  # the calibrated static scale

    def once():
        frt.frt_quantize_e4m3(x, static_scale=cal if a.static_scale else None, q=q, scale=s,
                              workspace=ws)

    once()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(a.reps):
        once()
    e1.record()
    torch.cuda.synchronize()
    if not a.quiet:
        print("quantize %d x %d: %.2f us per call" % (a.M, a.K, e0.elapsed_time(e1) * 1e3 / a.reps))


if __name__ == "__main__":
    main()
