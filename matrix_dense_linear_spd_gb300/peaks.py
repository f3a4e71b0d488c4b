"""Measure the arithmetic peaks that the roofline fractions are taken against.

Runs each microbenchmark kernel of ``bl_debug_peak`` (FP32 FFMA and packed FFMA2, FP64 DFMA and
DMMA, tcgen05 kind::tf32 and kind::f16/bf16) on the current GPU: the loop count is grown until a
launch takes at least ``--min-ms``, then the best of ``--reps`` launches (CUDA events on the
launching stream) gives the rate. The SM clock is sampled through NVML while the kernels run;
no GPU setting is changed. Writes ``profiles/fp_peaks.json`` (or ``--out``) and prints a table.

Derived figures recorded next to the rates:
  fp32      max(FFMA, FFMA2): the best FP32-accurate SIMT rate
  tf32x3    TF32 tensor rate / 3: the f32-accurate rate of the 3xTF32 split (three products)
  f32_roof  max(fp32, tf32x3): the FP32-accurate roof of an f32 factorisation on this GPU
  fp64      max(DFMA, DMMA)

Usage: python -m matrix_dense_linear_spd_gb300.peaks [--out PATH] [--min-ms 20] [--reps 5]
"""
from __future__ import annotations

import argparse
import ctypes
import json
import os
import sys
import time

_ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if _ROOT not in sys.path:
    sys.path.insert(0, _ROOT)

import matrix_dense_linear_spd_gb300 as bl  # noqa: E402

KINDS = {"ffma": 0, "ffma2": 1, "dfma": 2, "dmma": 3, "tf32": 4, "bf16": 5}


def measure(kind: str, sms: int, min_ms: float, reps: int, torch):
    lib = bl.get_lib()
    code = KINDS[kind]
    tc = kind in ("tf32", "bf16")
    blocks = sms if tc else sms * 8
    scratch = torch.zeros(4096, dtype=torch.float64, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    s = torch.cuda.current_stream()
    iters = 64
    flops = ctypes.c_double(0)
    best = None
    for _ in range(40):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s)
        st = lib.bl_debug_peak(code, blocks, iters, ctypes.c_void_p(scratch.data_ptr()),
                               ctypes.c_void_p(status.data_ptr()), ctypes.byref(flops), ctypes.c_void_p(s.cuda_stream))
        e1.record(s)
        torch.cuda.synchronize()
        if st != 0:
            raise RuntimeError(f"bl_debug_peak({kind}) failed: {bl.get_lib().bl_last_error().decode()}")
        ms = e0.elapsed_time(e1)
        if ms >= min_ms:
            break
        iters = int(iters * max(2.0, 1.2 * min_ms / max(ms, 1e-3)))
    times = []
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s)
        lib.bl_debug_peak(code, blocks, iters, ctypes.c_void_p(scratch.data_ptr()),
                          ctypes.c_void_p(status.data_ptr()), ctypes.byref(flops), ctypes.c_void_p(s.cuda_stream))
        e1.record(s)
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1))
    if int(status.item()) != 0:
        raise RuntimeError(f"{kind}: a tensor-core wait gave up")
    best = min(times)
    return {"tflops": flops.value / (best / 1e3) / 1e12, "ms": best, "iters": iters, "blocks": blocks,
            "flops_per_launch": flops.value}


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--out", default=os.path.join(_ROOT, "profiles", "fp_peaks.json"))
    ap.add_argument("--min-ms", type=float, default=20.0)
    ap.add_argument("--reps", type=int, default=5)
    ap.add_argument("--kinds", default=",".join(KINDS))
    a = ap.parse_args(argv)
    import torch
    from matrix_dense_linear_spd_gb300.clocks import ClockSampler
    props = torch.cuda.get_device_properties(0)
    sms = props.multi_processor_count
    sampler = ClockSampler(0).start()
    t0 = time.perf_counter()
    res = {}
    for k in a.kinds.split(","):
        res[k] = measure(k, sms, a.min_ms, a.reps, torch)
        print(f"{k:6s} {res[k]['tflops']:10.2f} TFLOP/s  ({res[k]['ms']:.2f} ms, {res[k]['blocks']} CTAs)", flush=True)
    t1 = time.perf_counter()
    sampler.stop()
    clk = sampler.summary(t0, t1)
    g = lambda k: res[k]["tflops"] if k in res else 0.0
    derived = {"fp32": max(g("ffma"), g("ffma2")), "tf32x3": g("tf32") / 3.0,
               "fp64": max(g("dfma"), g("dmma"))}
    derived["f32_roof"] = max(derived["fp32"], derived["tf32x3"])
    out = {"device": props.name, "sms": sms, "rates_tflops": {k: v["tflops"] for k, v in res.items()},
           "derived_tflops": derived, "detail": res, "clocks": clk,
           "command": "python -m matrix_dense_linear_spd_gb300.peaks",
           "method": "best of %d launches after growing the loop to >= %g ms; CUDA events" % (a.reps, a.min_ms)}
    os.makedirs(os.path.dirname(a.out), exist_ok=True)
    with open(a.out, "w") as f:
        json.dump(out, f, indent=1)
    print(json.dumps({"derived_tflops": derived, "clocks": clk}))
    return 0


if __name__ == "__main__":
    sys.exit(main())
