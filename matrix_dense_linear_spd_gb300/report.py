"""Per-workload report: every named synthetic workload measured with the benchmark protocol
(input restored and L2 flushed before each call, CUDA events around the call, trimmed mean
of the middle 60% of the repetitions), with
matrices/s, GB/s, GFLOP/s and the achieved fraction of the binding roof, next to cuSOLVER's
batched potrf (through torch.linalg.cholesky_ex) as a reference point.

Roofs: HBM copy bandwidth from MEASURED_PEAKS.json; FP32 and FP64 from unit counts at the
maximum SM clock (152 SMs x 128 FP32 lanes x 2 flops, and x 2 FP64 lanes x 2 flops, per clock).
The binding roof of a workload is the larger of bytes/HBM and flops/FP peak.

Usage: python -m matrix_dense_linear_spd_gb300.report [--workloads f32_n8,...] [--reps 20]
Prints one markdown table.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import sys

import numpy as np

_ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if _ROOT not in sys.path:
    sys.path.insert(0, _ROOT)

import synth  # noqa: E402

import matrix_dense_linear_spd_gb300 as bl  # noqa: E402

ESIZE = {"f32": 4, "f64": 8, "c64": 8, "c128": 16}
SMS, FP32_LANES, FP64_LANES = 152, 128, 2


def tri_sector_bytes(n, dtype, uplo):
    s = ESIZE[dtype]
    t = 0
    for c in range(n):
        lo, hi = ((c * n + c) * s, (c * n + n) * s) if uplo == "L" else ((c * n) * s, (c * n + c + 1) * s)
        t += (math.ceil(hi / 32) - lo // 32) * 32
    return t


def flops(n, dtype, nrhs=0):
    c = synth.is_complex(dtype)
    f = (4 * n ** 3 / 3 + 3 * n ** 2 + 5 * n / 3) if c else (n ** 3 / 3 + n ** 2 / 2 + n / 6)
    return f + nrhs * ((8 * n * n - 2 * n) if c else (2 * n * n - n)) * 2 / 2


def peaks(sm_mhz):
    path = os.path.join(_ROOT, "MEASURED_PEAKS.json")
    hbm = json.load(open(path))["hbm_gbs"] if os.path.exists(path) else 6800.0
    f32 = SMS * FP32_LANES * 2 * sm_mhz * 1e6 / 1e12
    f64 = SMS * FP64_LANES * 2 * sm_mhz * 1e6 / 1e12
    return hbm, f32, f64


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--workloads", default=",".join(synth.WORKLOADS))
    ap.add_argument("--reps", type=int, default=20)
    ap.add_argument("--no-vendor", action="store_true")
    a = ap.parse_args(argv)
    import torch
    dev = torch.cuda.get_device_properties(0)
    l2 = dev.L2_cache_size
    fa = torch.empty(max(2 * l2, 256 << 20) // 4, device="cuda")
    fb = torch.ones_like(fa)
    sink = torch.empty((), device="cuda")
    s = torch.cuda.current_stream()
    hbm, f32p, f64p = peaks(2070.0)
    print(f"| workload | op | uplo | route | ms/call | matrices/s | GB/s (triangle) | GFLOP/s | binding roof | "
          f"roof frac | cuSOLVER ms | x vs cuSOLVER |")
    print("|---|---|---|---|---|---|---|---|---|---|---|---|")
    for name in a.workloads.split(","):
        w = synth.workload(name)
        n, batch, dt = w.n, w.batch, w.dtype
        code = bl.DTYPE_CODES[dt]
        pr = torch.from_numpy(synth.to_colmajor(w.A)).cuda()
        wk = pr.clone()
        info = torch.empty(batch, dtype=torch.int32, device="cuda")
        ops = [("potrf", u, 0) for u in w.uplos]
        if w.nrhs:
            ops.append(("posv", "L", w.nrhs))
        for op, uplo, nrhs in ops:
            if nrhs:
                Bp = torch.from_numpy(synth.to_colmajor(w.B)).cuda()
                Bw = Bp.clone()

            def call():
                if op == "potrf":
                    bl.potrf_ptr(uplo, code, n, batch, wk.data_ptr(), n, n * n, info.data_ptr(), s.cuda_stream)
                else:
                    bl.posv_ptr(uplo, code, n, nrhs, batch, wk.data_ptr(), n, n * n, Bw.data_ptr(), n, n * nrhs,
                                info.data_ptr(), s.cuda_stream)

            ts = []
            for it in range(a.reps + 3):
                wk.copy_(pr)
                if nrhs:
                    Bw.copy_(Bp)
                fa.zero_()
                torch.sum(fb, dim=0, out=sink)
                e0, e1 = torch.cuda.Event(True), torch.cuda.Event(True)
                e0.record(s)
                call()
                e1.record(s)
                torch.cuda.synchronize()
                if it >= 3:
                    ts.append(e0.elapsed_time(e1))
            ts.sort()
            k = len(ts) // 5
            ms = statistics.mean(ts[k:len(ts) - k] or ts)
            route = bl.last_choice()
            expect = w.planted_info if w.planted_info is not None else np.zeros(batch, np.int32)
            ok = np.array_equal(info.cpu().numpy(), expect)
            byts = (2 * tri_sector_bytes(n, dt, uplo) + 4) * batch
            if nrhs:
                byts += 2 * n * nrhs * ESIZE[dt] * batch
            fl = flops(n, dt, nrhs) * batch
            fp = f64p if dt in ("f64", "c128") else f32p
            t_hbm = byts / (hbm * 1e9)
            t_fp = fl / (fp * 1e12)
            bind = "HBM" if t_hbm >= t_fp else ("FP64" if fp == f64p else "FP32")
            frac = max(t_hbm, t_fp) / (ms / 1e3)
            vend = "-"
            ratio = "-"
            if op == "potrf" and not a.no_vendor:
                Av = wk.view(batch, n, n)
                vt = []
                for it in range(min(a.reps, 8) + 2):
                    wk.copy_(pr)
                    fa.zero_()
                    torch.sum(fb, dim=0, out=sink)
                    e0, e1 = torch.cuda.Event(True), torch.cuda.Event(True)
                    e0.record(s)
                    torch.linalg.cholesky_ex(Av, upper=(uplo == "U"), check_errors=False)
                    e1.record(s)
                    torch.cuda.synchronize()
                    if it >= 2:
                        vt.append(e0.elapsed_time(e1))
                vt.sort()
                k = len(vt) // 5
                vms = statistics.mean(vt[k:len(vt) - k] or vt)
                vend = f"{vms:.4f}"
                ratio = f"{vms / ms:.1f}"
            flag = "" if ok else " (info MISMATCH)"
            print(f"| {name} b{batch} | {op}{'' if not nrhs else f' nrhs={nrhs}'} | {uplo} | `{route}` | {ms:.4f}{flag} | "
                  f"{batch / (ms / 1e3):.3g} | {byts / (ms / 1e3) / 1e9:.0f} | {fl / (ms / 1e3) / 1e9:.0f} | {bind} | "
                  f"{frac:.2f} | {vend} | {ratio} |", flush=True)
        del pr, wk
        torch.cuda.empty_cache()
    print(f"\nRoofs: HBM {hbm:.0f} GB/s (measured copy), FP32 {f32p:.1f} TFLOP/s and FP64 {f64p:.2f} TFLOP/s "
          f"(unit counts at 2070 MHz).")
    return 0


if __name__ == "__main__":
    sys.exit(main())
