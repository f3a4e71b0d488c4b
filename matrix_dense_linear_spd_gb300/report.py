"""Per-workload report: every named synthetic workload measured with the benchmark's protocol
(protocol.py: back-to-back calls on distinct pristine copies, inputs larger than four times L2,
CUDA events around each chunk; plus one isolated call after an L2 flush), with matrices/s, GB/s,
GFLOP/s and the achieved fraction of the binding roof, next to cuSOLVER's batched potrf
(cusolverDn<t>potrfBatched, in place, pointer arrays built untimed) as a reference point. The
vendor and library arms run interleaved chunk by chunk, in alternating order.

Roofs, all measured on the GPU the report runs on:
  HBM   the copy bandwidth in MEASURED_PEAKS.json;
  FP32  max(FFMA, packed FFMA2) from profiles/fp_peaks.json (python -m ...peaks);
  FP32-accurate tensor rate: the tcgen05 TF32 rate / 3 (the 3xTF32 split), for the routes whose
        contraction runs on the tensor cores; the f32 roof of such a route is max(FP32, TF32/3);
  FP64  max(DFMA, DMMA) from the same file.
The binding roof of a workload is the one whose time (bytes / bandwidth or flops / rate) is the
larger; roof fraction = that time / measured time.

Usage: python -m matrix_dense_linear_spd_gb300.report [--workloads f32_n8,...] [--steps 40]
       [--saturation]   adds f32 n=8 at 2^20 items and the f32 n=32 Lower batch-doubling curve
Prints markdown tables.
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
from matrix_dense_linear_spd_gb300 import protocol as P  # noqa: E402

ESIZE = {"f32": 4, "f64": 8, "c64": 8, "c128": 16}
TENSOR_ROUTES = (":tc=2",)        # routes whose contraction runs on tcgen05 with the 3xTF32 split


def tri_sector_bytes(n, dtype, uplo):
    s = ESIZE[dtype]
    t = 0
    for c in range(n):
        lo, hi = ((c * n + c) * s, (c * n + n) * s) if uplo == "L" else ((c * n) * s, (c * n + c + 1) * s)
        t += (math.ceil(hi / 32) - lo // 32) * 32
    return t


def flops(n, dtype, nrhs=0):
    """LAPACK counts: potrf, plus the two triangular solves per right-hand side."""
    c = synth.is_complex(dtype)
    f = (4 * n ** 3 / 3 + 3 * n ** 2 + 5 * n / 3) if c else (n ** 3 / 3 + n ** 2 / 2 + n / 6)
    return f + nrhs * ((8 * n * n - 2 * n) if c else (2 * n * n - n))


def roofs():
    """(HBM GB/s, FP32 TF/s, FP32-accurate tensor TF/s, FP64 TF/s, sources)."""
    hp = os.path.join(_ROOT, "MEASURED_PEAKS.json")
    fp = os.path.join(_ROOT, "profiles", "fp_peaks.json")
    hbm = json.load(open(hp))["hbm_gbs"] if os.path.exists(hp) else 6800.0
    src = ["HBM: " + ("MEASURED_PEAKS.json copy bandwidth" if os.path.exists(hp) else "fallback 6800 GB/s")]
    if not os.path.exists(fp):
        raise SystemExit("profiles/fp_peaks.json is missing: run python -m matrix_dense_linear_spd_gb300.peaks")
    d = json.load(open(fp))["derived_tflops"]
    src.append("FP: profiles/fp_peaks.json")
    return hbm, d["fp32"], d["tf32x3"], d["fp64"], src


def measure(w, op, uplo, nrhs, steps, torch, flush, l2, vendor, route=None):
    n, batch, dt = w.n, w.batch, w.dtype
    code = bl.DTYPE_CODES[dt]
    s = torch.cuda.current_stream()
    sp = s.cuda_stream
    pa = torch.from_numpy(synth.to_colmajor(w.A)).cuda()
    bufs = [pa]
    if nrhs:
        bufs.append(torch.from_numpy(synth.to_colmajor(w.B[:, :, :nrhs])).cuda())
    total_bytes = sum(b.numel() * b.element_size() for b in bufs)
    R = P.copies_per_chunk(total_bytes, l2, steps)
    rot = P.Rotation(bufs, R)
    infos = torch.zeros((R, batch), dtype=torch.int32, device="cuda")
    if route:
        bl.set_route(op, route)

    def call(i):
        if op == "potrf":
            bl.potrf_ptr(uplo, code, n, batch, rot.ptr(0, i), n, n * n, infos[i].data_ptr(), sp)
        else:
            bl.posv_ptr(uplo, code, n, nrhs, batch, rot.ptr(0, i), n, n * n, rot.ptr(1, i), n, n * nrhs,
                        infos[i].data_ptr(), sp)

    try:
        vcall = None
        if vendor is not None and op == "potrf":
            ptrs = [vendor.pointer_array(rot.ptr(0, i), batch, n * n, dt, pa.device) for i in range(R)]
            vcall = lambda i: vendor.potrf(uplo, dt, n, batch, ptrs[i], n, infos[i].data_ptr(), sp)
        ours, theirs = [], []
        P.time_back_to_back(call, rot, flush, R, s)                 # warm-up chunk
        if vcall:
            P.time_back_to_back(vcall, rot, flush, R, s)
        for rep in range(max(1, steps // R)):
            order = [(call, ours), (vcall, theirs)] if rep % 2 == 0 else [(vcall, theirs), (call, ours)]
            for fn, acc in order:
                if fn is None:
                    continue
                pc, _ = P.time_back_to_back(fn, rot, flush, R, s, warm_chunks=0)
                acc.extend(pc)
        # correctness of the library's last chunk: info as planted (or all zero)
        rot.restore()
        call(0)
        torch.cuda.synchronize()
        expect = w.planted_info if w.planted_info is not None else np.zeros(batch, np.int32)
        ok = np.array_equal(infos[0].cpu().numpy(), expect)
        chosen = bl.last_choice()
        iso = P.time_isolated(call, rot, flush, 15, s)
    finally:
        if route:
            bl.set_route(op, None)
    return {"ms": P.stats(ours)["median"], "rel_sd": P.stats(ours)["rel_sd"], "iso": P.stats(iso)["median"],
            "vms": P.stats(theirs)["median"] if theirs else None, "route": chosen, "info_ok": ok,
            "l2_resident": R * total_bytes < 4 * l2}


def row(name, w, op, uplo, nrhs, m, hbm, fp32, tf32x3, fp64):
    n, batch, dt = w.n, w.batch, w.dtype
    byts = (2 * tri_sector_bytes(n, dt, uplo) + 4) * batch
    if nrhs:
        byts += 2 * n * nrhs * ESIZE[dt] * batch
    fl = flops(n, dt, nrhs) * batch
    if dt in ("f64", "c128"):
        fp, fpname = fp64, "FP64"
    elif any(t in m["route"] for t in TENSOR_ROUTES):
        fp, fpname = max(fp32, tf32x3), ("FP32" if fp32 >= tf32x3 else "3xTF32")
    else:
        fp, fpname = fp32, "FP32"
    t_hbm, t_fp = byts / (hbm * 1e9), fl / (fp * 1e12)
    bind = "HBM" if t_hbm >= t_fp else fpname
    ms = m["ms"]
    frac = max(t_hbm, t_fp) / (ms / 1e3)
    vend = f"{m['vms']:.4f}" if m["vms"] else "-"
    ratio = f"{m['vms'] / ms:.1f}" if m["vms"] else "-"
    flag = "" if m["info_ok"] else " (info MISMATCH)"
    noisy = " (noisy)" if m["rel_sd"] > 0.10 else ""
    if m.get("l2_resident"):
        noisy += " (a chunk's copies fit in L2)"
    return (f"| {name} b{batch} | {op}{'' if not nrhs else f' nrhs={nrhs}'} | {uplo} | `{m['route']}` | "
            f"{ms:.4f}{flag}{noisy} | {m['iso']:.4f} | {batch / (ms / 1e3):.3g} | {byts / (ms / 1e3) / 1e9:.0f} | "
            f"{fl / (ms / 1e3) / 1e9:.0f} | {bind} | {frac:.2f} | {vend} | {ratio} |")


HEADER = ("| workload | op | uplo | route | ms/call (back to back) | ms (isolated call) | matrices/s | "
          "GB/s (triangle) | GFLOP/s | binding roof | roof frac | cuSOLVER ms | x vs cuSOLVER |\n"
          "|---|---|---|---|---|---|---|---|---|---|---|---|---|")


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--workloads", default=",".join(synth.WORKLOADS))
    ap.add_argument("--steps", type=int, default=40)
    ap.add_argument("--no-vendor", action="store_true")
    ap.add_argument("--saturation", action="store_true")
    ap.add_argument("--route", default=None, help="pin one route for every row (default: table choice)")
    a = ap.parse_args(argv)
    import torch
    dev = torch.cuda.get_device_properties(0)
    l2 = dev.L2_cache_size
    flush = P.L2Flush(l2, "cuda")
    hbm, fp32, tf32x3, fp64, src = roofs()
    vendor = None
    if not a.no_vendor:
        from matrix_dense_linear_spd_gb300.vendor import CusolverPotrfBatched
        vendor = CusolverPotrfBatched()
    print(HEADER)
    for name in [x for x in a.workloads.split(",") if x]:
        w = synth.workload(name)
        ops = [("potrf", u, 0) for u in w.uplos]
        if w.nrhs:
            ops.append(("posv", "L", w.nrhs))
        for op, uplo, nrhs in ops:
            m = measure(w, op, uplo, nrhs, a.steps, torch, flush, l2, vendor, a.route)
            print(row(name, w, op, uplo, nrhs, m, hbm, fp32, tf32x3, fp64), flush=True)
        del w
        torch.cuda.empty_cache()
    if a.saturation:
        print("\nSaturation (potrf Lower, same protocol):\n")
        print(HEADER)
        cases = [("f32_n8", 1 << 20)] + [("f32_n32", 1 << k) for k in range(10, 18)]
        for name, b in cases:
            w = synth.workload(name, batch=b)
            m = measure(w, "potrf", "L", 0, a.steps, torch, flush, l2, vendor)
            print(row(name, w, "potrf", "L", 0, m, hbm, fp32, tf32x3, fp64), flush=True)
            del w
            torch.cuda.empty_cache()
    print(f"\nRoofs: HBM {hbm:.0f} GB/s, FP32 {fp32:.1f} TFLOP/s, 3xTF32 {tf32x3:.1f} TFLOP/s (TF32 tensor / 3), "
          f"FP64 {fp64:.2f} TFLOP/s; sources: {'; '.join(src)}.")
    if vendor:
        vendor.close()
    return 0


if __name__ == "__main__":
    sys.exit(main())
