"""Benchmark: batched potrf throughput on the f32 n=32 batch=16384 workload (Lower).

One step = one bl_potrf call over the whole batch (pivot, scale, trailing update, load and
store of every item), inputs resident in HBM. The operation is in place, so every step factors
its own pristine copy of the batch: steps run back to back in chunks (CUDA events around each
chunk on the launching stream), the copies of a chunk together exceed four times the L2 size,
and they are restored and L2 flushed before each chunk, untimed (protocol.py).

Printed JSON line (one per run, rank 0):
  value        matrices/s over all ranks (weak scaling: every rank factors its own batch)
  e2e          the same metric through the public C ABI with the batch in pinned host memory:
               host->device copy, bl_potrf, device->host copy of the factor and info, per step
               (two streams alternate, so copies overlap the other step's kernel)
  roofline     achieved algorithmic GB/s of the potrf kernel against the measured HBM copy
               bandwidth (MEASURED_PEAKS.json); algorithmic bytes = the referenced triangle read
               and written at 32-byte sector granularity plus the 4-byte info per item
  cpu_baseline the CPU oracle (long double) on the host cores, on a bounded sample
  also         Upper potrf, posv (nrhs = 4), one isolated call, and cuSOLVER potrfBatched on the
               same batch and protocol (vendor reference point)

--impl reference times the CPU oracle alone on the same workload (the reference arm).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np

import synth

METRIC = "batched potrf matrices/s & GB/s (f32 n=32 b16384); % of HBM/FP roofline"
UNIT = "matrices/s"
ESIZE = {"f32": 4, "f64": 8, "c64": 8, "c128": 16}


# ------------------------------------------------------------------ byte / flop accounting

def triangle_sector_bytes(n: int, dtype: str, uplo: str = "L") -> int:
    """Bytes of the referenced triangle of one contiguous (lda = n) item at 32-byte sector
    granularity, counted once (read) -- the item base is assumed sector aligned."""
    s = ESIZE[dtype]
    total = 0
    for c in range(n):
        if uplo == "L":
            lo, hi = (c * n + c) * s, (c * n + n) * s      # rows c..n-1 of column c
        else:
            lo, hi = (c * n) * s, (c * n + c + 1) * s      # rows 0..c of column c
        total += (math.ceil(hi / 32) - lo // 32) * 32
    return total


def potrf_bytes(n: int, dtype: str, uplo: str = "L") -> int:
    return 2 * triangle_sector_bytes(n, dtype, uplo) + 4


def potrf_flops(n: int, dtype: str) -> float:
    if synth.is_complex(dtype):
        return 4 * n ** 3 / 3 + 3 * n ** 2 + 5 * n / 3
    return n ** 3 / 3 + n ** 2 / 2 + n / 6


# ------------------------------------------------------------------ helpers

def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


def kernel_source_sha(files):
    """Short hash of the kernel source files a measured kernel is built from."""
    h = hashlib.sha1()
    csrc = os.path.join(ROOT, "matrix_dense_linear_spd_gb300", "csrc")
    for f in files:
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel_tag: str):
    """DRAM bytes per launch (read + write) from the committed ncu record, if it was taken on
    the current sources of that kernel; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    e = d.get(kernel_tag)
    if not e or e.get("source_sha") != kernel_source_sha(e.get("source_files", [])):
        return None
    return e.get("dram_bytes_per_launch")


def aggregate(ms_local: float, batch: int, dist=None, device=None):
    """Weak-scaling aggregate over ranks: every rank factors its own batch, the job time is the
    slowest rank's, and the value counts the matrices of all ranks. Returns (ms_max, value)."""
    import torch
    ms_max = ms_local
    ws = 1
    if dist is not None and dist.is_initialized():
        ws = dist.get_world_size()
        t = torch.tensor([ms_local], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms_max = float(t.item())
    return ms_max, ws * batch / (ms_max / 1e3)


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def host_cpu_model() -> str:
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu model")):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.processor() or platform.machine()


def cpu_oracle_rate(w, uplo: str, target_s: float = 10.0, max_items: int | None = None, reps: int = 3):
    """Oracle matrices/s on the host cores over a bounded sample of the workload: the leading
    items, grown until one run takes about target_s / reps (at most the whole batch); then the
    sample is run repeatedly, at least `reps` times and until about target_s of CPU work is done,
    and the median run is reported. Returns (rate, items per run, median s, cores, long-double
    mantissa bits, runs)."""
    import oracle
    cores = os.cpu_count() or 1
    n = w.n
    cap = w.batch if max_items is None else min(max_items, w.batch)
    k = min(max(cores, 64), cap)
    per_run = target_s / max(reps, 1)
    while True:
        buf = synth.to_colmajor(w.A[:k])
        t0 = time.perf_counter()
        oracle.run(uplo, n, k, buf, n, n * n, threads=cores)
        t = time.perf_counter() - t0
        if t >= per_run or k >= cap:
            break
        k = min(cap, max(k * 2, int(k * per_run / max(t, 1e-3))))
    ts, total = [], 0.0
    while len(ts) < reps or total < target_s:
        t0 = time.perf_counter()
        oracle.run(uplo, n, k, buf, n, n * n, threads=cores)
        ts.append(time.perf_counter() - t0)
        total += ts[-1]
        if len(ts) >= 1000:
            break
    t = statistics.median(ts)
    return k / t, k, t, cores, oracle.long_double_digits(), len(ts)


# ------------------------------------------------------------------ the GPU arm

def run_ours(args, ws, rank, local):
    import torch
    import matrix_dense_linear_spd_gb300 as bl
    from matrix_dense_linear_spd_gb300 import protocol as P
    from matrix_dense_linear_spd_gb300.clocks import ClockSampler

    torch.cuda.set_device(local)
    dist = None
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream()
    sptr = stream.cuda_stream

    w = synth.workload(args.workload)
    n, batch, dtype = w.n, w.batch, w.dtype
    code = bl.DTYPE_CODES[dtype]
    esz = ESIZE[dtype]
    buf = synth.to_colmajor(w.A)
    pristine = torch.from_numpy(buf).to(dev)
    item_bytes = pristine.numel() * pristine.element_size()
    l2 = torch.cuda.get_device_properties(local).L2_cache_size
    flush = P.L2Flush(l2, dev)
    R = P.copies_per_chunk(item_bytes, l2, args.steps)
    rot = P.Rotation([pristine], R)
    infos = torch.zeros((R, batch), dtype=torch.int32, device=dev)

    def potrf_call(uplo):
        return lambda i: bl.potrf_ptr(uplo, code, n, batch, rot.ptr(0, i), n, n * n, infos[i].data_ptr(), sptr)

    call_l = potrf_call("L")
    # untimed: the first call selects and configures; then a clock-warming phase
    rot.restore()
    call_l(0)
    torch.cuda.synchronize()
    route = bl.last_choice()
    sampler = ClockSampler(local).start()
    t_end = time.perf_counter() + args.warm_seconds
    while time.perf_counter() < t_end:
        rot.restore()
        for i in range(R):
            call_l(i)
        torch.cuda.synchronize()

    # ---- the timed region: exactly `steps` calls, back to back on distinct pristine copies
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    per_call, total_ms = P.time_back_to_back(call_l, rot, flush, args.steps, stream,
                                             warm_chunks=max(1, math.ceil(args.warmup / R)))
    t1 = time.perf_counter()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    sampler.stop()
    ms_step = total_ms / args.steps
    ms_max, value = aggregate(ms_step, batch, dist, dev)
    ok_info = int(infos.abs().sum().item()) == 0
    st_main = P.stats(per_call)

    also = {}
    if not args.no_extras:
        # one call on its own (restore, L2 flush, events around the single call)
        iso = P.time_isolated(call_l, rot, flush, 30, stream)
        also["potrf_lower_isolated_call"] = {"ms_per_call": P.stats(iso)["median"], "rel_sd": P.stats(iso)["rel_sd"],
                                             "protocol": "restore + L2 flush, then events around one call; median of 30"}
        # Upper on the same batch
        call_u = potrf_call("U")
        pu, tu = P.time_back_to_back(call_u, rot, flush, args.steps, stream)
        route_u = bl.last_choice()
        msu = tu / args.steps
        bu = potrf_bytes(n, dtype, "U")
        also["potrf_upper"] = {"matrices_per_s": batch / (msu / 1e3), "ms_per_call": msu, "route": route_u,
                               "gbs": bu * batch / (msu / 1e3) / 1e9, "rel_sd": P.stats(pu)["rel_sd"]}
        # posv with nrhs right-hand sides (A and B restored together)
        nrhs = w.nrhs or 4
        Bh = w.B if w.B is not None else synth.rhs_uniform(np.random.default_rng(9), n, nrhs, batch, dtype)
        Bp = torch.from_numpy(synth.to_colmajor(Bh)).to(dev)
        rot2 = P.Rotation([pristine, Bp], R)
        posv = lambda i: bl.posv_ptr("L", code, n, nrhs, batch, rot2.ptr(0, i), n, n * n, rot2.ptr(1, i), n,
                                     n * nrhs, infos[i].data_ptr(), sptr)
        pp, tp = P.time_back_to_back(posv, rot2, flush, args.steps, stream)
        route_p = bl.last_choice()
        msp = tp / args.steps
        also["posv_nrhs%d" % nrhs] = {"matrices_per_s": batch / (msp / 1e3), "ms_per_call": msp, "route": route_p,
                                      "rel_sd": P.stats(pp)["rel_sd"]}
        del rot2
        # vendor reference point: cuSOLVER potrfBatched, in place, pointer arrays built untimed,
        # same protocol; then ours again (second pass, reversed order) to expose drift
        try:
            from matrix_dense_linear_spd_gb300.vendor import CusolverPotrfBatched
            cus = CusolverPotrfBatched()
            ptrs = [cus.pointer_array(rot.ptr(0, i), batch, n * n, dtype, dev) for i in range(R)]
            vend = {}
            for up in ("L", "U"):
                vcall = lambda i, up=up: cus.potrf(up, dtype, n, batch, ptrs[i], n, infos[i].data_ptr(), sptr)
                pv, tv = P.time_back_to_back(vcall, rot, flush, args.steps, stream)
                msv = tv / args.steps
                vend["lower" if up == "L" else "upper"] = {"matrices_per_s": batch / (msv / 1e3), "ms_per_call": msv,
                                                          "rel_sd": P.stats(pv)["rel_sd"],
                                                          "info_all_zero": int(infos.abs().sum().item()) == 0}
            cus.close()
            also["cusolver_potrfBatched"] = vend
        except Exception as e:  # the reference point is context; its absence is reported
            also["cusolver_potrfBatched"] = {"unavailable": str(e)[:200]}
        p2, t2 = P.time_back_to_back(call_l, rot, flush, args.steps, stream)
        also["potrf_lower_second_pass"] = {"ms_per_call": t2 / args.steps, "rel_sd": P.stats(p2)["rel_sd"],
                                           "vs_first_pass": (t2 / args.steps) / ms_step}
    del rot

    # ---- e2e through the C ABI with pinned host buffers: every step copies its batch in, factors
    # it and copies the factor and info out; two streams alternate so one step's copies overlap
    # the other's work, as a caller streaming batches would run it
    host_in = torch.from_numpy(buf).pin_memory()
    host_out = [torch.empty_like(host_in).pin_memory() for _ in range(2)]
    host_info = [torch.empty(batch, dtype=torch.int32).pin_memory() for _ in range(2)]
    dbuf = [torch.empty_like(pristine) for _ in range(2)]
    dinfo = [torch.empty(batch, dtype=torch.int32, device=dev) for _ in range(2)]
    streams = [torch.cuda.Stream(dev) for _ in range(2)]

    def e2e_step(k):
        s_ = streams[k & 1]
        with torch.cuda.stream(s_):
            dbuf[k & 1].copy_(host_in, non_blocking=True)
            bl.potrf_ptr("L", code, n, batch, dbuf[k & 1].data_ptr(), n, n * n, dinfo[k & 1].data_ptr(), s_.cuda_stream)
            host_out[k & 1].copy_(dbuf[k & 1], non_blocking=True)
            host_info[k & 1].copy_(dinfo[k & 1], non_blocking=True)

    for k in range(args.warmup):
        e2e_step(k)
    torch.cuda.synchronize()
    flush()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for s_ in streams:
        s_.wait_event(e0)
    for k in range(args.steps):
        e2e_step(k)
    for s_ in streams:
        ev = torch.cuda.Event()
        ev.record(s_)
        stream.wait_event(ev)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / args.steps
    e2e_info_ok = all(int(h.abs().sum().item()) == 0 for h in host_info)
    e2e_step_max, _ = aggregate(e2e_ms, batch, dist, dev)

    peaks, peak_src = measured_peaks()
    alg_bytes = potrf_bytes(n, dtype, "L") * batch
    achieved = alg_bytes / (ms_step / 1e3) / 1e9
    kernel_tag = f"potrf_{dtype}_n{n}_{route}"
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_max, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": dtype, "data": "synthetic (seeded SPD batch, A = B*B^T + n*I)",
        "config": {"workload": f"potrf {dtype} Lower n={n} batch={batch} (seed 1)",
                   "lda": n, "stride": n * n, "route": route,
                   "l2": (f"inputs larger than L2: each step factors its own pristine copy of the batch; chunks of "
                          f"{R} back-to-back steps ({R * item_bytes >> 20} MiB of inputs, L2 {l2 >> 20} MiB), "
                          f"copies restored and L2 flushed ({flush.mib} MiB write + read) before each chunk, untimed"),
                   "parallelism": f"weak: {ws} independent batches"},
        "timing": {"per_step_ms_median": st_main["median"], "rel_sd": st_main["rel_sd"], "chunks": st_main["n"],
                   "steps_per_chunk": R, "noisy": st_main["rel_sd"] > 0.10},
        "gbs": alg_bytes * ws / (ms_max / 1e3) / 1e9,
        "gbs_full_storage": (2 * n * n * esz + 4) * batch * ws / (ms_max / 1e3) / 1e9,
        "gflops": potrf_flops(n, dtype) * batch * ws / (ms_max / 1e3) / 1e9,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": achieved / peaks["hbm_gbs"], "traffic": recorded_traffic(kernel_tag),
                     "algorithmic_bytes_per_launch": alg_bytes, "kernel": kernel_tag,
                     "peak_source": f"{peak_src} (copy bandwidth, burst: of measured)"},
        "e2e": {"value": ws * batch / (e2e_step_max / 1e3), "unit": UNIT,
                "h2d_bytes_per_step": host_in.numel() * host_in.element_size(),
                "d2h_bytes_per_step": host_out[0].numel() * host_out[0].element_size() + batch * 4,
                "info_all_zero": e2e_info_ok,
                "protocol": "pinned host buffers; per step: H2D of the batch, bl_potrf, D2H of factor and info; "
                            "two streams alternate (copies of one step overlap the other's kernel); events around "
                            "all steps"},
        "gpu_launches": args.steps,
        "clocks": sampler.summary(t0 - args.warm_seconds, t1),
        "info_all_zero": ok_info,
        "also": also,
    }
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        rate, k, t, cores, ldig, runs = cpu_oracle_rate(w, "L", target_s=args.cpu_seconds)
        line["cpu_baseline"] = {"value": rate, "unit": UNIT, "cores": cores, "kind": "oracle",
                                "sample": (f"{'the whole batch' if k == w.batch else f'the first {k} items'} "
                                           f"({k} matrices) per run, {runs} runs (~{runs * t:.0f} s of CPU "
                                           f"work), median run {t:.3f} s"),
                                "cpu": host_cpu_model(),
                                "long_double": {64: "x87 80-bit extended", 113: "IEEE binary128 (software)"}.get(
                                    ldig, f"{ldig}-bit mantissa")}
    if dist:
        dist.destroy_process_group()
    return line if rank == 0 else None


def run_reference(args):
    """The reference arm: the CPU oracle on the host cores, each step a bounded sample."""
    import oracle
    w = synth.workload(args.workload)
    cores = os.cpu_count() or 1
    rate0, k, t, _, ldig, _ = cpu_oracle_rate(w, "L", target_s=min(args.cpu_seconds, 3.0), max_items=2048, reps=1)
    per_step = max(1, min(w.batch, int(rate0 * args.reference_step_seconds)))
    buf = synth.to_colmajor(w.A[:per_step])
    for _ in range(args.warmup):
        oracle.run("L", w.n, per_step, buf, w.n, w.n * w.n, threads=cores)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle.run("L", w.n, per_step, buf, w.n, w.n * w.n, threads=cores)
        times.append(time.perf_counter() - t0)
    ms = 1e3 * sum(times) / len(times)
    value = per_step / (ms / 1e3)
    fmt = {64: "x87 80-bit extended", 113: "IEEE binary128 (software)"}.get(ldig, f"{ldig}-bit mantissa")
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
        "config": {"workload": f"potrf {w.dtype} Lower n={w.n} batch={w.batch} (seed 1)",
                   "sample_per_step": per_step},
        "timing": {"per_step_ms_median": 1e3 * statistics.median(times)},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"{per_step} items per step (leading items of the workload)",
                         "cpu": host_cpu_model(), "long_double": fmt},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="f32_n32", choices=list(synth.WORKLOADS))
    ap.add_argument("--warm-seconds", type=float, default=1.0)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--reference-step-seconds", type=float, default=0.5)
    ap.add_argument("--no-extras", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    ws, rank, local = dist_env()
    if args.impl == "reference":
        if rank != 0:
            return 0
        print(json.dumps(run_reference(args)), flush=True)
        return 0
    line = run_ours(args, ws, rank, local)
    if line is not None:
        print(json.dumps(line), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
