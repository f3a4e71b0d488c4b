"""Benchmark: batched potrf throughput on the f32 n=32 batch=16384 workload (Lower).

One step = one bl_potrf call over the whole batch (pivot, scale, trailing update, load and
store of every item), inputs resident in HBM. The operation is in place, so before every
timed step the input is restored from a pristine device copy and L2 is flushed (both
untimed); the step itself is timed with CUDA events on the launching stream.

Printed JSON line (one per run, rank 0):
  value        matrices/s over all ranks (weak scaling: every rank factors its own batch)
  e2e          the same metric through the public C ABI with the batch in pinned host memory:
               host->device copy, bl_potrf, device->host copy of the factor and info, per step
  roofline     achieved algorithmic GB/s of the potrf kernel against the measured HBM copy
               bandwidth (MEASURED_PEAKS.json); algorithmic bytes = the referenced triangle read
               and written at 32-byte sector granularity plus the 4-byte info per item
  cpu_baseline the CPU oracle (long double) on the host cores, on a bounded sample
  also         Upper potrf and posv (nrhs = 4) on the same batch, same protocol

--impl reference times the CPU oracle alone on the same workload (the reference arm).
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
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


# ------------------------------------------------------------------ clocks (NVML via ctypes)

class ClockSampler:
    """Samples SM clock and clock-event reasons every few ms in a background thread."""
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, torch_device: int = 0, period: float = 0.005):
        self.period = period
        self.samples = []
        self.max_mhz = None
        self.ok = False
        self._stop = threading.Event()
        try:
            import torch
            self.nvml = ctypes.CDLL("libnvidia-ml.so.1")
            if self.nvml.nvmlInit_v2() != 0:
                raise OSError("nvmlInit failed")
            self.handle = ctypes.c_void_p()
            uuid = None
            try:
                uuid = str(torch.cuda.get_device_properties(torch_device).uuid)
            except Exception:
                pass
            rc = 1
            if uuid:
                for cand in (uuid, "GPU-" + uuid):
                    rc = self.nvml.nvmlDeviceGetHandleByUUID(cand.encode(), ctypes.byref(self.handle))
                    if rc == 0:
                        break
            if rc != 0:
                rc = self.nvml.nvmlDeviceGetHandleByIndex_v2(0, ctypes.byref(self.handle))
            if rc != 0:
                raise OSError("no NVML handle")
            m = ctypes.c_uint()
            if self.nvml.nvmlDeviceGetMaxClockInfo(self.handle, 1, ctypes.byref(m)) == 0:
                self.max_mhz = m.value
            self.ok = True
        except Exception:
            self.ok = False

    def _one(self):
        c = ctypes.c_uint()
        r = ctypes.c_ulonglong()
        if self.nvml.nvmlDeviceGetClockInfo(self.handle, 1, ctypes.byref(c)) != 0:
            return
        self.nvml.nvmlDeviceGetCurrentClocksEventReasons(self.handle, ctypes.byref(r))
        self.samples.append((time.perf_counter(), c.value, r.value))

    def _run(self):
        while not self._stop.is_set():
            self._one()
            time.sleep(self.period)

    def start(self):
        if self.ok:
            self._t = threading.Thread(target=self._run, daemon=True)
            self._t.start()
        return self

    def stop(self):
        if self.ok:
            self._stop.set()
            self._t.join()

    def summary(self, t0=None, t1=None):
        if not self.ok or not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": [], "samples": 0,
                    "source": "nvml unavailable"}
        sel = [s for s in self.samples if (t0 is None or s[0] >= t0) and (t1 is None or s[0] <= t1)]
        if len(sel) < 3:
            sel = self.samples
        reasons = set()
        for _, _, r in sel:
            for bit, name in self.REASONS.items():
                if r & bit:
                    reasons.add(name)
        return {"sm_mhz": statistics.median(s[1] for s in sel), "sm_max_mhz": self.max_mhz,
                "reasons": sorted(reasons), "samples": len(sel), "source": "nvml"}


# ------------------------------------------------------------------ helpers

class L2Flush:
    """Evict L2 between timed steps: write one buffer larger than L2, then read a second one,
    so the lines left in L2 are clean and no write-back of the flush lands in the timed
    kernel."""

    def __init__(self, l2_bytes: int, device):
        import torch
        n = max(2 * l2_bytes, 256 << 20) // 4
        self.a = torch.empty(n, dtype=torch.float32, device=device)
        self.b = torch.ones(n, dtype=torch.float32, device=device)
        self.sink = torch.empty((), dtype=torch.float32, device=device)
        self.mib = n * 4 >> 20

    def zero_(self):
        self.a.zero_()
        import torch
        torch.sum(self.b, dim=0, out=self.sink)


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


def cpu_oracle_rate(w, uplo: str, target_s: float = 8.0, max_items: int = 4096):
    """Oracle matrices/s on the host cores over a bounded leading sample of the workload."""
    import oracle
    cores = os.cpu_count() or 1
    n = w.n
    k = min(max(cores, 64), w.batch)
    t = 0.0
    while True:
        buf = synth.to_colmajor(w.A[:k])
        t0 = time.perf_counter()
        oracle.run(uplo, n, k, buf, n, n * n, threads=cores)
        t = time.perf_counter() - t0
        if t >= target_s or k >= min(max_items, w.batch):
            break
        k = min(min(max_items, w.batch), max(k * 2, int(k * target_s / max(t, 1e-3))))
    return k / t, k, t, cores


# ------------------------------------------------------------------ the GPU arm

def run_ours(args, ws, rank, local):
    import torch
    import matrix_dense_linear_spd_gb300 as bl

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
    buf = synth.to_colmajor(w.A)
    pristine = torch.from_numpy(buf).to(dev)
    work = pristine.clone()
    info = torch.empty(batch, dtype=torch.int32, device=dev)
    l2 = torch.cuda.get_device_properties(local).L2_cache_size
    flusher = L2Flush(l2, dev)
    flush = flusher

    def potrf_once(uplo):
        bl.potrf_ptr(uplo, code, n, batch, work.data_ptr(), n, n * n, info.data_ptr(), sptr)

    nrhs = w.nrhs or 4
    Bp = torch.from_numpy(synth.to_colmajor(w.B if w.B is not None else
                                            synth.rhs_uniform(np.random.default_rng(9), n, nrhs, batch, dtype))).to(dev)
    Bw = Bp.clone()

    def posv_once(uplo):
        bl.posv_ptr(uplo, code, n, nrhs, batch, work.data_ptr(), n, n * n, Bw.data_ptr(), n, n * nrhs,
                    info.data_ptr(), sptr)

    def timed(fn, uplo, steps, warmup, restore_b=False):
        for _ in range(warmup):
            work.copy_(pristine)
            if restore_b:
                Bw.copy_(Bp)
            flush.zero_()
            fn(uplo)
        torch.cuda.synchronize()
        evs = []
        for _ in range(steps):
            work.copy_(pristine)
            if restore_b:
                Bw.copy_(Bp)
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn(uplo)
            e1.record(stream)
            evs.append((e0, e1))
        torch.cuda.synchronize()
        return [a.elapsed_time(b) for a, b in evs]

    # untimed: first call selects and configures, then a clock-warming phase
    potrf_once("L")
    torch.cuda.synchronize()
    route = bl.last_choice()
    sampler = ClockSampler(local).start()
    t_end = time.perf_counter() + args.warm_seconds
    while time.perf_counter() < t_end:
        for _ in range(20):
            work.copy_(pristine)
            potrf_once("L")
        torch.cuda.synchronize()

    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    ms = timed(potrf_once, "L", args.steps, args.warmup)
    t1 = time.perf_counter()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    sampler.stop()
    ms_step = sum(ms) / len(ms)
    ms_max, value = aggregate(ms_step, batch, dist, dev)
    ok_info = int(info.abs().sum().item()) == 0

    # extras on the same batch: Upper potrf and posv
    also = {}
    if not args.no_extras:
        msu = timed(potrf_once, "U", args.steps, 2)
        route_u = bl.last_choice()
        msp = timed(posv_once, "L", args.steps, 2, restore_b=True)
        route_p = bl.last_choice()
        bu = potrf_bytes(n, dtype, "U")
        # vendor reference point: cuSOLVER batched potrf through torch.linalg.cholesky_ex
        # (out of place: its time includes torch's copy of the input into the output)
        Acm = work.view(batch, n, n)
        vend = {}
        for up in (False, True):
            for _ in range(3):
                torch.linalg.cholesky_ex(Acm, upper=up, check_errors=False)
            vt = []
            for _ in range(max(10, args.steps // 4)):
                work.copy_(pristine)
                flush.zero_()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                torch.linalg.cholesky_ex(Acm, upper=up, check_errors=False)
                e1.record(stream)
                vt.append((e0, e1))
            torch.cuda.synchronize()
            ms_v = statistics.median(a.elapsed_time(b) for a, b in vt)
            vend["upper" if up else "lower"] = {"matrices_per_s": batch / (ms_v / 1e3), "ms_per_call": ms_v}
        also = {
            "cusolver_potrf_via_torch": vend,
            "potrf_upper": {"matrices_per_s": batch / (statistics.mean(msu) / 1e3),
                            "ms_per_call": statistics.mean(msu), "route": route_u,
                            "gbs": bu * batch / (statistics.mean(msu) / 1e3) / 1e9},
            "posv_nrhs%d" % nrhs: {"matrices_per_s": batch / (statistics.mean(msp) / 1e3),
                                   "ms_per_call": statistics.mean(msp), "route": route_p},
        }

    # e2e through the C ABI with pinned host buffers
    host_in = torch.from_numpy(buf).pin_memory()
    host_out = torch.empty_like(host_in).pin_memory()
    host_info = torch.empty(batch, dtype=torch.int32).pin_memory()
    e2e_ms = []
    for it in range(args.warmup + args.steps):
        flush.zero_()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        work.copy_(host_in, non_blocking=True)
        potrf_once("L")
        host_out.copy_(work, non_blocking=True)
        host_info.copy_(info, non_blocking=True)
        e1.record(stream)
        torch.cuda.synchronize()
        if it >= args.warmup:
            e2e_ms.append(e0.elapsed_time(e1))
    e2e_step, _ = aggregate(statistics.mean(e2e_ms), batch, dist, dev)

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
                              "l2": "flushed before every step: write of %d MiB then read of another %d MiB (L2 left clean); input restored untimed" % (flusher.mib, flusher.mib),
                   "parallelism": f"weak: {ws} independent batches"},
        "gbs": alg_bytes * ws / (ms_max / 1e3) / 1e9,
        "gbs_full_storage": (2 * n * n * ESIZE[dtype] + 4) * batch * ws / (ms_max / 1e3) / 1e9,
        "gflops": potrf_flops(n, dtype) * batch * ws / (ms_max / 1e3) / 1e9,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": achieved / peaks["hbm_gbs"], "traffic": recorded_traffic(kernel_tag),
                     "algorithmic_bytes_per_launch": alg_bytes, "kernel": kernel_tag,
                     "peak_source": f"{peak_src} (copy bandwidth, burst)"},
        "e2e": {"value": ws * batch / (e2e_step / 1e3), "unit": UNIT,
                "h2d_bytes_per_step": host_in.numel() * host_in.element_size(),
                "d2h_bytes_per_step": host_out.numel() * host_out.element_size() + host_info.numel() * 4},
        "gpu_launches": args.steps,
        "clocks": sampler.summary(t0 - args.warm_seconds, t1),
        "info_all_zero": ok_info,
        "also": also,
    }
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        rate, k, t, cores = cpu_oracle_rate(w, "L", target_s=args.cpu_seconds)
        line["cpu_baseline"] = {"value": rate, "unit": UNIT, "cores": cores, "kind": "oracle",
                                "sample": f"first {k} items of the workload, {t:.1f} s wall"}
    if dist:
        dist.destroy_process_group()
    return line if rank == 0 else None


def run_reference(args):
    """The reference arm: the CPU oracle on the host cores, each step a bounded sample."""
    import oracle  # noqa: F401
    w = synth.workload(args.workload)
    cores = os.cpu_count() or 1
    rate0, k, t, _ = cpu_oracle_rate(w, "L", target_s=min(args.cpu_seconds, 3.0), max_items=2048)
    per_step = max(1, min(w.batch, int(rate0 * args.reference_step_seconds)))
    buf = synth.to_colmajor(w.A[:per_step])
    import oracle as orc
    for _ in range(args.warmup):
        orc.run("L", w.n, per_step, buf, w.n, w.n * w.n, threads=cores)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        orc.run("L", w.n, per_step, buf, w.n, w.n * w.n, threads=cores)
        times.append(time.perf_counter() - t0)
    ms = 1e3 * statistics.mean(times)
    value = per_step / (ms / 1e3)
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
        "config": {"workload": f"potrf {w.dtype} Lower n={w.n} batch={w.batch} (seed 1)",
                   "sample_per_step": per_step},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"{per_step} items per step (leading items of the workload)"},
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
    ap.add_argument("--cpu-seconds", type=float, default=8.0)
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
