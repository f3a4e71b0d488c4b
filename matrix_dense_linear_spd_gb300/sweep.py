"""Tuner: time every compiled variant on a grid of shapes and write the selection tables.

Method (BatchLAS "Flat kernel selection", section 6, the tuner): every candidate is pinned and
run through the public entry point; each run is verified against a host check (a relative
residual ||A - L L^H|| / ||A|| in float64 on a few items, and info == 0) and a failing candidate
is dropped from that cell; candidates are timed interleaved, the order rotated every rep, with
the trimmed mean (middle 60%) kept. Timing protocol as in bench.py: input restored and L2 flushed before every
rep (untimed), CUDA events around the call.

Output: a JSONL ledger (one record per cell and candidate) and tables
``<op>.<device>.txt`` whose rows list every verified candidate fastest first, e.g.
``dtype=f32 uplo=L n=32 batch=16384 | warp:p=8:r=4 0.0190 | tile:p=4:s=8 0.0831 # measured``.

Usage: python -m matrix_dense_linear_spd_gb300.sweep --op potrf --out DIR [--quick]
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import sys
import time

import numpy as np

_ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if _ROOT not in sys.path:
    sys.path.insert(0, _ROOT)

import synth  # noqa: E402

import matrix_dense_linear_spd_gb300 as bl  # noqa: E402

ESIZE = {"f32": 4, "f64": 8, "c64": 8, "c128": 16}
EPS = {"f32": 2.0 ** -24, "c64": 2.0 ** -24, "f64": 2.0 ** -53, "c128": 2.0 ** -53}

POTRF_N = [4, 8, 12, 16, 17, 24, 32, 33, 40, 48, 64, 65, 72, 96, 128, 144, 160, 192, 256, 384, 512]
POSV_N = [4, 8, 16, 17, 32, 33, 64, 65, 128, 144, 256, 512]


def batch_for(n: int, dtype: str, budget_bytes: int = 512 << 20, cap: int = 32768) -> int:
    b = budget_bytes // (n * n * ESIZE[dtype])
    return int(max(64, min(cap, 1 << int(np.log2(max(b, 1))))))


def residual_ok(A, F, uplo, dtype, items):
    for b in items:
        a = A[b].astype(np.complex128 if synth.is_complex(dtype) else np.float64)
        f = F[b].astype(a.dtype)
        f = np.tril(f) if uplo == "L" else np.triu(f)
        prod = f @ np.conj(f.T) if uplo == "L" else np.conj(f.T) @ f
        res = np.linalg.norm(a - prod) / np.linalg.norm(a)
        if not np.isfinite(res) or res > 64 * a.shape[0] * EPS[dtype]:
            return False
    return True


class Cell:
    def __init__(self, op, dtype, uplo, n, batch, nrhs, torch):
        self.op, self.dtype, self.uplo, self.n, self.batch, self.nrhs = op, dtype, uplo, n, batch, nrhs
        rng = np.random.default_rng(1000 + n)
        self.A = synth.spd_bbt(rng, n, batch, dtype)
        self.pristine = torch.from_numpy(synth.to_colmajor(self.A)).cuda()
        self.work = self.pristine.clone()
        self.info = torch.empty(batch, dtype=torch.int32, device="cuda")
        if op != "potrf":
            self.Bh = synth.rhs_uniform(rng, n, nrhs, batch, dtype)
            self.Bp = torch.from_numpy(synth.to_colmajor(self.Bh)).cuda()
            self.Bw = self.Bp.clone()

    def restore(self):
        self.work.copy_(self.pristine)
        if self.op != "potrf":
            self.Bw.copy_(self.Bp)

    def call(self, stream):
        code = bl.DTYPE_CODES[self.dtype]
        n = self.n
        if self.op == "potrf":
            bl.potrf_ptr(self.uplo, code, n, self.batch, self.work.data_ptr(), n, n * n, self.info.data_ptr(), stream)
        else:
            bl.posv_ptr(self.uplo, code, n, self.nrhs, self.batch, self.work.data_ptr(), n, n * n,
                        self.Bw.data_ptr(), n, n * self.nrhs, self.info.data_ptr(), stream)


def trimmed_mean(v):
    """Mean of the middle 60% of the samples: CUDA event times come in coarse ticks here
    (about 1 us), so a median of short calls is quantised; a trimmed mean resolves them."""
    v = sorted(v)
    k = len(v) // 5
    mid = v[k:len(v) - k] or v
    return sum(mid) / len(mid)


def run_cell(cell, cands, torch, flush, reps):
    s = torch.cuda.current_stream()
    sp = s.cuda_stream
    ok = []
    for c in cands:                               # verification pass (untimed)
        bl.set_route(cell.op, c)
        try:
            cell.restore()
            cell.call(sp)
        except bl.BLError:
            continue
        finally:
            bl.set_route(cell.op, None)
        torch.cuda.synchronize()
        if int(cell.info.abs().sum().item()) != 0:
            continue
        items = sorted({0, cell.batch - 1})
        F = synth.from_colmajor(cell.work.cpu().numpy(), cell.n, cell.n, cell.batch)
        if residual_ok(cell.A, F, cell.uplo, cell.dtype, items):
            ok.append(c)
    times = {c: [] for c in ok}
    for rep in range(reps + 1):
        order = ok[rep % max(1, len(ok)):] + ok[:rep % max(1, len(ok))]
        for c in order:
            bl.set_route(cell.op, c)
            try:
                cell.restore()
                flush.zero_()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(s)
                cell.call(sp)
                e1.record(s)
                torch.cuda.synchronize()
            finally:
                bl.set_route(cell.op, None)
            if rep > 0:                             # rep 0 warms every candidate
                times[c].append(e0.elapsed_time(e1))
    return {c: trimmed_mean(v) for c, v in times.items() if v}


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--op", choices=["potrf", "posv"], default="potrf")
    ap.add_argument("--dtypes", default="f32,f64,c64,c128")
    ap.add_argument("--uplos", default="L,U")
    ap.add_argument("--n", default=None, help="comma list overriding the n grid")
    ap.add_argument("--nrhs", default="1,4,8")
    ap.add_argument("--batches", default=None, help="comma list overriding the batch rule")
    ap.add_argument("--reps", type=int, default=7)
    ap.add_argument("--out", required=True)
    ap.add_argument("--max-seconds", type=float, default=1e9)
    a = ap.parse_args(argv)
    import torch
    os.makedirs(a.out, exist_ok=True)
    dev = torch.cuda.get_device_properties(0)
    devkey = f"sm_{dev.major}{dev.minor}"
    l2 = dev.L2_cache_size
    # evict L2 between reps: write one buffer larger than L2, then read another, so L2 is left
    # clean and no write-back of the flush lands inside a timed call
    fa = torch.empty(max(2 * l2, 256 << 20) // 4, dtype=torch.float32, device="cuda")
    fb = torch.ones_like(fa)
    sink = torch.empty((), dtype=torch.float32, device="cuda")

    class _Flush:
        @staticmethod
        def zero_():
            fa.zero_()
            torch.sum(fb, dim=0, out=sink)
    flush = _Flush()
    ns = [int(x) for x in a.n.split(",")] if a.n else (POTRF_N if a.op == "potrf" else POSV_N)
    nrhss = [int(x) for x in a.nrhs.split(",")] if a.op == "posv" else [0]
    ledger = open(os.path.join(a.out, f"{a.op}.{devkey}.jsonl"), "a")
    rows = []
    t_start = time.time()
    for dtype in a.dtypes.split(","):
        cands_all = [sp for sp, cap, rhs in bl.routes(dtype)]
        for uplo in a.uplos.split(","):
            for n in ns:
                batches = [int(x) for x in a.batches.split(",")] if a.batches else [batch_for(n, dtype)]
                for batch in batches:
                    for nrhs in nrhss:
                        if time.time() - t_start > a.max_seconds:
                            break
                        cell = Cell(a.op, dtype, uplo, n, batch, nrhs, torch)
                        res = run_cell(cell, cands_all, torch, flush, a.reps)
                        del cell
                        ranked = sorted(res.items(), key=lambda kv: kv[1])
                        for c, ms in ranked:
                            ledger.write(json.dumps({"op": a.op, "device": devkey, "dtype": dtype, "uplo": uplo,
                                                     "n": n, "nrhs": nrhs, "batch": batch, "candidate": c,
                                                     "ms": ms}) + "\n")
                        ledger.flush()
                        key = f"dtype={dtype} uplo={uplo} n={n}" + (f" nrhs={nrhs}" if a.op == "posv" else "") \
                            + f" batch={batch}"
                        cells = " | ".join(f"{c} {ms:.5f}" for c, ms in ranked)
                        rows.append(f"{key} | {cells} # measured")
                        best = ranked[0] if ranked else ("-", 0)
                        print(f"{key}: best {best[0]} {best[1]:.4f} ms ({len(ranked)} verified)", flush=True)
    keys = "dtype:exact uplo:exact n:log:3" + (" nrhs:log" if a.op == "posv" else "") + " batch:log"
    with open(os.path.join(a.out, f"{a.op}.{devkey}.txt"), "w") as f:
        f.write(f"# op={a.op} device={devkey} source=ledger:{a.op}.{devkey}.jsonl "
                f"date={time.strftime('%Y-%m-%d')} reps={a.reps} (trimmed-mean ms per call, whole batch)\n")
        f.write(f"# keys: {keys}\n")
        for r in rows:
            f.write(r + "\n")
    return 0


if __name__ == "__main__":
    sys.exit(main())
