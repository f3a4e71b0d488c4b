"""Tuner: time every compiled variant on a grid of shapes and write the selection tables.

Method (BatchLAS "Flat kernel selection", section 6, the tuner; sections 6.1-6.4: grid, edge
refinement, noise protocol, table regeneration):

* grid: potrf n over 34 values including the +1 rungs (17, 33, 65, 129) x batch in {128, 512,
  2048, 8192, 32768}; posv 12 values of n x nrhs in {1, 4, 8} x batch in {1024, 16384}; per dtype
  and uplo (a cell is skipped when one copy of its batch would exceed the memory budget);
* every candidate is pinned and run through the public entry point and verified first (info
  all zero and a float64 residual ||A - L L^H|| / ||A|| on a few items of a small batch); a
  candidate that fails is dropped from the cell;
* timing: the benchmark's back-to-back protocol (protocol.py: each call on its own pristine
  copy, the copies of a chunk larger than four times L2, L2 flushed before each chunk), the
  candidates interleaved in two passes, the second in reverse order; a candidate's time is the
  median of its chunks over both passes; when the two passes disagree by more than 10% on the
  cell's winner, the cell is measured once more and that measurement replaces it;
* edge refinement: along n, between neighbouring grid points whose winners differ, the midpoint
  is measured (recursively, up to --bisect levels) so the table rows bracket every change of
  winner;
* every measurement is appended to a JSONL ledger; the tables are regenerated from the ledger
  alone (ledger_to_tables), fastest candidate first per row.

Usage: python -m matrix_dense_linear_spd_gb300.sweep --op potrf --out DIR [--dtypes f32]
       [--n 4,8,...] [--batches 128,...] [--max-seconds S]
       python -m matrix_dense_linear_spd_gb300.sweep --tables-from DIR/potrf.sm_103.jsonl --out DIR
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

ESIZE = {"f32": 4, "f64": 8, "c64": 8, "c128": 16}
EPS = {"f32": 2.0 ** -24, "c64": 2.0 ** -24, "f64": 2.0 ** -53, "c128": 2.0 ** -53}

N_GRID = [1, 2, 3, 4, 5, 6, 7, 8, 12, 16, 17, 20, 24, 28, 32, 33, 40, 48, 56, 64, 65, 72, 80, 96,
          112, 128, 129, 144, 160, 192, 256, 320, 384, 512]
BATCHES = [128, 512, 2048, 8192, 32768]
POSV_N = [4, 8, 16, 17, 32, 33, 64, 65, 128, 144, 256, 512]
POSV_BATCHES = [1024, 16384]
NOISE = 0.10                       # pass disagreement that triggers a re-measurement


# ------------------------------------------------------------------ ledger -> tables (host only)

def cell_key(r):
    return (r["op"], r["dtype"], r["uplo"], int(r["n"]), int(r.get("nrhs", 0)), int(r["batch"]))


def ledger_to_tables(records):
    """Rows per op from ledger records. A cell's latest measurement (the largest (run, attempt))
    replaces earlier ones; a candidate's time is the median of its samples in that measurement;
    candidates are ranked by time, ties by spelling. Returns {op: [(key dict, [(spelling, ms),
    ...]), ...]} with rows ordered by dtype, uplo, n, nrhs, batch."""
    cells = {}
    for r in records:
        if r.get("kind", "time") != "time":
            continue
        k = cell_key(r)
        att = (float(r.get("run", 0)), int(r.get("attempt", 0)))
        c = cells.setdefault(k, {"attempt": att, "samples": {}})
        if att > c["attempt"]:
            cells[k] = c = {"attempt": att, "samples": {}}
        elif att < c["attempt"]:
            continue
        c["samples"].setdefault(r["candidate"], []).append(float(r["ms"]))
    out = {}
    dorder = {"f32": 0, "f64": 1, "c64": 2, "c128": 3}
    for k in sorted(cells, key=lambda k: (k[0], dorder.get(k[1], 9), k[2], k[3], k[4], k[5])):
        op, dtype, uplo, n, nrhs, batch = k
        ranked = sorted(((sp, statistics.median(v)) for sp, v in cells[k]["samples"].items()),
                        key=lambda t: (t[1], t[0]))
        key = {"dtype": dtype, "uplo": uplo, "n": n, "batch": batch}
        if op != "potrf":
            key["nrhs"] = nrhs
        out.setdefault(op, []).append((key, ranked))
    return out


def format_table(op, devkey, rows, source, date=None, top=12):
    keys = "dtype:exact uplo:exact n:log:3" + (" nrhs:log" if op != "potrf" else "") + " batch:log"
    lines = [f"# op={op} device={devkey} source=ledger:{source} date={date or time.strftime('%Y-%m-%d')} "
             f"(median ms per call over two interleaved passes, back-to-back protocol, whole batch; "
             f"the {top} fastest verified candidates per row)",
             f"# keys: {keys}"]
    for key, ranked in rows:
        head = f"dtype={key['dtype']} uplo={key['uplo']} n={key['n']}"
        if op != "potrf":
            head += f" nrhs={key['nrhs']}"
        head += f" batch={key['batch']}"
        lines.append(head + " | " + " | ".join(f"{sp} {ms:.5f}" for sp, ms in ranked[:top]) + " # measured")
    return "\n".join(lines) + "\n"


def read_ledger(path):
    import gzip
    opener = gzip.open if path.endswith(".gz") else open
    with opener(path, "rt") as f:
        return [json.loads(x) for x in f if x.strip()]


LEDGER_DIR = os.path.join(os.path.dirname(os.path.abspath(__file__)), "tuned", "ledger")


def shipped_ledgers(op):
    """The committed ledgers of `op` (tuned/ledger/<op>_run<k>.jsonl.gz), in run order; the
    shipped table of `op` is their verdict."""
    import glob
    import re
    files = glob.glob(os.path.join(LEDGER_DIR, f"{op}_run*.jsonl.gz"))
    return sorted(files, key=lambda p: int(re.search(r"_run(\d+)\.", os.path.basename(p)).group(1)))


def write_tables(ledger_path, out_dir, devkey=None):
    recs = []
    for p in ledger_path.split(","):
        recs += read_ledger(p)
    devkey = devkey or (recs[0]["device"] if recs else "sm_103")
    written = []
    for op, rows in ledger_to_tables(recs).items():
        path = os.path.join(out_dir, f"{op}.{devkey}.txt")
        with open(path, "w") as f:
            f.write(format_table(op, devkey, rows, ",".join(os.path.basename(p) for p in ledger_path.split(","))))
        written.append(path)
    return written


def bisect_points(winners, max_gap=1):
    """Midpoints to measure along n: for neighbouring grid points (a, wa), (b, wb) with wa != wb
    and b - a > max_gap, the integer midpoint. `winners` is [(n, winner)] sorted by n."""
    pts = []
    for (a, wa), (b, wb) in zip(winners, winners[1:]):
        if wa != wb and b - a > max_gap:
            pts.append((a + b) // 2)
    return pts


# ------------------------------------------------------------------ measurement (GPU)

def residual_ok(A, F, uplo, dtype, items):
    import synth
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
    """Inputs of one cell on the device: R pristine copies for the back-to-back protocol."""

    def __init__(self, op, dtype, uplo, n, batch, nrhs, torch, l2, steps):
        import synth
        from matrix_dense_linear_spd_gb300 import protocol as P
        self.op, self.dtype, self.uplo, self.n, self.batch, self.nrhs = op, dtype, uplo, n, batch, nrhs
        rng = np.random.default_rng(1000 + n)
        self.A = synth.spd_bbt(rng, n, batch, dtype)
        bufs = [torch.from_numpy(synth.to_colmajor(self.A)).cuda()]
        if op != "potrf":
            self.B = synth.rhs_uniform(rng, n, nrhs, batch, dtype)
            bufs.append(torch.from_numpy(synth.to_colmajor(self.B)).cuda())
        total = sum(b.numel() * b.element_size() for b in bufs)
        self.rot = P.Rotation(bufs, P.copies_per_chunk(total, l2, steps))
        self.infos = torch.zeros((self.rot.r, batch), dtype=torch.int32, device="cuda")
        self.iptr = [self.infos[i].data_ptr() for i in range(self.rot.r)]
        self.aptr = [self.rot.ptr(0, i) for i in range(self.rot.r)]
        self.bptr = [self.rot.ptr(1, i) for i in range(self.rot.r)] if op != "potrf" else None

    def call(self, i, stream, batch=None):
        import matrix_dense_linear_spd_gb300 as bl
        code = bl.DTYPE_CODES[self.dtype]
        n, b = self.n, batch or self.batch
        if self.op == "potrf":
            bl.potrf_ptr(self.uplo, code, n, b, self.aptr[i], n, n * n, self.iptr[i], stream)
        else:
            bl.posv_ptr(self.uplo, code, n, self.nrhs, b, self.aptr[i], n, n * n, self.bptr[i], n, n * self.nrhs,
                        self.iptr[i], stream)


def verify(cell, cands, torch):
    """(candidates that run the cell's shape correctly, candidates that ran but failed the
    check), on a sub-batch of at most 256 items. A candidate that cannot run the shape (the pin
    is refused) is in neither list."""
    import matrix_dense_linear_spd_gb300 as bl
    import synth
    sp = torch.cuda.current_stream().cuda_stream
    vb = min(cell.batch, 256)
    ok, bad = [], []
    for c in cands:
        bl.set_route(cell.op, c)
        try:
            cell.rot.restore()
            cell.infos.zero_()
            cell.call(0, sp, vb)
            torch.cuda.synchronize()
        except bl.BLError:
            continue
        finally:
            bl.set_route(cell.op, None)
        F = synth.from_colmajor(cell.rot.work[0][0][: vb * cell.n * cell.n].cpu().numpy(), cell.n, cell.n, vb)
        if int(cell.infos[0, :vb].abs().sum().item()) == 0 and \
                residual_ok(cell.A, F, cell.uplo, cell.dtype, sorted({0, vb - 1})):
            ok.append(c)
        else:
            bad.append(c)
    return ok, bad


def time_cell(cell, cands, torch, flush, chunks):
    """{candidate: (median pass-1 ms, median pass-2 ms, all samples)} over two interleaved
    passes (the second in reverse order), `chunks` back-to-back chunks per candidate per pass."""
    import matrix_dense_linear_spd_gb300 as bl
    from matrix_dense_linear_spd_gb300 import protocol as P
    s = torch.cuda.current_stream()
    res = {c: ([], []) for c in cands}
    for pas, order in enumerate((cands, cands[::-1])):
        for rep in range(chunks + 1):
            for c in order:
                bl.set_route(cell.op, c)
                try:
                    pc, _ = P.time_back_to_back(lambda i: cell.call(i, s.cuda_stream), cell.rot, flush, cell.rot.r, s,
                                                warm_chunks=0)
                finally:
                    bl.set_route(cell.op, None)
                if rep > 0:                                   # rep 0 warms every candidate
                    res[c][pas].extend(pc)
    return res


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--op", choices=["potrf", "posv"], default="potrf")
    ap.add_argument("--dtypes", default="f32,f64,c64,c128")
    ap.add_argument("--uplos", default="L,U")
    ap.add_argument("--n", default=None, help="comma list overriding the n grid")
    ap.add_argument("--nrhs", default="1,4,8")
    ap.add_argument("--batches", default=None, help="comma list overriding the batch grid")
    ap.add_argument("--chunks", type=int, default=2, help="timed chunks per candidate per pass")
    ap.add_argument("--bisect", type=int, default=2, help="levels of edge refinement along n")
    ap.add_argument("--mem-budget", type=float, default=1.0, help="GiB per copy of a cell's batch")
    ap.add_argument("--out", required=True)
    ap.add_argument("--max-seconds", type=float, default=1e9)
    ap.add_argument("--tables-from", default=None, help="only regenerate tables from these ledgers (comma list)")
    ap.add_argument("--regenerate", action="store_true",
                    help="only regenerate both tables from every committed ledger (tuned/ledger), into --out")
    ap.add_argument("--cells", default=None,
                    help="explicit cells instead of the grid: dtype:uplo:n:batch[:nrhs] separated by commas")
    ap.add_argument("--min-n", type=int, default=0, help="skip grid points below this n")
    a = ap.parse_args(argv)
    os.makedirs(a.out, exist_ok=True)
    if a.tables_from:
        for p in write_tables(a.tables_from, a.out):
            print(p)
        return 0
    if a.regenerate:
        for op in ("potrf", "posv"):
            for p in write_tables(",".join(shipped_ledgers(op)), a.out):
                print(p)
        return 0
    import torch
    import matrix_dense_linear_spd_gb300 as bl
    from matrix_dense_linear_spd_gb300 import protocol as P
    dev = torch.cuda.get_device_properties(0)
    devkey = f"sm_{dev.major}{dev.minor}"
    l2 = dev.L2_cache_size
    flush = P.L2Flush(l2, "cuda")
    ns = [int(x) for x in a.n.split(",")] if a.n else (N_GRID if a.op == "potrf" else POSV_N)
    batches = [int(x) for x in a.batches.split(",")] if a.batches else (BATCHES if a.op == "potrf" else POSV_BATCHES)
    nrhss = [int(x) for x in a.nrhs.split(",")] if a.op == "posv" else [0]
    ledger_path = os.path.join(a.out, f"{a.op}.{devkey}.jsonl")
    ledger = open(ledger_path, "a")
    t_start = time.time()

    def log(rec):
        ledger.write(json.dumps(rec) + "\n")
        ledger.flush()

    run = round(t_start, 3)

    def measure(dtype, uplo, n, batch, nrhs, cands_all):
        base = {"op": a.op, "device": devkey, "dtype": dtype, "uplo": uplo, "n": n, "nrhs": nrhs, "batch": batch,
                "run": run}
        cell = Cell(a.op, dtype, uplo, n, batch, nrhs, torch, l2, 20)
        cands, bad = verify(cell, cands_all, torch)
        for c in bad:
            log(dict(base, kind="rejected", candidate=c))
        best = None
        for attempt in range(2):
            res = time_cell(cell, cands, torch, flush, a.chunks)
            for c, (p1, p2) in res.items():
                for pas, v in ((0, p1), (1, p2)):
                    for ms in v:
                        log(dict(base, kind="time", candidate=c, ms=ms, attempt=attempt, pass_=pas))
            med = {c: statistics.median(p1 + p2) for c, (p1, p2) in res.items() if p1 + p2}
            if not med:
                break
            best = min(med, key=med.get)
            m1, m2 = statistics.median(res[best][0]), statistics.median(res[best][1])
            if abs(m1 - m2) <= NOISE * min(m1, m2):
                break
        del cell
        torch.cuda.empty_cache()
        return best

    if a.cells:
        for spec in a.cells.split(","):
            f = spec.split(":")
            dtype, uplo, n, batch = f[0], f[1], int(f[2]), int(f[3])
            nrhs = int(f[4]) if len(f) > 4 else 0
            w = measure(dtype, uplo, n, batch, nrhs, [sp for sp, cap, rhs in bl.routes(dtype)])
            print(f"{a.op} {dtype} {uplo} n={n} nrhs={nrhs} batch={batch}: {w} (cell)", flush=True)
        ledger.close()
        for p in write_tables(ledger_path, a.out, devkey):
            print(p)
        return 0

    for dtype in a.dtypes.split(","):
        cands_all = [sp for sp, cap, rhs in bl.routes(dtype)]
        for uplo in a.uplos.split(","):
            for batch in batches:
                for nrhs in nrhss:
                    winners = []
                    for n in ns:
                        if n < a.min_n or n * n * ESIZE[dtype] * batch > a.mem_budget * (1 << 30):
                            continue
                        if time.time() - t_start > a.max_seconds:
                            break
                        w = measure(dtype, uplo, n, batch, nrhs, cands_all)
                        print(f"{a.op} {dtype} {uplo} n={n} nrhs={nrhs} batch={batch}: {w}", flush=True)
                        if w:
                            winners.append((n, w))
                    done = {n for n, _ in winners}
                    for level in range(a.bisect):
                        pts = [m for m in bisect_points(sorted(winners)) if m not in done]
                        for m in pts:
                            if time.time() - t_start > a.max_seconds:
                                break
                            w = measure(dtype, uplo, m, batch, nrhs, cands_all)
                            print(f"{a.op} {dtype} {uplo} n={m} nrhs={nrhs} batch={batch}: {w} (edge)", flush=True)
                            done.add(m)
                            if w:
                                winners.append((m, w))
    ledger.close()
    for p in write_tables(ledger_path, a.out, devkey):
        print(p)
    return 0


if __name__ == "__main__":
    sys.exit(main())
