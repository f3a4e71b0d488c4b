"""Run one op a few times on a seeded synthetic batch -- a small, self-contained case for
profilers (ncu) and quick timings. Prints the route and the median CUDA-event time per call.

Usage:
  python -m matrix_dense_linear_spd_gb300.profile_case --op potrf --dtype f32 --n 32 \
      --batch 65536 [--uplo L] [--nrhs 4] [--route warp:p=8:r=4] [--reps 3]
"""
from __future__ import annotations

import argparse
import os
import statistics
import sys

import numpy as np

_ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if _ROOT not in sys.path:
    sys.path.insert(0, _ROOT)

import synth  # noqa: E402

import matrix_dense_linear_spd_gb300 as bl  # noqa: E402


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--op", choices=["potrf", "posv", "potrs"], default="potrf")
    ap.add_argument("--dtype", choices=list(synth.DTYPES), default="f32")
    ap.add_argument("--n", type=int, default=32)
    ap.add_argument("--batch", type=int, default=65536)
    ap.add_argument("--uplo", default="L")
    ap.add_argument("--nrhs", type=int, default=4)
    ap.add_argument("--route", default=None)
    ap.add_argument("--reps", type=int, default=3)
    ap.add_argument("--seed", type=int, default=1)
    a = ap.parse_args(argv)
    import torch
    rng = np.random.default_rng(a.seed)
    A = synth.spd_bbt(rng, a.n, a.batch, a.dtype)
    pristine = torch.from_numpy(synth.to_colmajor(A)).cuda()
    work = pristine.clone()
    info = torch.empty(a.batch, dtype=torch.int32, device="cuda")
    code = bl.DTYPE_CODES[a.dtype]
    n = a.n
    if a.op != "potrf":
        Bp = torch.from_numpy(synth.to_colmajor(synth.rhs_uniform(rng, n, a.nrhs, a.batch, a.dtype))).cuda()
        Bw = Bp.clone()
    if a.route:
        bl.set_route(a.op, a.route)
    s = torch.cuda.current_stream()
    times = []
    for _ in range(a.reps):
        work.copy_(pristine)
        if a.op != "potrf":
            Bw.copy_(Bp)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s)
        if a.op == "potrf":
            bl.potrf_ptr(a.uplo, code, n, a.batch, work.data_ptr(), n, n * n, info.data_ptr(), s.cuda_stream)
        elif a.op == "posv":
            bl.posv_ptr(a.uplo, code, n, a.nrhs, a.batch, work.data_ptr(), n, n * n, Bw.data_ptr(), n,
                        n * a.nrhs, info.data_ptr(), s.cuda_stream)
        else:
            bl.potrs_ptr(a.uplo, code, n, a.nrhs, a.batch, pristine.data_ptr(), n, n * n, Bw.data_ptr(), n,
                         n * a.nrhs, s.cuda_stream)
        e1.record(s)
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1))
    bad = int((info != 0).sum().item()) if a.op != "potrs" else 0
    print(f"{a.op} {a.dtype} uplo={a.uplo} n={n} batch={a.batch} route={bl.last_choice()} "
          f"median {statistics.median(times):.4f} ms, failed items {bad}")
    return 0 if bad == 0 else 1


if __name__ == "__main__":
    sys.exit(main())
