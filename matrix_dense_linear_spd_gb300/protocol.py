"""Timing protocol shared by the benchmark, the per-workload report and the tuner.

The operations work in place, so every timed call needs a pristine input. Two ways of timing
are provided, both with CUDA events on the launching stream:

* back to back (the throughput figure): a chunk of R calls is enqueued without any host
  synchronisation or other work between them, call i factoring its own pristine copy i of the
  batch. The R copies together are larger than four times the L2 cache, and L2 is flushed after
  the copies are restored, so every call reads its input from HBM. Events bracket the chunk;
  the per-call time is the chunk time divided by R, so launch latency overlaps the previous
  call as it does for a caller issuing calls in a stream. Copies are restored (untimed) before
  each chunk.
* isolated (one call on its own): restore, flush L2, then events around a single call. This
  adds the launch latency and the event overhead of one call to every measurement.

Statistics: median over chunks (or calls), and the relative standard deviation; a rel_sd above
10% marks a measurement as noisy ("Small-n baseline" page, noise protocol).
"""
from __future__ import annotations

import math
import statistics


class L2Flush:
    """Evict L2: write one buffer larger than L2, then read a second one, so the lines left in
    L2 are clean and no write-back of the flush lands inside a timed call."""

    def __init__(self, l2_bytes: int, device):
        import torch
        n = max(2 * l2_bytes, 256 << 20) // 4
        self.a = torch.empty(n, dtype=torch.float32, device=device)
        self.b = torch.ones(n, dtype=torch.float32, device=device)
        self.sink = torch.empty((), dtype=torch.float32, device=device)
        self.mib = n * 4 >> 20

    def __call__(self):
        import torch
        self.a.zero_()
        torch.sum(self.b, dim=0, out=self.sink)


def copies_per_chunk(item_bytes_total: int, l2_bytes: int, steps: int, max_bytes: int = 4 << 30,
                     target: int = 20) -> int:
    """Calls per back-to-back chunk: enough distinct copies to exceed 4x L2 and, memory
    permitting, about `target` calls so the chunk's first launch is amortised."""
    need = max(1, math.ceil(4 * l2_bytes / max(item_bytes_total, 1)))
    fit = max(1, max_bytes // max(item_bytes_total, 1))
    return max(1, min(steps, max(need, min(target, fit))))


class Rotation:
    """R pristine copies of one or more device buffers (e.g. A and B), restored together."""

    def __init__(self, pristine: list, r: int):
        import torch
        self.pristine = pristine
        self.r = r
        self.work = [torch.empty((r,) + tuple(p.shape), dtype=p.dtype, device=p.device) for p in pristine]

    def restore(self):
        for w, p in zip(self.work, self.pristine):
            w.copy_(p.unsqueeze(0).expand_as(w))

    def ptr(self, buf: int, i: int) -> int:
        return self.work[buf][i].data_ptr()


def stats(v):
    v = list(v)
    med = statistics.median(v)
    mean = statistics.mean(v)
    sd = statistics.pstdev(v) if len(v) > 1 else 0.0
    return {"median": med, "mean": mean, "rel_sd": (sd / mean) if mean > 0 else 0.0, "n": len(v),
            "min": min(v), "max": max(v)}


def time_back_to_back(call, rot: Rotation, flush, steps: int, stream, warm_chunks: int = 1):
    """Per-call ms of each chunk (chunks of rot.r calls; `call(i)` enqueues the call on copy i).
    Returns (per-call ms list over the timed chunks, total ms over exactly `steps` calls)."""
    import torch
    for _ in range(warm_chunks):
        rot.restore()
        flush()
        for i in range(rot.r):
            call(i)
    torch.cuda.synchronize()
    per_call, total, done = [], 0.0, 0
    while done < steps:
        k = min(rot.r, steps - done)
        rot.restore()
        flush()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(k):
            call(i)
        e1.record(stream)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1)
        total += ms
        per_call.append(ms / k)
        done += k
    return per_call, total


def time_isolated(call, rot: Rotation, flush, reps: int, stream, warmup: int = 2):
    """ms of single calls, each after a restore and an L2 flush (events around the call)."""
    import torch
    out = []
    for it in range(warmup + reps):
        rot.restore()
        flush()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        call(0)
        e1.record(stream)
        torch.cuda.synchronize()
        if it >= warmup:
            out.append(e0.elapsed_time(e1))
    return out
