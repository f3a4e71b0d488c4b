"""Batch sharding across ranks: the items of a batch are independent, so a batch splits into
contiguous per-rank slices with no exchange step and no collective on the data path (each rank
factors its slice on its own GPU; only timings are reduced).

batch_slice(batch, world, rank) -> (start, count): balanced contiguous slices; the first
batch % world ranks take one item more. Slices are disjoint and cover [0, batch) in rank order.
"""
from __future__ import annotations


def batch_slice(batch: int, world: int, rank: int):
    if batch < 0 or world < 1 or not 0 <= rank < world:
        raise ValueError(f"bad slice request batch={batch} world={world} rank={rank}")
    base, extra = divmod(batch, world)
    start = rank * base + min(rank, extra)
    return start, base + (1 if rank < extra else 0)
