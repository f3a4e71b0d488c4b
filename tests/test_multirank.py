"""The batch shards across ranks with no data-path collective (every rank factors its own
items); the benchmark only reduces its timing. These tests run that host logic on CPU with
world_size 2 over gloo: the timing reduction, and the contiguous slicing of one batch, checked
item for item against a single-rank run of the oracle."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms_local = 2.0 if rank == 0 else 3.0           # rank 1 is the slow one
    ms_max, value = bench.aggregate(ms_local, batch=1000, dist=dist, device="cpu")
    out[rank] = (ms_max, value)
    dist.barrier()
    dist.destroy_process_group()


def test_weak_scaling_aggregate_takes_the_slowest_rank():
    world = 2
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_worker, args=(world, _free_port(), out), nprocs=world, join=True)
    for r in range(world):
        ms_max, value = out[r]
        assert ms_max == 3.0
        assert value == pytest.approx(world * 1000 / 3e-3)


def test_single_rank_aggregate_is_local():
    import bench
    ms, value = bench.aggregate(4.0, batch=10, dist=None)
    assert ms == 4.0 and value == pytest.approx(10 / 4e-3)


@pytest.mark.parametrize("batch,world", [(37, 2), (8, 3), (5, 8), (0, 2), (1024, 4)])
def test_batch_slices_are_contiguous_disjoint_and_balanced(batch, world):
    from matrix_dense_linear_spd_gb300.shard import batch_slice
    nxt = 0
    counts = []
    for r in range(world):
        start, count = batch_slice(batch, world, r)
        assert start == nxt
        nxt = start + count
        counts.append(count)
    assert nxt == batch
    assert max(counts) - min(counts) <= 1


N_SLICE, BATCH_SLICE = 9, 37


def _slice_worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import oracle
    import synth
    from matrix_dense_linear_spd_gb300.shard import batch_slice
    A = synth.spd_bbt(np.random.default_rng(5), N_SLICE, BATCH_SLICE, "f64")
    A[3, 4, 4] = -1.0                                # a planted failure in rank 0's slice
    A[30, 0, 0] = -1.0                               # and one in rank 1's
    start, count = batch_slice(BATCH_SLICE, world, rank)
    buf = synth.to_colmajor(A[start:start + count])
    f, _, info = oracle.run("L", N_SLICE, count, buf, N_SLICE, N_SLICE * N_SLICE)
    parts = [None] * world
    dist.all_gather_object(parts, (start, f.astype(np.float64), info))
    if rank == 0:
        out["parts"] = parts
    dist.barrier()
    dist.destroy_process_group()


def test_sliced_batch_reassembles_to_the_single_rank_result():
    import oracle
    import synth
    world = 2
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_slice_worker, args=(world, _free_port(), out), nprocs=world, join=True)
    A = synth.spd_bbt(np.random.default_rng(5), N_SLICE, BATCH_SLICE, "f64")
    A[3, 4, 4] = -1.0
    A[30, 0, 0] = -1.0
    f_all, _, info_all = oracle.run("L", N_SLICE, BATCH_SLICE, synth.to_colmajor(A), N_SLICE, N_SLICE * N_SLICE)
    F = np.zeros((BATCH_SLICE, N_SLICE, N_SLICE))
    info = np.full(BATCH_SLICE, -7, np.int32)
    for start, f, inf in out["parts"]:
        F[start:start + len(inf)] = f
        info[start:start + len(inf)] = inf
    assert np.array_equal(info, info_all) and info[3] == 5 and info[30] == 1
    assert np.array_equal(F, f_all.astype(np.float64))
