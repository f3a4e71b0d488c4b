"""The batch shards across ranks with no data-path collective (every rank factors its own
items); the benchmark only reduces its timing. These tests run that host logic on CPU with
world_size 2 over gloo."""
import os
import socket

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
