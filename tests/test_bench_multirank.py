"""The multi-rank plumbing of bench.py on CPU: two gloo ranks, max-over-ranks timing
and the whole-job throughput (replicas: tokens of every rank / slowest rank)."""

import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    local_ms = 100.0 + 50.0 * rank          # rank 1 is the slow one
    total = bench.reduce_max(local_ms, "cpu")
    value = bench.whole_job_throughput(world, 10, 1000, total)
    out[rank] = (total, value)
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_aggregation():
    world = 2
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_worker, args=(world, _free_port(), out), nprocs=world, join=True)
    for r in range(world):
        total, value = out[r]
        assert total == 150.0
        assert value == pytest.approx(2 * 10 * 1000 / 0.150)


def test_single_process_identity():
    import bench
    assert bench.reduce_max(3.5, "cpu") == 3.5
    assert bench.whole_job_throughput(1, 4, 100, 2000.0) == pytest.approx(200.0)
