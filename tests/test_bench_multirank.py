"""The benchmark's multi-rank bookkeeping (replicas, one per GPU), on CPU with two gloo ranks:
the reported time is the slowest rank's and the value counts every rank's work."""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        my_secs = 2.0 if rank == 1 else 1.0            # rank 1 is the slow one
        secs, value = bench.whole_job(my_secs, 1e12, 10, world, dist, torch.device("cpu"))
        out[rank] = (secs, value)
    finally:
        dist.destroy_process_group()


def test_whole_job_uses_slowest_rank_and_all_work():
    world = 2
    port = _free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    for rank in range(world):
        secs, value = res[rank]
        assert secs == 2.0                              # the max over ranks
        assert value == pytest.approx(1e12 * 10 * world / 2.0 / 1e12)


def test_whole_job_single_rank():
    sys.path.insert(0, ROOT)
    import bench
    secs, value = bench.whole_job(0.5, 2e12, 4, 1, None, torch.device("cpu"))
    assert secs == 0.5 and value == pytest.approx(16.0)
