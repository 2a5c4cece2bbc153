"""The bench's multi-rank timing on CPU ranks (gloo, world size 2): the job
throughput is the work of all ranks over the slowest rank's time."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    import torch
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    rmax, rsum, barrier = bench.make_reducers(world, torch.device("cpu"))
    barrier()
    local_seconds = [2.0, 3.0][rank]          # rank 1 is the slowest
    local_work = [10.0, 30.0][rank]
    value, t = bench.aggregate(local_seconds, local_work, rmax, rsum)
    out[rank] = (value, t)
    dist.destroy_process_group()


def test_aggregate_two_gloo_ranks():
    world, port = 2, _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank, args=(world, port, out), nprocs=world, join=True)
        for r in range(world):
            value, t = out[r]
            assert t == pytest.approx(3.0)
            assert value == pytest.approx((10.0 + 30.0) / 3.0)


def test_single_rank_is_identity():
    import torch
    import bench
    rmax, rsum, barrier = bench.make_reducers(1, torch.device("cpu"))
    barrier()
    assert bench.aggregate(2.0, 8.0, rmax, rsum) == (4.0, 2.0)
