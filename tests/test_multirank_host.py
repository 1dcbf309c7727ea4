"""The benchmark's multi-rank aggregation on CPU with two gloo ranks.

Every rank runs an independent replica, so whole-job throughput is all ranks' units divided by
the slowest rank's time; the only collective is a MAX all-reduce of one scalar.
"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, times, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    t_max, value = bench.aggregate(times[rank], units_per_rank=1000, device="cpu")
    out[rank] = (t_max, value)
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_aggregate_takes_the_slowest_rank():
    world = 2
    port = _free_port()
    times = [40.0, 50.0]  # ms
    with mp.get_context("spawn").Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, port, times, out), nprocs=world, join=True)
        res = dict(out)
    for r in range(world):
        t_max, value = res[r]
        assert t_max == 50.0
        assert value == pytest.approx(world * 1000 / 0.050)


def test_single_process_aggregate():
    import bench
    t_max, value = bench.aggregate(25.0, units_per_rank=500)
    assert t_max == 25.0 and value == pytest.approx(500 / 0.025)
