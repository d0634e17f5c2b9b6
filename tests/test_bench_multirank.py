"""The bench's multi-rank logic on CPU: two gloo ranks, the slowest rank's time sets the job's time,
and the job's value is the work of all ranks over that time (replicas of the whole workload)."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = 100.0 + 50.0 * rank                 # rank 1 is the slow one
        slowest = bench.reduce_max(local_ms, dist)
        dist.barrier()
        out[rank] = (slowest, bench.whole_job_rate(2.0e12, world, slowest))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    world = 2
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_rank_main, args=(world, _free_port(), out), nprocs=world, join=True)
        res = dict(out)
    assert res[0] == res[1]
    slowest, rate = res[0]
    assert slowest == 150.0
    assert rate == pytest.approx(2 * 2.0e12 / 0.150)


def test_single_rank_helpers():
    assert bench.reduce_max(3.5, None) == 3.5
    assert bench.whole_job_rate(1.0e12, 1, 1000.0) == pytest.approx(1.0e12)
    assert bench.measured_traffic("no_such_workload") is None
