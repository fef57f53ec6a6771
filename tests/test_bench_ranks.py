"""The bench's multi-rank host logic on CPU: two gloo ranks, as torchrun
would launch them (one process per GPU, replicas on their own batches)."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        f = bench.max_over_ranks_fn(world, torch.device("cpu"))
        local_ms = 10.0 + 5.0 * rank           # rank 1 is the slower one
        mx = f(local_ms)
        value = bench.job_throughput(world, 8192, 4, mx)
        seeds = [bench.rank_seed(b, rank) for b in (1003, 1103, 1203)]
        out[rank] = (mx, value, seeds)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_time():
    world, port = 2, _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    # every rank sees the slowest rank's time
    assert res[0][0] == res[1][0] == 15.0
    # whole-job tokens/s: both ranks' tokens over the slowest time
    assert res[0][1] == pytest.approx(2 * 8192 * 4 / 15e-3)
    # each rank draws its own inputs
    assert set(res[0][2]).isdisjoint(res[1][2])


def test_one_rank_is_the_identity():
    f = bench.max_over_ranks_fn(1, torch.device("cpu"))
    assert f(3.5) == 3.5
    assert bench.job_throughput(1, 8192, 10, 2.0) == pytest.approx(8192 * 10 / 2e-3)
