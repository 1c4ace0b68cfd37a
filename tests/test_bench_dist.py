"""bench.py's multi-rank aggregation on CPU: two gloo ranks, each with its
own step time, agree on the slowest rank's time and the whole-job value."""
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


def _worker(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port),
                      RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        step_ms = [2.0, 3.0][rank]
        ms, value = bench.aggregate_ranks(step_ms, 6_000_000, world)
        results[rank] = (ms, value, bench.dist_env())
    finally:
        dist.destroy_process_group()


def test_two_rank_aggregation():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        results = m.dict()
        mp.spawn(_worker, args=(world, port, results), nprocs=world, join=True)
        res = dict(results)
    for rank in range(world):
        ms, value, env = res[rank]
        assert ms == 3.0                              # the slowest rank
        assert value == pytest.approx(2 * 6_000_000 / 3e-3 / 1e9)
        assert env == (rank, world, rank)


def test_single_rank_aggregation():
    ms, value = bench.aggregate_ranks(1.5, 3_000_000, 1)
    assert ms == 1.5 and value == pytest.approx(2.0)
