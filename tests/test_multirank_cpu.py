"""The benchmark's multi-rank host logic on CPU: two gloo ranks on 127.0.0.1.

Replicas only: each rank runs its own batches (own token seed), the job's
throughput is all ranks' tokens over the slowest rank's time, and the only
collectives are the timing barrier and the max over ranks.
"""
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


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dist.barrier()
        my_ms = 10.0 + 5.0 * rank  # rank 1 is the slow one
        got = bench.max_over_ranks(my_ms, world, "cpu")
        out[rank] = (got, bench.rank_seed(0, rank), bench.job_tokens_per_s(32, world, 100, got))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time_and_distinct_batches():
    world = 2
    with mp.get_context("spawn").Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, _free_port(), out), nprocs=world, join=True)
        res = dict(out)
    assert res[0][0] == res[1][0] == 15.0
    assert res[0][1] != res[1][1]
    # 2 ranks x 32 tokens x 100 steps in 15 ms
    assert res[0][2] == pytest.approx(2 * 32 * 100 / 0.015)


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks(3.5, 1, "cpu") == 3.5
    assert bench.job_tokens_per_s(32, 1, 10, 1.0) == pytest.approx(320_000.0)
