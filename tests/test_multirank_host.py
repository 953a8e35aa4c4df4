"""The N > 1 bench path on CPU: two gloo ranks on 127.0.0.1.

Every rank runs its own copy of the workload (weak scaling; no collective on
the data path).  The only exchange is the reduction of the timings: the job's
time is the slowest rank's, and the job's rate counts every rank's work.
"""
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


def _rank(rank, world, port, results):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        my_ms = [12.5, 17.25][rank]                     # rank 1 is the slow one
        worst = bench.max_over_ranks(my_ms, world, torch.device("cpu"))
        results[rank] = (worst, bench.job_throughput(1.0e12, 4, world, worst))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time_and_count_all_work():
    port = _free_port()
    with mp.get_context("spawn").Manager() as mgr:     # no fork of a threaded process
        results = mgr.dict()
        mp.spawn(_rank, args=(2, port, results), nprocs=2, join=True)
        got = dict(results)
    for rank in (0, 1):
        worst, rate = got[rank]
        assert worst == 17.25
        assert rate == pytest.approx(2 * 1.0e12 * 4 / (17.25e-3) / 1e12)


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks(3.0, 1, torch.device("cpu")) == 3.0
    assert bench.job_throughput(5e11, 10, 1, 2.0) == pytest.approx(2500.0)
