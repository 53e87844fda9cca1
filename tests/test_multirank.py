"""Replicas-only multi-GPU path of bench.py, exercised on CPU with two gloo ranks.

The decode path has no exchange step, so N GPUs run N independent replicas; the
only cross-rank work is the barrier and the max over ranks of the timed region.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import torch
    import torch.distributed as dist

    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = bench.max_over_ranks(1.0 + 2.5 * rank, torch.device("cpu"))
        dist.barrier()
        out[rank] = (ms, bench.job_gbs(world, 10**9, ms))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_job_throughput_with_two_gloo_ranks():
    world = 2
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.spawn(_rank_main, args=(world, _free_port(), out), nprocs=world, join=True)
    for r in range(world):
        ms, gbs = out[r]
        assert ms == pytest.approx(3.5)                       # the slowest rank's time
        assert gbs == pytest.approx(2 * 1.0 / 3.5e-3)         # 2 replicas x 1 GB / 3.5 ms


def test_single_process_is_its_own_max():
    import torch

    import bench
    assert bench.max_over_ranks(4.25, torch.device("cpu")) == 4.25
    assert bench.job_gbs(1, 2 * 10**9, 2.0) == pytest.approx(1000.0)
