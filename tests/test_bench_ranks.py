"""The benchmark's multi-rank bookkeeping on CPU with gloo, world size 2:
the job time is the slowest rank's and the whole-job value counts every
rank's calls; the reference arm runs on rank 0 only."""
from __future__ import annotations

import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import bench

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms_local = [3.0, 5.0][rank]
        out[rank] = bench.aggregate_over_ranks(ms_local, steps=100, world=world)
    finally:
        dist.destroy_process_group()


def test_aggregate_over_two_gloo_ranks():
    world, port = 2, _free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.start_processes(_rank_main, args=(world, port, out), nprocs=world, join=True, start_method="spawn")
        res = dict(out)
    for rank in range(world):
        ms_max, us_call = res[rank]
        assert ms_max == 5.0  # the slower rank
        assert us_call == pytest.approx(5.0e3 / (100 * 2))  # 200 calls in 5 ms


def test_single_rank_needs_no_process_group():
    import bench

    assert bench.aggregate_over_ranks(2.0, steps=10, world=1) == (2.0, 200.0)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch):
    import argparse

    import bench

    monkeypatch.setenv("RANK", "1")
    args = argparse.Namespace(workload="m4_n2880_k512", steps=1, warmup=3)
    assert bench.run_reference(args) is None
