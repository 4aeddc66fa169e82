"""Host-side logic of bench.py's N > 1 path (independent replicas, one per rank), run as two
gloo ranks on the CPU: the slowest rank's times win, the job's value counts every rank's bytes,
and the reference arm does its work on rank 0 only."""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int) -> None:
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r took (10 + r) ms in total and (20 - r) ms end to end
        step_ms, e2e_ms = bench.reduce_max_over_ranks([10.0 + rank, 20.0 - rank], "cpu")
        assert step_ms == 10.0 + (world - 1)
        assert e2e_ms == 20.0
        v = bench.whole_job_gbs(world, 1e9, 5, step_ms)
        assert abs(v - world * 5.0 / (step_ms * 1e-3)) < 1e-9
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_rank():
    mp.start_processes(_rank_main, args=(2, _free_port()), nprocs=2, join=True, start_method="spawn")


def test_single_process_reduce_is_identity():
    assert bench.reduce_max_over_ranks([3.0, 4.0], "cpu") == [3.0, 4.0]
    assert bench.whole_job_gbs(1, 2e9, 10, 1000.0) == pytest.approx(20.0)


def test_reference_arm_runs_on_rank_zero_only():
    class Args:
        steps, warmup, gpus, ref_seconds_per_step = 1, 3, 2, 0.01

    # a rank other than 0 returns at once, without touching the oracle
    assert bench.run_reference(Args(), world=2, rank=1) == 0
