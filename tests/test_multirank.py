"""The bench's multi-rank path on CPU: two gloo ranks agree on the slowest
rank's time, the whole-job rate counts every rank's rows, and the reference
arm does its work on rank 0 only."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, times, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = bench.max_over_ranks(times[rank], world, "cpu")
        rate = bench.whole_job_rate(world, 512, 10, ms)
        dist.barrier()
        out[rank] = (ms, rate)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    world, port = 2, _free_port()
    times = [3.5, 7.25]
    out = mp.get_context("spawn").Manager().dict()  # no fork of this (threaded) process
    mp.spawn(_rank, args=(world, port, times, out), nprocs=world, join=True)
    for r in range(world):
        ms, rate = out[r]
        assert ms == 7.25
        assert rate == pytest.approx(2 * 512 * 10 / 7.25e-3)


def test_single_rank_is_unchanged():
    assert bench.max_over_ranks(4.0, 1) == 4.0
    assert bench.whole_job_rate(1, 64, 100, 2.0) == pytest.approx(64 * 100 / 2e-3)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")

    class A:
        steps, warmup, workload = 1, 0, "c1"

    bench.run_reference(A(), None, "")  # rank 1: returns before touching the workload
    assert capsys.readouterr().out == ""
