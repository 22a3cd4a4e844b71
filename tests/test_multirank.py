"""The bench's multi-rank host logic on CPU: two gloo ranks stand in for two GPUs.

The chain has no exchange step, so N GPUs run N independent replicas; what the ranks
share is the timing: every rank times its replica, the job's time is the slowest rank's
(an all-reduce MAX), and the whole-job value counts every replica's work.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, secs, out):
    import torch
    import torch.distributed as dist
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        sec = bench.max_over_ranks(secs[rank], dist, torch.device("cpu"))
        out.put((rank, sec))
        dist.barrier()
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("secs", [(1.25, 3.5), (2.0, 0.5)])
def test_job_time_is_the_slowest_rank(secs):
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, secs, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = dict(out.get(timeout=10) for _ in range(2))
    assert got == {0: max(secs), 1: max(secs)}


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks(0.75, None, None) == 0.75


def test_whole_job_value_counts_every_replica():
    flops = 6.442450944e9                      # the FFN chain's MMA flops per step
    one = bench.whole_job_value(flops, 1000, 0.01, 1)
    assert one == pytest.approx(644.2450944)
    # two replicas doing the same work in the same (slowest-rank) time: twice the value
    assert bench.whole_job_value(flops, 1000, 0.01, 2) == pytest.approx(2 * one)


def test_rank_environment(monkeypatch):
    monkeypatch.setenv("WORLD_SIZE", "4")
    monkeypatch.setenv("RANK", "3")
    monkeypatch.setenv("LOCAL_RANK", "1")
    assert bench.dist_env() == (4, 3, 1)
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        monkeypatch.delenv(k)
    assert bench.dist_env() == (1, 0, 0)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch):
    # under torchrun the other ranks exit at once, without work (args is never read)
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    assert bench.run_reference(None) is None
