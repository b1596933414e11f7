"""CPU checks of bench.py's multi-process path (the N-GPU launch runs one replica per rank).

- two gloo ranks: every rank gets the slowest rank's time, and the whole-job rate is
  world x units / that time (weak scaling);
- the reference arm does its work on rank 0 only: other ranks return at once."""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, times, q):
    import torch.distributed as dist
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        slowest = bench.max_over_ranks(times[rank], world)
        rate = bench.whole_job_rate(world, 4255, slowest / 1e3)
        q.put((rank, slowest, rate))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_ranks_take_the_slowest_rank_and_scale_weakly():
    world, times = 2, [20.0, 27.5]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, times, q)) for r in range(world)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r for r, _, _ in got] == [0, 1]
    for _, slowest, rate in got:
        assert slowest == 27.5
        assert rate == pytest.approx(2 * 4255 / 0.0275)


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks(12.5, 1) == 12.5
    assert bench.whole_job_rate(1, 4255, 0.025) == pytest.approx(170200.0)


def test_reference_arm_runs_on_rank_0_only(monkeypatch):
    monkeypatch.setenv("RANK", "1")
    assert bench.run_reference(None) is None      # returns before touching the oracle or its arguments
