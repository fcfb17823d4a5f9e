"""The multi-GPU path is replicas only (segments and kv heads are independent;
there is no exchange step): every rank runs its own step, the job is timed by
the slowest rank and its throughput is the units of all ranks over that time.
Two gloo ranks on the CPU exercise bench.py's cross-rank reduction."""

from __future__ import annotations

import os
import socket

import pytest

torch = pytest.importorskip("torch")


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    import sys

    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    torch.distributed.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = 10.0 + 5.0 * rank          # rank 1 is the slow replica
        t = bench.max_over_ranks(local_ms, world, "cpu")
        rate = bench.job_rate(1810 * 100, world, t / 1e3)
        torch.distributed.barrier()
        q.put((rank, t, rate))
    finally:
        torch.distributed.destroy_process_group()


def test_two_gloo_replicas_take_the_slowest_rank():
    import multiprocessing as mp

    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, t, rate in got:
        assert t == 15.0                       # max over ranks
        assert rate == pytest.approx(2 * 1810 * 100 / 0.015)


def test_single_rank_needs_no_collective():
    import sys

    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench

    assert bench.max_over_ranks(7.5, 1, "cpu") == 7.5
    assert bench.job_rate(100, 1, 2.0) == 50.0


def test_clock_samples_are_summarised_over_the_timed_region():
    """The bench's nvidia-smi summary keeps the samples inside the timed
    region (median SM clock, throttle reasons seen there) and falls back to
    every sample, labelled, when the region caught none."""
    import datetime

    import bench

    def line(t, sm, cap):
        ts = datetime.datetime.fromtimestamp(t).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
        return (f"{ts}, 0, {sm}, 2070, 900.0, 0x0, Not Active, Not Active, Not Active, "
                f"{'Active' if cap else 'Not Active'}\n")

    t0 = 1_800_000_000.0
    lines = [line(t0 + 0.00, 2070, False), line(t0 + 0.02, 1980, True),
             line(t0 + 0.04, 2010, True), line(t0 + 0.06, 2070, False), "garbage\n"]
    c = bench.ClockSampler(0)
    samples = c.parse(lines)
    assert len(samples) == 4
    c.t_begin, c.t_end = t0 + 0.01, t0 + 0.05
    s = c.summary(samples)
    assert s["samples_in_region"] == 2 and s["sm_mhz"] == 1995.0
    assert s["reasons"] == ["sw_power_cap"] and s["sm_max_mhz"] == 2070.0
    c.t_begin, c.t_end = t0 + 0.07, t0 + 0.08
    s = c.summary(samples)
    assert s["samples_in_region"] == 0 and s["sm_mhz"] == 2040.0 and "whole run" in s["window"]
    assert c.summary([])["samples"] == 0
