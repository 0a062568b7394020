"""The multi-rank (replica) host logic of bench.py on CPU: two gloo ranks.

bench.py under torchrun runs the same workload on every rank's GPU with no
collective on the data path; the only cross-rank steps are the barriers
around the timed region and the max over ranks of the step time, from which
the whole-job value is computed.  These run here with the gloo backend."""
from __future__ import annotations

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank: int, world: int, port: int, out):
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        dist.barrier()
        t = bench.max_over_ranks(1.0 + 3.0 * rank)          # per-rank step times 1.0, 4.0 (ms)
        v = bench.whole_job_value(world, t)
        dist.barrier()
        out.put((rank, t, v))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_rank():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(out.get(timeout=10) for _ in range(2))
    assert [g[0] for g in got] == [0, 1]
    for _, t, v in got:
        assert t == 4.0                 # both ranks see the slowest rank's time
        assert v == pytest.approx(500.0)   # 2 ranks x one step per 4 ms


def test_single_rank_is_unchanged(monkeypatch):
    import bench
    assert bench.max_over_ranks(2.5) == 2.5
    assert bench.whole_job_value(1, 2.0) == pytest.approx(500.0)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch):
    import argparse

    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    args = argparse.Namespace(steps=1, warmup=3)
    assert bench.run_reference(args) is None
