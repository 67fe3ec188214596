"""bench.py's multi-GPU path, run as world_size-2 gloo ranks on CPU.

With several GPUs bench.py runs one independent replica per rank (the
sharded step has no data-path collective); the ranks only meet at a barrier
and in a max over their elapsed times, and rank 0 reports the job-wide
throughput.  These tests exercise that plumbing with the gloo backend."""
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


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier(dist)
        my_ms = 100.0 + 50.0 * rank                 # rank 1 is the slow replica
        ms_max = bench.max_over_ranks(dist, my_ms)
        value = bench.job_value(1000, 10, world, ms_max)
        q.put((rank, ms_max, value, bench.dist_env()))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_replica():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms_max, value, env in res:
        assert ms_max == 150.0                      # every rank sees the max
        assert value == pytest.approx(1000 * 10 * 2 / 0.150)
        assert env == (2, rank, rank)


def _reference_worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import io
    import contextlib
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        bench.run_reference(None, world, rank)      # ranks other than 0 return without work
    q.put((rank, buf.getvalue()))


def test_reference_arm_runs_on_rank_zero_only():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    p = ctx.Process(target=_reference_worker, args=(1, world, port, q))  # rank 1 of 2
    p.start()
    rank, out = q.get(timeout=120)
    p.join(timeout=60)
    assert p.exitcode == 0 and rank == 1 and out == ""


def test_job_value_single_rank():
    assert bench.job_value(1_364_297_728, 200, 1, 1752.0) == pytest.approx(
        1_364_297_728 * 200 / 1.752)


class _FakeStep:
    """Just what run_e2e reads before its first CUDA call."""

    def __init__(self):
        self.info = {"total_numel": 64, "unpadded_numel": 60}
        self.N = 2
        self.n_out = 1
        self.out_numel = 64
        self.grads = [torch.zeros(64, dtype=torch.bfloat16) for _ in range(2)]

        class _PS:
            dtype = torch.bfloat16
        self.ps = _PS()


def _e2e_worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank), LOCAL_WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    real_empty = torch.empty

    def empty(*a, pin_memory=False, **k):
        # rank 1 cannot pin host memory; rank 0 can (served unpinned on CPU)
        if pin_memory and rank == 1:
            raise RuntimeError("pinned allocation refused (injected)")
        return real_empty(*a, **k)
    torch.empty = empty
    try:
        res = bench.run_e2e(_FakeStep(), None, None, dist)
        q.put((rank, res))
    finally:
        torch.empty = real_empty
        dist.destroy_process_group()


def test_e2e_ranks_leave_together_when_one_cannot_pin():
    """A rank whose pinned host allocation fails must not leave the others
    waiting at the timed region's barrier: every rank reports the leg skipped."""
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_e2e_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, r in res:
        assert r["value"] is None
        assert "pinned host allocation failed" in r["skipped"]
    assert "injected" in res[1][1]["skipped"]


def test_host_stall_detection():
    """The re-timing guard fires on one step far above the rest, not on jitter."""
    assert not bench.host_stall([])
    assert not bench.host_stall([8.7] * 200)
    assert not bench.host_stall([8.7] * 199 + [9.5])           # ordinary jitter
    assert bench.host_stall([8.7] * 199 + [4550.0])            # a multi-second stall
    assert bench.host_stall([0.44, 4550.0, 0.44])
    assert not bench.host_stall([0.02] * 99 + [0.5])           # 25x, but under 1 ms


def _run_reference_line(monkeypatch, budget_s):
    import argparse
    import contextlib
    import io
    import json

    import workloads as W
    ps = W.llama_1b2(world_size=8, layers=3, hidden=48, ffn=136, vocab=96)  # 4 groups
    monkeypatch.setattr(bench, "make_workload", lambda name: ps)
    monkeypatch.setattr(bench, "REFERENCE_BUDGET_S", budget_s)
    args = argparse.Namespace(workload="small", steps=2, warmup=2, n_out=1, step_kind="fused")
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        bench.run_reference(args, 1, 0)
    return json.loads(buf.getvalue().strip().splitlines()[-1]), ps


def test_reference_arm_runs_the_whole_workload_within_its_budget(monkeypatch):
    out, ps = _run_reference_line(monkeypatch, 1e9)
    assert out["impl"] == "reference" and out["steps"] == 2 and out["warmup"] == 2
    assert out["cpu_baseline"]["sample"].startswith("the whole workload per step: all 4 groups")
    assert out["value"] > 0 and out["e2e"]["value"] == out["value"]


def test_reference_arm_cuts_to_a_prefix_of_groups_past_its_budget(monkeypatch):
    """When the first warm-up step says the warm-up and timed steps would
    take longer than REFERENCE_BUDGET_S, each step runs a prefix of the
    groups, the sample says how many, and the line still times K steps."""
    out, ps = _run_reference_line(monkeypatch, 0.0)
    assert out["steps"] == 2
    sample = out["cpu_baseline"]["sample"]
    first = ps.numels()[:ps.groups[0]]
    assert sample.startswith(f"the first 1 of 4 groups per step ({sum(first):,} params)"), sample
