"""The multi-GPU path of the bench is replicas only: one process per GPU,
each running the whole step, the job timed by its slowest replica.  Its
host logic -- the max over ranks and the whole-job aggregate -- runs here
as two gloo ranks on the CPU, plus the reference arm's rank rule."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank: int, world: int, port: int, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        mine = [12.5, 20.0][rank]  # each replica's own elapsed ms
        worst = bench.max_over_ranks(mine, world, torch.device("cpu"))
        q.put((rank, worst, bench.aggregate_gbs(1_000_000_000, 10, world, worst)))
    finally:
        dist.destroy_process_group()


def test_two_replicas_take_the_slowest_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [w for _, w, _ in got] == [20.0, 20.0]
    # 2 replicas x 10 steps x 1 GB in 20 ms
    assert got[0][2] == pytest.approx(1000.0)


def test_one_rank_needs_no_process_group():
    assert bench.max_over_ranks(3.5, 1, torch.device("cpu")) == 3.5
    assert bench.aggregate_gbs(2_000_000_000, 5, 1, 10.0) == pytest.approx(1000.0)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch):
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")

    class Args:
        steps, warmup = 1, 1
    assert bench.run_reference(Args()) is None
