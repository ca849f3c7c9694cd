"""The replicas-only multi-GPU path of bench.py, on CPU: two gloo ranks agree
on the slowest rank's time and on the whole-job GB/s, and the reference arm
runs on rank 0 only (the other ranks exit at once)."""

import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, times, out):
    import bench

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = bench.max_over_ranks(times[rank], dist, torch.device("cpu"))
        value = bench.aggregate_gbs(world, 1_000_000_000, 10, ms)
        out.put((rank, ms, value))
    finally:
        dist.destroy_process_group()


def test_two_ranks_take_the_slowest_time():
    world, times = 2, [12.5, 20.0]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, times, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms, value in res:
        assert ms == 20.0
        # 2 ranks x 1 GB x 10 steps in 20 ms
        assert value == pytest.approx(1000.0)


def test_single_rank_needs_no_collective():
    import bench

    assert bench.max_over_ranks(7.0, None, None) == 7.0
    assert bench.aggregate_gbs(1, 16_212_295_680, 20, 122.0) == pytest.approx(2657.75, rel=1e-4)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    import bench

    class Args:
        steps, warmup, gpus = 1, 0, 2

    monkeypatch.setenv("RANK", "1")
    assert bench.run_reference(Args()) == 0
    assert capsys.readouterr().out == ""
