"""The benchmark's multi-rank bookkeeping on CPU ranks (gloo, world size 2).

With N GPUs every rank runs its own replica of the decode step (the units are
independent, so nothing is exchanged on the data path); the only cross-rank
steps are the barriers around the timed region and the maximum of the ranks'
times.  These tests run that logic on two gloo ranks and check the whole-job
rate, and that the reference arm's non-zero ranks exit without work.
"""
import math
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, times, out_q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dist.barrier()
        got = bench.max_over_ranks(dist, times[rank], "cpu")
        dist.barrier()
        out_q.put((rank, got))
    finally:
        dist.destroy_process_group()


def test_max_over_two_gloo_ranks():
    world = 2
    times = [[10.0, float("nan")], [12.5, float("nan")]]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, times, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs)
    results = dict(q.get(timeout=10) for _ in range(world))
    for r in range(world):
        assert results[r][0] == 12.5                       # the slowest rank's time on every rank
        assert math.isnan(results[r][1])                   # no end-to-end number stays none


def test_whole_job_rate_is_weak_scaling_over_slowest_rank():
    # 4 GB per step per rank, 100 steps, slowest rank 80 ms
    one = bench.whole_job_rate(4e9, 100, 1, 80.0)
    two = bench.whole_job_rate(4e9, 100, 2, 80.0)
    assert one == pytest.approx(5000.0)
    assert two == pytest.approx(2 * one)
    assert bench.whole_job_rate(4e9, 1, 1, float("nan")) is None


def test_single_rank_needs_no_group():
    assert bench.max_over_ranks(None, [3.0, 4.0], "cpu") == [3.0, 4.0]


def test_reference_arm_nonzero_rank_exits_without_work(monkeypatch, capsys):
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("LOCAL_RANK", "1")

    class Args:
        steps, warmup, gpus = 3, 3, 2

    assert bench.run_reference(Args()) == 0
    assert capsys.readouterr().out == ""
