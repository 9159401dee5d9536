"""The bench's multi-rank path on CPU: world-size-2 gloo groups on 127.0.0.1.
The data path is replicas only (no collective); the ranks meet only to time
the job by its slowest rank."""
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    torch.distributed.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dt = bench.max_over_ranks(1.0 + 0.5 * rank, world)
        q.put((rank, dt, bench.job_tokens_per_s(world, 16, 100, dt)))
    finally:
        torch.distributed.destroy_process_group()


def test_two_ranks_take_the_slowest_time():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    # both ranks see the slower rank's 1.5 s; the job processed 2 x 16 x 100 tokens
    assert [g[1] for g in got] == [1.5, 1.5]
    assert all(abs(g[2] - 2 * 16 * 100 / 1.5) < 1e-9 for g in got)


def test_single_rank_is_unchanged():
    assert bench.max_over_ranks(0.25, 1) == 0.25
    assert bench.job_tokens_per_s(1, 16, 4, 0.5) == 128.0


def test_reference_arm_runs_on_rank_zero_only():
    class Args:
        workload, steps, warmup = "m1", 1, 0

    assert bench.run_reference(Args(), 1, 2) is None
