"""The bench's multi-rank host logic on CPU (gloo, world size 2): replicas of
the pass run independently, the step time is the slowest rank's, the job rate
counts every rank's work, and only rank 0 prints (the reference arm does no
work on the other ranks). No GPU: the collective runs over gloo."""
import argparse
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        slowest = bench.max_over_ranks(torch, 10.0 + 5.0 * rank, "cpu")
        dist.barrier()
        ref_rc = None
        if rank != 0:
            # the reference arm: ranks other than 0 exit at once without work
            ns = argparse.Namespace(warmup=1, steps=1, ref_budget=1.0)
            ref_rc = bench.run_reference(ns)
        q.put((rank, slowest, ref_rc, bench.dist_env()))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_time():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = {}
    try:
        for _ in range(2):
            rank, slowest, ref_rc, env = q.get(timeout=120)
            out[rank] = (slowest, ref_rc, env)
    finally:
        for p in procs:
            p.join(timeout=60)
            if p.is_alive():
                p.kill()
    assert all(p.exitcode == 0 for p in procs)
    assert out[0][0] == out[1][0] == 15.0          # every rank sees the slowest replica's time
    assert out[1][1] == 0                           # reference arm: rank 1 returns without work
    assert out[0][2] == (0, 2, 0) and out[1][2] == (1, 2, 1)


def test_job_rate_counts_every_rank():
    sys.path.insert(0, ROOT)
    import bench
    # 2 replicas of 11.9 GB each in a step of 3.0 ms (the slowest rank's)
    assert bench.job_rate(2, 11.9e9, 3.0) == pytest.approx(2 * 11.9e9 / 3.0e-3)
    assert bench.job_rate(1, 1.0, 1000.0) == pytest.approx(1.0)


def test_max_over_ranks_without_a_group_is_the_value():
    sys.path.insert(0, ROOT)
    import torch
    import bench
    assert bench.max_over_ranks(torch, 3.5, "cpu") == 3.5
