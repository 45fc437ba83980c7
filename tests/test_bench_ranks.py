"""The benchmark's multi-rank host logic on CPU: two processes over the gloo
backend (127.0.0.1), no GPU.  Each rank processes its own units with no
exchange; the job's step time is the slowest rank's; only rank 0 reports."""

import contextlib
import io
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world),
                      RANK=str(rank), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench

    try:
        dist.init_process_group("gloo", rank=rank, world_size=world)
        w, r, lr = bench.rank_env()
        step_ms = 1.0 + 0.5 * rank  # rank 1 is the slower one
        slowest = bench.max_over_ranks(step_ms)
        rate = bench.job_throughput(w, 8192, slowest)
        # The reference arm: rank 0 alone runs and prints; the others return.
        out = io.StringIO()
        printed = None
        if r != 0:
            with contextlib.redirect_stdout(out):
                bench.run_reference(None, r)
            printed = out.getvalue()
        dist.barrier()
        q.put((r, w, lr, slowest, rate, printed))
    finally:
        if dist.is_initialized():
            dist.destroy_process_group()


def test_two_gloo_ranks():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    results = {}
    try:
        for _ in range(world):
            r, w, lr, slowest, rate, printed = q.get(timeout=120)
            results[r] = (w, lr, slowest, rate, printed)
    finally:
        for p in procs:
            p.join(timeout=60)
            if p.is_alive():
                p.kill()
    assert all(p.exitcode == 0 for p in procs)
    for r in range(world):
        w, lr, slowest, rate, printed = results[r]
        assert (w, lr) == (world, r)
        assert slowest == 1.5  # max over ranks, the same on every rank
        assert rate == pytest.approx(2 * 8192 / 1.5e-3)
    assert results[1][4] == ""  # a non-zero rank prints nothing on the reference arm


def test_single_process_identity():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.max_over_ranks(3.25) == 3.25
    assert bench.job_throughput(1, 8192, 0.5) == pytest.approx(8192 / 0.5e-3)
