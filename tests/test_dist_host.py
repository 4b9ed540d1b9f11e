"""The multi-process plumbing of bench.py on the CPU: two `gloo` ranks.

On one GPU the path has no data-path collective (each GPU runs a full replica
with the ranks emulated in its memory); the process group only carries the
barrier around the timed region and the maximum of the step time over ranks,
and under torchrun only rank 0 runs the CPU reference arm."""
import argparse
import contextlib
import io
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    w, r, _ = bench.dist_env()
    dist = bench.init_dist(w, "gloo")
    try:
        got = bench.max_over_ranks(dist, 1.5 * (r + 1))   # rank 0: 1.5, rank 1: 3.0
        dist.barrier()
        q.put((r, w, got))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_barrier_and_max_over_ranks():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    results = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert results == [(0, 2, 3.0), (1, 2, 3.0)]


def test_reference_arm_runs_on_rank_zero_only(monkeypatch):
    """A non-zero rank of `bench.py --impl reference` exits 0 without work or output."""
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    out = io.StringIO()
    with contextlib.redirect_stdout(out):
        rc = bench.run_reference(argparse.Namespace(gpus=2, steps=1, warmup=0))
    assert rc == 0 and out.getvalue() == ""


def test_single_process_needs_no_process_group():
    import bench
    assert bench.init_dist(1, "gloo") is None
    assert bench.max_over_ranks(None, 2.5) == 2.5
