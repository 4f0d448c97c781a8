"""The bench's multi-rank host logic on CPU: two gloo ranks.

With N ranks every rank runs its own replica of the step (weak scaling, no
collective on the data path); the step time is the slowest rank's, and the
job's throughput counts the bytes of all ranks.  The reference arm runs on
rank 0 only; the other ranks return without work or output.
"""
import argparse
import contextlib
import io
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402

WORLD = 2
STEP_MS = [1.25, 3.5]  # rank 1 is the slow one
BYTES_PER_RANK = 99_090_432


def free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def rank_main(rank, port, out):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=WORLD)
    try:
        dist.barrier()
        ms = bench.max_over_ranks(STEP_MS[rank], dist, "cpu")
        out[rank] = (ms, bench.job_gbs(BYTES_PER_RANK, WORLD, ms))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_ranks_agree_on_the_slowest_step():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        mp.start_processes(rank_main, args=(free_port(), out), nprocs=WORLD, join=True,
                           start_method="spawn")
        res = dict(out)
    want_ms = max(STEP_MS)
    want_gbs = BYTES_PER_RANK * WORLD / (want_ms * 1e-3) / 1e9
    for rank in range(WORLD):
        ms, gbs = res[rank]
        assert ms == want_ms
        assert gbs == pytest.approx(want_gbs, rel=1e-12)


def test_one_rank_needs_no_process_group():
    assert bench.max_over_ranks(2.5, None, "cpu") == 2.5
    assert bench.job_gbs(10**9, 1, 1000.0) == pytest.approx(1.0)


def test_reference_arm_runs_on_rank_zero_only():
    args = argparse.Namespace(steps=3, warmup=3, gpus=2)
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        bench.run_reference(args, rank=1, world=2)
    assert buf.getvalue() == ""
