"""The N > 1 host logic of bench.py on the CPU: two ranks on the gloo backend.

bench.py runs one replica of the workload per rank (independent batches, no collective on
the data path); the only cross-rank steps are the barriers around the timed region and
taking the slowest rank's time.  These tests drive that logic with gloo ranks in spawned
processes (no GPU), and check that the reference arm runs on rank 0 only."""
import contextlib
import io
import multiprocessing as mp
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # each rank "timed" its own replica; the slowest one (rank 1 here) decides
        my_ms = 100.0 + 25.0 * rank
        dist.barrier()
        slowest = bench.max_over_ranks(my_ms)
        value = bench.aggregate_tflops(1e12, 10, world, slowest)
        dist.barrier()
        out.put((rank, slowest, value))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    try:
        got = dict((r, (ms, v)) for r, ms, v in (out.get(timeout=120) for _ in procs))
    finally:
        for p in procs:
            p.join(timeout=60)
            if p.is_alive():
                p.kill()
    assert all(p.exitcode == 0 for p in procs)
    for r in range(2):
        ms, v = got[r]
        assert ms == 125.0
        # whole-job rate: both ranks' units over the slowest rank's time
        assert v == pytest.approx(1e12 * 10 * 2 / 0.125 / 1e12)


def test_single_process_needs_no_group():
    assert bench.max_over_ranks(42.5) == 42.5
    assert bench.aggregate_tflops(2e12, 5, 1, 1000.0) == pytest.approx(10.0)
    # weak scaling: N replicas in the same time carry N times the work
    assert bench.aggregate_tflops(2e12, 5, 4, 1000.0) == pytest.approx(40.0)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch):
    class Args:
        steps, warmup, gpus = 1, 3, 2
    monkeypatch.setenv("RANK", "1")
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        bench.run_reference(Args, bench.GQA_CAUSAL)
    assert buf.getvalue() == ""
