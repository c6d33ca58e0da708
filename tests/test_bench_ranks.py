"""The multi-rank path of bench.py on CPU: two gloo ranks (replicas, no data-path collective).

Each rank reports its own step time; the job's time is the slowest rank's (an all-reduce
MAX) and its value counts every rank's nodes.  Under torchrun the reference arm runs on
rank 0 only: the other ranks return at once and print nothing.
"""
import io
import os
import socket
import contextlib

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, times, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dist.barrier()
        total = bench.max_over_ranks(times[rank], world, "cpu")
        out.put((rank, total, bench.job_value(256, world, total, 10)))
    finally:
        dist.destroy_process_group()


def test_two_ranks_take_the_slowest_time_and_count_all_nodes():
    ctx = mp.get_context("spawn")
    q = ctx.SimpleQueue()
    times = [0.61, 0.73]
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, times, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get() for _ in range(2))
    for rank, total, value in got:
        assert total == pytest.approx(0.73)
        assert value == pytest.approx(256 * 2 / (0.73 / 10 * 1e-3))


def test_one_rank_needs_no_process_group():
    assert bench.max_over_ranks(1.5, 1, "cpu") == 1.5
    assert bench.job_value(100, 1, 20.0, 10) == pytest.approx(100 / 2e-3)


def test_reference_arm_runs_on_rank_zero_only():
    class Args:
        config, warmup, steps, ref_heads = 1, 3, 1, 0
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        assert bench.run_reference(Args(), rank=1, world=2) is None
    assert buf.getvalue() == ""
