"""The replica path (one process per GPU, no data-path collective) on CPU: two gloo ranks.

Every rank times its own replica; the job is as slow as its slowest rank, so the timings are
reduced with MAX and every rank receives the result; the whole-job value counts every rank's work
over that time.  The reference arm prints from rank 0 only."""
import contextlib
import io
import os
import socket
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    torch.distributed.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        # rank r took 1+r ms for the step and 10-r ms end to end
        got = bench.max_over_ranks([1.0 + rank, 10.0 - rank], world)
        q.put((rank, got))
        torch.distributed.barrier()
    finally:
        torch.distributed.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res[0] == res[1] == [2.0, 10.0]


def test_whole_job_value_and_single_rank_passthrough():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks([3.5, 1], 1) == [3.5, 1.0]
    # 2 ranks, 1e12 ops each, slowest rank 4 ms -> 500 TOPS for the job
    assert bench.whole_job_tops(1e12, 2, 4.0) == pytest.approx(500.0)


def test_reference_arm_prints_from_rank_zero_only():
    sys.path.insert(0, ROOT)
    import bench

    class A:
        warmup, steps, gpus = 0, 0, 2
    out = io.StringIO()
    with contextlib.redirect_stdout(out):
        bench.run_reference(A(), rank=1, world=2)
    assert out.getvalue() == ""
