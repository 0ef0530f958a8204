"""The benchmark's multi-rank host logic on CPU: two gloo ranks, no GPU.

Each rank runs the same per-GPU workload (replicas, weak scaling).  The job's
time is the slowest rank's, every rank must agree on it, and the reported
value is the units of all ranks over that time.
"""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = [3.0, 5.0][rank]                # rank 1 is the slow one
    bench.barrier(world)
    total = bench.max_over_ranks(ms, world)
    rate = bench.whole_job_rate(1000.0, world, total)
    out.put((rank, total, rate))
    bench.barrier(world)
    dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_slowest_time_and_whole_job_rate():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(out.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, total, rate in res:
        assert total == pytest.approx(5.0)
        assert rate == pytest.approx(2 * 1000.0 / 5e-3)


def test_single_rank_is_identity():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(7.5, 1) == 7.5
    assert bench.whole_job_rate(10.0, 1, 2.0) == pytest.approx(5000.0)
