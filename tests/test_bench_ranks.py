"""The benchmark's multi-rank logic on CPU: two gloo ranks, each with its own
batch, the job time is the slowest rank's and the job value counts the steps
of every rank.  No data-path collective exists, so this is all N > 1 adds."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    import torch
    import torch.distributed as dist
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = 10.0 + 5.0 * rank  # rank 1 is the slow one
        job_ms = bench.max_over_ranks(ms, torch.device("cpu"))
        q.put((rank, bench.rank_seed(rank), job_ms, bench.job_value(world, 100, job_ms)))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, s0, t0, v0), (r1, s1, t1, v1) = res
    assert s0 != s1  # independent batches
    assert t0 == t1 == 15.0  # the slowest rank's time
    assert v0 == v1 == pytest.approx(2 * 100 / 0.015)


def test_single_process_needs_no_group():
    import torch
    import bench
    assert bench.max_over_ranks(12.5, torch.device("cpu")) == 12.5
    assert bench.job_value(1, 10, 10.0) == pytest.approx(1000.0)
