"""The N > 1 path of bench.py on CPU: world_size-2 gloo process groups.

Each GPU runs an independent replica, so the only cross-rank step is the
timing reduction: every rank's times are max-reduced (the slowest rank sets
the job time) and the whole-job rate counts every rank's work.  No data-path
collective exists to test.
"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        mine = [10.0 + rank, 5.0 - rank, 7.5 * (rank + 1)]
        got = bench.reduce_max_over_ranks(mine, dist)
        rate = bench.weak_scaling_rate(units_per_rank=1e9, world=world, steps=4, max_ms=got[0])
        out[rank] = (got, rate)
    finally:
        dist.destroy_process_group()


def test_two_rank_timing_reduction_and_weak_scaling():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    for r in range(2):
        got, rate = out[r]
        assert got == [11.0, 5.0, 15.0]  # per-element max over the ranks
        assert rate == pytest.approx(2 * 1e9 * 4 / 11e-3)


def test_single_process_is_identity():
    import bench
    assert bench.reduce_max_over_ranks([1.5, 2.0]) == [1.5, 2.0]
    assert bench.weak_scaling_rate(100.0, 1, 2, 1000.0) == pytest.approx(200.0)
