"""The N>1 bench path on CPU: world-size-2 gloo ranks.

The decode path shards by sequence with no data-path collective: every rank
runs an independent replica, and the only cross-rank step is the timing
reduction -- the slowest rank's time and the sum of the units processed.
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


def _worker(rank, world, port, out):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    r, w, local = bench.dist_env()
    d = bench.init_dist(w, "gloo")
    bench.barrier(d)
    t, u = bench.reduce_max_sum(d, elapsed=10.0 + 5 * r, units=100.0 * (r + 1))
    out.put((r, t, u))
    d.destroy_process_group()


def test_two_rank_reduction_takes_max_time_and_sum_of_units():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res == [(0, 15.0, 300.0), (1, 15.0, 300.0)]


def test_single_rank_needs_no_process_group():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert bench.init_dist(1, "gloo") is None
    assert bench.reduce_max_sum(None, 3.0, 7.0) == (3.0, 7.0)
