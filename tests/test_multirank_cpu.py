"""The benchmark's multi-rank plumbing on CPU (gloo, world size 2).

The KDA core shards by (sequence, head) with no exchange, so with N ranks
each rank runs its own copy of the workload and the only cross-rank traffic
is the timing barrier and the max-reduction of the timed region.  This test
runs those helpers in two spawned processes.
"""
import multiprocessing as mp
import os
import socket

import pytest


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist

    import bench
    r, ws = bench.dist_setup("gloo")
    times = {0: 12.5, 1: 20.0}
    slowest = bench.max_over_ranks(times[r], ws)
    bench.barrier(ws)
    out.put((r, ws, slowest))
    dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_two_rank_barrier_and_max_reduction():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    results = sorted(out.get(timeout=90) for _ in procs)
    for p in procs:
        p.join(timeout=30)
        assert p.exitcode == 0
    assert results == [(0, 2, 20.0), (1, 2, 20.0)]


def test_single_rank_needs_no_process_group():
    import bench
    os.environ.pop("WORLD_SIZE", None)
    r, ws = bench.dist_setup("gloo")
    assert (r, ws) == (0, 1)
    assert bench.max_over_ranks(3.5, ws) == 3.5
    bench.barrier(ws)  # no-op
