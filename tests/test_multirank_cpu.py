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


_STUB = r'''
import json, os, sys
sys.path.insert(0, {root!r})
import bench
import torch.distributed as dist
rank, ws = bench.dist_setup("gloo")
bench.barrier(ws)
slowest = bench.max_over_ranks(10.0 + rank, ws)
with open(os.path.join({out!r}, f"rank{{rank}}.txt"), "w") as f:
    f.write(f"{{rank}} {{ws}} {{os.environ['LOCAL_RANK']}}")
if rank == 0:
    print(json.dumps({{"n_gpus": ws, "slowest": slowest}}), flush=True)
dist.destroy_process_group()
'''


@pytest.mark.timeout(180)
def test_bench_launches_its_own_ranks(tmp_path, capfd):
    """`bench.py --gpus N` started without torchrun launches N local ranks
    itself (bench.spawn_ranks, torch.distributed.run on 127.0.0.1): run that
    launcher with a stub workload on gloo and check that both ranks ran with
    their own RANK / LOCAL_RANK and that one JSON line came out of rank 0."""
    import json

    import bench
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    stub = tmp_path / "stub.py"
    stub.write_text(_STUB.format(root=root, out=str(tmp_path)))
    env = dict(os.environ)
    env.pop("WORLD_SIZE", None)
    rc = bench.spawn_ranks(2, str(stub), [], env=env, timeout=150)
    assert rc == 0
    seen = sorted((tmp_path / f"rank{r}.txt").read_text() for r in range(2))
    assert seen == ["0 2 0", "1 2 1"]
    lines = [ln for ln in capfd.readouterr().out.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    assert json.loads(lines[0]) == {"n_gpus": 2, "slowest": 11.0}


def test_bench_refuses_more_ranks_than_visible_gpus():
    """Asked for more GPUs than are visible, bench.py stops with a clear
    message before launching anything (this host has no GPU)."""
    import subprocess
    import sys

    import torch
    if torch.cuda.is_available():
        pytest.skip("needs a host without GPUs")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ)
    env.pop("WORLD_SIZE", None)
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--gpus", "2"],
                       capture_output=True, text=True, env=env, timeout=120)
    assert r.returncode != 0
    assert "only 0 CUDA device(s)" in r.stderr
