"""The benchmark's multi-rank host logic on CPU (gloo, world size 2).

Each rank runs its own workload (weak scaling, no collective on the data
path); the only cross-rank steps are the barriers around the timed region
and the reductions of the elapsed time (max) and of the units processed
(sum).  Those are exercised here with two gloo processes.
"""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    w, r, _ = bench.dist_env()
    dist = bench.init_dist(w, "gloo")
    bench.barrier(dist)
    ms = bench.max_over_ranks(dist, 10.0 + rank)          # rank 1 is the slowest
    units = bench.sum_over_ranks(dist, 1000.0 * (rank + 1))
    bench.barrier(dist)
    q.put((r, ms, units))
    dist.destroy_process_group()


def test_two_rank_reductions():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [o[0] for o in out] == [0, 1]
    for _, ms, units in out:
        assert ms == 11.0           # max over ranks
        assert units == 3000.0      # whole-job units: sum over ranks


def test_single_rank_needs_no_process_group(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("WORLD_SIZE", "1")
    w, r, lr = bench.dist_env()
    assert (w, r) == (1, 0)
    assert bench.init_dist(w, "gloo") is None
    assert bench.max_over_ranks(None, 3.5) == 3.5
    assert bench.sum_over_ranks(None, 7.0) == 7.0


def test_reference_arm_other_ranks_exit_without_work(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    assert bench.run_reference(type("A", (), {"steps": 1, "warmup": 3})()) is None
