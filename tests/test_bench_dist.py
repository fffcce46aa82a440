"""The benchmark's multi-rank aggregation (max of time, sum of steps) over a
world of 2 gloo ranks on the CPU."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank), SRH_DIST_BACKEND="gloo")
    import bench
    dist, r, w, _ = bench.dist_setup(world)
    secs, steps = bench.aggregate(dist, 1.0 + rank, 10 * (rank + 1))
    q.put((r, w, secs, steps))
    dist.destroy_process_group()


def test_aggregate_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    assert [g[:2] for g in got] == [(0, 2), (1, 2)]
    for _, _, secs, steps in got:
        assert secs == 2.0 and steps == 30


def test_single_process_aggregate_is_identity():
    import bench
    assert bench.aggregate(None, 3.5, 7) == (3.5, 7)
