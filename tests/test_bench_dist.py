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


def test_reference_arm_prints_the_contract_line():
    """`bench.py --impl reference` (the oracle on the host cores) prints one JSON
    line with the metric, the reference tag, its CPU baseline and a host-only e2e."""
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference", "--config", "tiny",
                        "--steps", "3", "--warmup", "1"], capture_output=True, text=True, timeout=600, cwd=root)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["metric"] == "decode steps/s" and line["unit"] == "steps/s"
    assert line["value"] > 0 and line["steps"] == 3 and line["higher_is_better"] is True
    assert line["config"]["workload"] == "tiny"
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == line["value"] and cb["sample"]
    assert line["e2e"] == {"value": line["value"], "unit": "steps/s", "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}


def test_bench_names_the_scoring_kernel_the_library_picks():
    """bench.py reports which fm_score kernel a workload runs; its threshold is the
    library's (the tensor-core kernel from kTcMinChunks chunks per call)."""
    import re
    import bench
    from srh_workload import configs as C
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    txt = open(os.path.join(root, "sparse_retrieval_host_gb300", "csrc", "srh_internal.cuh")).read()
    m = re.search(r"kTcMinChunks\s*=\s*1LL\s*<<\s*(\d+)", txt)
    assert m and bench.TC_SCORE_MIN_CHUNKS == 1 << int(m.group(1))
    assert "mma.sync" in bench.scoring_kernel(C.CTX8K) and "mma.sync" in bench.scoring_kernel(C.CTX256K)
    assert "tcgen05" in bench.scoring_kernel(C.CTX1M) and "tcgen05" in bench.scoring_kernel(C.batch_sweep(16))
