"""bench.py's multi-process path on the CPU: gloo ranks, world size 2.

The operation shards into independent problems, so N GPUs run N replicas and
the only communication is a host barrier plus the maximum of the per-rank
timings.  These tests run that logic as real processes over gloo, without a GPU.
"""
import json
import os
import socket
import subprocess
import sys

import pytest

torch = pytest.importorskip("torch")

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port),
                      WORLD_SIZE=str(world), RANK=str(rank), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    ws, r, local = bench.dist_env()
    sync = bench.RankSync.create(ws)
    sync()                                   # plain barrier
    secs = sync(0.5 + rank)                  # each rank's timing; max comes back
    value = bench.whole_job_value(100.0, ws, secs)
    sync.close()
    out.put((r, local, secs, value))


def test_rank_sync_takes_the_max_over_two_gloo_ranks():
    ctx = torch.multiprocessing.get_context("spawn")
    q = ctx.Queue()
    port = free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r for r, *_ in results] == [0, 1]
    assert [l for _, l, *_ in results] == [0, 1]
    # both ranks see the slower rank's time; value counts both ranks' units
    assert all(secs == 1.5 for _, _, secs, _ in results)
    assert all(abs(v - 200.0 / 1.5) < 1e-9 for *_, v in results)


def test_rank_sync_single_rank_is_a_no_op():
    sys.path.insert(0, ROOT)
    import bench
    sync = bench.RankSync.create(1)
    assert sync() is None
    assert sync(0.25) == 0.25
    sync.close()
    assert bench.whole_job_value(10.0, 1, 2.0) == 5.0


def test_reference_arm_under_torchrun_prints_one_line_from_rank_0():
    port = free_port()
    env = dict(os.environ, OMP_NUM_THREADS="2")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port),
           "bench.py", "--impl", "reference", "--gpus", "2", "--steps", "2", "--warmup", "3",
           "--workload", "tiny_8x1024x1024", "--reference-budget", "2"]
    res = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [l for l in res.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, res.stdout
    out = json.loads(lines[0])
    assert out["impl"] == "reference"
    assert out["n_gpus"] == 2 and out["steps"] == 2 and out["warmup"] == 3
    assert out["value"] > 0 and out["unit"] == "GB/s"
    assert out["e2e"]["value"] == out["value"]
    assert out["cpu_baseline"]["kind"] == "oracle"
