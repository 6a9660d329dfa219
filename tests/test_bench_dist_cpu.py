"""Multi-rank host logic of bench.py on CPU (gloo, world size 2).

The convolution path shards into independent replicas, so the only
cross-rank work is host-side: the max of the timed region over ranks and the
whole-job throughput derived from it, plus the reference arm's rule that rank
0 alone runs and prints.  No GPU is involved.
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank), BENCH_DIST_BACKEND="gloo")
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist
    w, r, _ = bench.dist_setup()
    assert (w, r) == (world, rank)
    try:
        got_max = bench.dist_max(1.5 + rank, world, "cpu")
        # Rank 1 is the slow one: 4 steps of 3 ms against rank 0's 4 x 2 ms.
        step_ms = [2.0 + rank] * 4
        ms, value = bench.whole_job_value(step_ms, 6e9, world, "cpu")
        bench.dist_barrier(world)
        out.put((rank, got_max, ms, value))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_value():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(world))
    for rank, got_max, ms, value in res:
        assert got_max == 2.5
        assert ms == pytest.approx(3.0)                # the slowest rank's step time
        # 2 replicas x 4 steps x 6 GFLOP in 12 ms = 4 TFLOP/s
        assert value == pytest.approx(2 * 4 * 6e9 / 12e-3 / 1e12)


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.dist_max(3.25, 1, "cpu") == 3.25
    ms, value = bench.whole_job_value([1.0, 3.0], 1e9, 1, "cpu")
    assert ms == pytest.approx(2.0)
    assert value == pytest.approx(2e9 / 4e-3 / 1e12)


def test_reference_arm_prints_once_under_torchrun(tmp_path):
    env = dict(os.environ, BENCH_DIST_BACKEND="gloo", PYTHONPATH=ROOT)
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
           "--steps", "1", "--warmup", "3", "--workload", "tiny_bf16"]
    proc = subprocess.run(cmd, cwd=str(tmp_path), env=env, capture_output=True, text=True,
                          timeout=600)
    assert proc.returncode == 0, proc.stderr[-2000:]
    lines = [l for l in proc.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, proc.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2
    assert line["value"] > 0 and line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0
