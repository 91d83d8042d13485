"""The multi-process (replicas) path of bench.py on CPU: the max-over-ranks
timing and the job throughput with two gloo ranks, and the reference arm
under the torch.distributed launcher (rank 0 prints one line, the other rank
exits without work). No GPU."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, results):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = [3.5, 7.25][rank]
        results[rank] = bench.max_over_ranks(ms, dist, "cpu")
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_with_two_gloo_ranks():
    import torch.multiprocessing as mp
    mgr = mp.get_context("spawn").Manager()
    results = mgr.dict()
    mp.spawn(_rank_main, args=(2, _free_port(), results), nprocs=2, join=True)
    assert dict(results) == {0: 7.25, 1: 7.25}


def test_max_over_ranks_without_process_group_and_job_throughput():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(2.5, None, "cpu") == 2.5
    # 2 ranks x 1000 calls bounded by the slowest rank's 20 ms
    assert bench.job_calls_per_s(2, 1000, 20.0) == pytest.approx(100000.0)


def test_reference_arm_under_the_launcher_two_ranks():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2", "--steps", "1",
           "--warmup", "3", "--config", "tiny"]
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1")
    p = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [l for l in p.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, p.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["unit"] == "us/call"
    assert d["value"] > 0 and d["cpu_baseline"]["kind"] == "oracle"
