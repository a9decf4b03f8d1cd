"""The bench's multi-process path on CPU: world size 2 over gloo (no GPU).

Under torchrun every rank decodes its own replica (no collective on the data path); the
ranks meet only to take the maximum of their times, and rank 0 alone prints the line.
"""
import json
import os
import socket
import subprocess
import sys

import torch.multiprocessing as mp

import dist_helpers

ROOT = dist_helpers.ROOT


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_max_over_ranks_on_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    results = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=dist_helpers.max_over_ranks_worker, args=(r, 2, port, results)) for r in range(2)]
    for p in procs:
        p.start()
    got = dict(results.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert got == {0: [2.0, 5.0, 3.0], 1: [2.0, 5.0, 3.0]}


def test_job_throughput_counts_every_replica():
    sys.path.insert(0, ROOT)
    import bench
    # 2 ranks x 1 GB each in 1 ms -> 2000 GB/s for the job
    assert abs(bench.job_gbs(1e9, 2, 1.0) - 2000.0) < 1e-9
    assert bench.max_over_ranks([1.5, 2.5], 1) == [1.5, 2.5]


def test_reference_arm_under_torchrun_prints_one_line_from_rank_0():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           "bench.py", "--impl", "reference", "--config", "0", "--steps", "1", "--warmup", "0",
           "--cpu-seconds", "1"]
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle"
