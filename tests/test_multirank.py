"""The bench's multi-rank path on CPU: world size 2 over gloo, rendezvous on 127.0.0.1.

The forward scan shards by (batch, head) with no exchange, so N GPUs run N replicas; what
crosses ranks is the timing (the job's time is the slowest rank's, a MAX all-reduce) and the
reporting (rank 0 alone prints; the whole-job rate counts every rank's tokens).  These tests
run that host logic in two real processes; the reference arm is launched under torchrun.
"""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

WORKER = r"""
import json, os, sys
sys.path.insert(0, os.environ["REPO_ROOT"])
import torch.distributed as dist
import bench
dist.init_process_group("gloo", rank=int(os.environ["RANK"]), world_size=int(os.environ["WORLD_SIZE"]))
rank, ws = dist.get_rank(), dist.get_world_size()
ms = bench.max_over_ranks(10.0 + 5.0 * rank, ws, dist, "cpu")   # rank 1 is the slow one
rate = bench.job_rate(1000, ws, ms)
dist.barrier()
dist.destroy_process_group()
print(json.dumps({"rank": rank, "ms": ms, "rate": rate}))
"""


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_job_time_is_the_slowest_rank_and_rate_counts_all_ranks():
    port = _free_port()
    procs = []
    for rank in range(2):
        env = dict(os.environ, MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                   WORLD_SIZE="2", LOCAL_RANK=str(rank), REPO_ROOT=ROOT)
        procs.append(subprocess.Popen([sys.executable, "-c", WORKER], env=env, stdout=subprocess.PIPE,
                                      stderr=subprocess.PIPE, text=True))
    outs = []
    for p in procs:
        out, err = p.communicate(timeout=180)
        assert p.returncode == 0, err
        outs.append(json.loads(out.strip().splitlines()[-1]))
    for o in outs:
        assert o["ms"] == 15.0
        assert o["rate"] == pytest.approx(2 * 1000 / 15e-3)


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.max_over_ranks(3.5, 1, None, "cpu") == 3.5
    assert bench.job_rate(500, 1, 2.0) == pytest.approx(250000.0)


def test_reference_arm_under_torchrun_prints_once_from_rank_0():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--workload", "tiny_fp32", "--steps", "1", "--warmup", "0",
           "--cpu-seconds", "0.2"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle"
