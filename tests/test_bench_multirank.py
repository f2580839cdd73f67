"""The benchmark's multi-rank path on the CPU, with world size 2 over gloo.

The path is "replicas only": each rank runs its own problem and the one
collective is the maximum of the timings over ranks (the job's time is its
slowest rank's).  These tests run that collective as two processes over
gloo, check the whole-job throughput formula, and launch the reference arm
under torch.distributed.run with two processes (rank 0 alone prints one JSON
line; both exit 0).
"""
import json
import os
import socket
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402

_RANK_SCRIPT = """
import os, sys
sys.path.insert(0, {root!r})
import torch.distributed as dist
import bench
dist.init_process_group("gloo", init_method="env://")
rank = dist.get_rank()
print("RESULT", rank, bench.max_over_ranks(10.0 + 5.0 * rank, device="cpu"), flush=True)
dist.destroy_process_group()
"""


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_max_over_ranks_two_gloo_ranks():
    port = _free_port()
    procs = []
    for rank in range(2):
        env = dict(os.environ, RANK=str(rank), WORLD_SIZE="2", LOCAL_RANK=str(rank),
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
        procs.append(subprocess.Popen([sys.executable, "-c", _RANK_SCRIPT.format(root=ROOT)], env=env,
                                      stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True))
    results = {}
    for p in procs:
        out, err = p.communicate(timeout=120)
        assert p.returncode == 0, err[-2000:]
        for line in out.splitlines():
            if line.startswith("RESULT"):
                _, rank, value = line.split()
                results[int(rank)] = float(value)
    assert results == {0: 15.0, 1: 15.0}


def test_max_over_ranks_single_process():
    assert bench.max_over_ranks(3.25, device="cpu") == 3.25


def test_job_throughput_counts_every_rank():
    # 2 ranks x 32768 tokens in a 0.5 ms step of the slowest rank
    assert bench.job_tokens_per_s(32768, 2, 0.5) == 2 * 32768 / 0.5e-3


def test_reference_arm_under_torchrun_two_ranks():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes", "1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--workload", "tiny_fp32", "--steps", "1", "--warmup", "1",
           "--cpu-pairs", "2"]
    out = subprocess.run(cmd, capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0
