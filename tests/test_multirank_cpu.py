"""The benchmark's multi-rank host logic on CPU: two gloo ranks (one process each), as torchrun would
start them on two GPUs.  The path runs replicas with no exchange on the data path; what the ranks
share is the timing: the job's time is the slowest rank's, and the job's rate counts every rank's work."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
torch = pytest.importorskip("torch")


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


_CHILD = r"""
import json, os, sys
sys.path.insert(0, os.environ["ROOT"])
import torch
import bench
rank, world = int(os.environ["RANK"]), int(os.environ["WORLD_SIZE"])
torch.distributed.init_process_group("gloo", init_method="tcp://127.0.0.1:%s" % os.environ["PORT"], rank=rank,
                                     world_size=world)
local_ms = [3.0, 5.0][rank]  # rank 1 is the slow one
slowest = bench.max_over_ranks(local_ms, torch.device("cpu"))
torch.distributed.barrier()
print(json.dumps({"rank": rank, "max": slowest, "rate": bench.job_rate(world, 2e9, slowest)}))
torch.distributed.destroy_process_group()
"""


def test_two_ranks_agree_on_the_slowest_time():
    port = str(_free_port())
    procs = []
    for rank in range(2):
        env = dict(os.environ, ROOT=ROOT, RANK=str(rank), WORLD_SIZE="2", PORT=port, MASTER_ADDR="127.0.0.1",
                   CUDA_VISIBLE_DEVICES="")
        procs.append(subprocess.Popen([sys.executable, "-c", _CHILD], env=env, stdout=subprocess.PIPE,
                                      stderr=subprocess.PIPE, text=True))
    outs = []
    for p in procs:
        out, err = p.communicate(timeout=120)
        assert p.returncode == 0, err
        outs.append(json.loads(out.strip().splitlines()[-1]))
    for o in outs:
        assert o["max"] == 5.0
        # 2 ranks x 2 GFLOP in 5 ms: 0.8 TFLOP/s for the whole job
        assert abs(o["rate"] - 0.8) < 1e-12


def test_single_process_needs_no_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(7.5) == 7.5
    assert abs(bench.job_rate(1, 1e12, 1000.0) - 1.0) < 1e-12


def test_reference_arm_prints_only_on_rank_zero():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1", CUDA_VISIBLE_DEVICES="")
    p = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "1"], env=env, capture_output=True, text=True, timeout=120)
    assert p.returncode == 0, p.stderr
    assert p.stdout.strip() == ""
