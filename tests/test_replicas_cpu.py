"""The multi-process (replica) path of bench.py on CPU: world size 2 over
gloo, rendezvous on 127.0.0.1.  The GEMM path has no exchange step, so the
only collectives are the timing barrier and the max over ranks."""
from __future__ import annotations

import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


_WORKER = r"""
import os, sys, json
sys.path.insert(0, {root!r})
import bench
rank, world, local, dist = bench.dist_setup(world)
bench.barrier(dist)
m = bench.max_over_ranks(dist, 1.5 + rank)
print(json.dumps({{"rank": rank, "world": world, "max": m}}), flush=True)
dist.destroy_process_group()
"""


def test_barrier_and_max_over_ranks_gloo():
    port = _free_port()
    procs = []
    for rank in range(2):
        env = dict(os.environ, WORLD_SIZE="2", RANK=str(rank), LOCAL_RANK=str(rank),
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), CUDA_VISIBLE_DEVICES="")
        code = _WORKER.format(root=ROOT).replace("dist_setup(world)", "dist_setup(2)")
        procs.append(subprocess.Popen([sys.executable, "-c", code], env=env, stdout=subprocess.PIPE,
                                      stderr=subprocess.PIPE, text=True))
    outs = [p.communicate(timeout=120) for p in procs]
    for p, (out, err) in zip(procs, outs):
        assert p.returncode == 0, err[-2000:]
    got = sorted((json.loads(o.strip().splitlines()[-1]) for o, _ in outs), key=lambda d: d["rank"])
    assert [d["world"] for d in got] == [2, 2]
    assert [d["max"] for d in got] == [2.5, 2.5]   # the slower rank's time, on every rank


@pytest.mark.timeout(300)
def test_reference_arm_under_torchrun_prints_one_line():
    """bench.py --impl reference launched as 2 ranks: rank 0 alone times the
    oracle and prints the JSON line; the other rank exits 0 without work."""
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "1",
           "--workload", "ragged_197x131x77"]
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="", OMP_NUM_THREADS="2")
    r = subprocess.run(cmd, env=env, capture_output=True, text=True, timeout=280, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["kind"] == "oracle"
