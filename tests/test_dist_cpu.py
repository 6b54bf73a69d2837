"""The multi-process side of bench.py on CPU (no GPU): two `gloo` ranks agree
on the slowest rank's time, and under two ranks the reference arm is run and
printed by rank 0 alone while rank 1 exits without work."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

RANK_SCRIPT = r"""
import os, sys, json
sys.path.insert(0, os.environ["BENCH_ROOT"])
import torch
import torch.distributed as dist
import bench
dist.init_process_group("gloo")
rank = dist.get_rank()
t = bench.max_over_ranks(dist, torch, 1.5 + rank)       # rank 1 is the slower one
bench.barrier(dist, torch)
print(json.dumps({"rank": rank, "max": t}), flush=True)
dist.destroy_process_group()
"""


def _env(rank, port):
    e = dict(os.environ, MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE="2", RANK=str(rank),
             LOCAL_RANK=str(rank), BENCH_ROOT=ROOT, BENCH_BACKEND="gloo")
    return e


def _free_port():
    import socket
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_two_gloo_ranks_take_the_slowest_time():
    port = _free_port()
    procs = [subprocess.Popen([sys.executable, "-c", RANK_SCRIPT], env=_env(r, port), stdout=subprocess.PIPE,
                              stderr=subprocess.PIPE, text=True) for r in range(2)]
    outs = [p.communicate(timeout=120) for p in procs]
    for p, (o, e) in zip(procs, outs):
        assert p.returncode == 0, e
    got = sorted(json.loads(o.strip().splitlines()[-1])["max"] for o, _ in outs)
    assert got == [2.5, 2.5]


def test_reference_arm_prints_on_rank_zero_only():
    pytest.importorskip("torch")
    port = _free_port()
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--config", "tiny", "--steps", "2",
           "--warmup", "1"]
    procs = [subprocess.Popen(cmd, env=_env(r, port), stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True,
                              cwd=ROOT) for r in range(2)]
    outs = [p.communicate(timeout=300) for p in procs]
    for p, (o, e) in zip(procs, outs):
        assert p.returncode == 0, e
    line = json.loads(outs[0][0].strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0 and line["n_gpus"] == 2
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert outs[1][0].strip() == ""
