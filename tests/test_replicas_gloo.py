"""The multi-process path of bench.py on CPU (gloo, world size 2).

The decode-pool path shards into independent replicas (requests, pools and
tags are per GPU; nothing on the data path is exchanged), so the N > 1 path is
only the process-group plumbing: rendezvous, barrier, max over ranks of the
timed region, per-rank workload seeds, and rank-0-only output of the CPU
reference arm.  These run here as two CPU processes with the GPU hidden.
"""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

_PLUMBING = r"""
import json, sys
sys.path.insert(0, {root!r})
import bench
rank, world, local = bench.dist_setup(2)
m = bench.max_over_ranks(1.5 + rank, world)
bench.barrier(world)
from workloads import WORKLOADS
wl = WORKLOADS["tiny"](seed=100 + rank)
import torch.distributed as dist
print(json.dumps({{"rank": rank, "world": world, "backend": dist.get_backend(),
                   "max": m, "q0": int(wl.q.reshape(-1)[:64].astype("int64").sum())}}))
dist.destroy_process_group()
"""


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _run_two(cmd_for_rank, timeout=300):
    port = _free_port()
    procs = []
    for r in range(2):
        env = dict(os.environ, CUDA_VISIBLE_DEVICES="", MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port),
                   WORLD_SIZE="2", RANK=str(r), LOCAL_RANK=str(r))
        procs.append(subprocess.Popen(cmd_for_rank(r), cwd=ROOT, env=env, stdout=subprocess.PIPE,
                                      stderr=subprocess.PIPE, text=True))
    outs = []
    for p in procs:
        try:
            out, err = p.communicate(timeout=timeout)
        except subprocess.TimeoutExpired:
            for q in procs:
                q.kill()
            raise
        outs.append((p.returncode, out, err))
    return outs


def test_rendezvous_barrier_and_max_over_ranks():
    code = _PLUMBING.format(root=ROOT)
    outs = _run_two(lambda r: [sys.executable, "-c", code])
    lines = []
    for rc, out, err in outs:
        assert rc == 0, err[-2000:]
        lines.append(json.loads(out.strip().splitlines()[-1]))
    lines.sort(key=lambda d: d["rank"])
    assert [d["world"] for d in lines] == [2, 2]
    assert all(d["backend"] == "gloo" for d in lines)
    assert all(d["max"] == 2.5 for d in lines)          # max over ranks of 1.5 + rank
    assert lines[0]["q0"] != lines[1]["q0"]              # replicas draw their own requests


@pytest.mark.timeout(600)
def test_reference_arm_prints_once_from_rank_zero():
    outs = _run_two(lambda r: [sys.executable, "bench.py", "--impl", "reference", "--gpus", "2",
                               "--steps", "2", "--warmup", "1", "--workload", "tiny"], timeout=600)
    (rc0, out0, err0), (rc1, out1, err1) = outs
    assert rc0 == 0, err0[-2000:]
    assert rc1 == 0, err1[-2000:]
    line = json.loads(out0.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert out1.strip() == ""
