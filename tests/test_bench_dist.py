"""The bench's multi-process plumbing on CPU (gloo, world size 2): barrier, max over ranks,
and the reference arm running on rank 0 only.  One process per rank, as torchrun would
launch them; rendezvous on 127.0.0.1."""
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


_WORKER = r"""
import json, os, sys
sys.path.insert(0, os.environ["W4_ROOT"])
import bench
ws, rank = bench.dist_init("gloo")
bench.barrier()
m = bench.max_over_ranks(float(rank + 1))
print(json.dumps({"rank": rank, "ws": ws, "max": m}))
"""


def _launch(code_or_args, nproc=2, extra_env=None):
    port = _free_port()
    procs = []
    for r in range(nproc):
        env = dict(os.environ, RANK=str(r), LOCAL_RANK=str(r), WORLD_SIZE=str(nproc),
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), W4_ROOT=ROOT,
                   CUDA_VISIBLE_DEVICES="")
        env.update(extra_env or {})
        cmd = [sys.executable, "-c", code_or_args] if isinstance(code_or_args, str) \
            else [sys.executable] + code_or_args
        procs.append(subprocess.Popen(cmd, env=env, cwd=ROOT, stdout=subprocess.PIPE,
                                      stderr=subprocess.PIPE, text=True))
    outs = []
    for p in procs:
        out, err = p.communicate(timeout=300)
        assert p.returncode == 0, err
        outs.append(out)
    return outs


def test_max_over_ranks_and_barrier():
    outs = _launch(_WORKER)
    rows = [json.loads(o.strip().splitlines()[-1]) for o in outs]
    assert sorted(r["rank"] for r in rows) == [0, 1]
    assert all(r["ws"] == 2 and r["max"] == 2.0 for r in rows)


def test_reference_arm_prints_once_on_rank_0():
    outs = _launch(["bench.py", "--impl", "reference", "--workload", "tiny_m1_k512_n512_g128",
                    "--steps", "3", "--warmup", "1", "--gpus", "2"])
    lines = [ln for o in outs for ln in o.strip().splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0 and d["cpu_baseline"]["kind"] == "oracle"
    assert d["e2e"]["h2d_bytes_per_step"] == 0
