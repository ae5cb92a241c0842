"""The bench's multi-process plumbing on CPU (gloo, world size 2): timing is
the max over ranks, and the reference arm prints on rank 0 only."""
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


CHILD = r"""
import os, sys, json
sys.path.insert(0, {root!r})
import bench
ws, rank = bench.dist_init(use_cuda=False)
assert ws == 2
v = bench.max_over_ranks(10.0 + rank)
bench.barrier()
print(json.dumps({{"rank": rank, "max": v}}), flush=True)
"""


def _launch(code, world=2):
    port = _free_port()
    procs = []
    for r in range(world):
        env = dict(os.environ, WORLD_SIZE=str(world), RANK=str(r), LOCAL_RANK=str(r),
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
        procs.append(subprocess.Popen([sys.executable, "-c", code], env=env, stdout=subprocess.PIPE,
                                      stderr=subprocess.PIPE, text=True))
    outs = []
    for p in procs:
        o, e = p.communicate(timeout=180)
        assert p.returncode == 0, e
        outs.append(o)
    return outs


def test_max_over_ranks_gloo():
    outs = _launch(CHILD.format(root=ROOT))
    for o in outs:
        d = json.loads(o.strip().splitlines()[-1])
        assert d["max"] == 11.0


def test_reference_arm_prints_on_rank0_only():
    code = (f"import sys; sys.path.insert(0, {ROOT!r}); import bench; "
            "bench.main(['--impl', 'reference', '--steps', '1', '--warmup', '0', '--workload', 'tiny_nvfp4'])")
    outs = _launch(code)
    lines0 = [l for l in outs[0].splitlines() if l.startswith("{")]
    lines1 = [l for l in outs[1].splitlines() if l.startswith("{")]
    assert len(lines0) == 1 and not lines1
    d = json.loads(lines0[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0
