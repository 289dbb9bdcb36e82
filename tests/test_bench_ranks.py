"""bench.py's multi-rank path on the CPU (gloo, two ranks).

The path runs one independent replica per GPU. Only the barrier and the
max-over-ranks step time cross ranks, and the reference arm runs on rank 0
alone. These tests check both with two gloo ranks on 127.0.0.1, no GPU.
"""
import json
import os
import socket
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

_RANK_SCRIPT = """
import argparse, json, sys
sys.path.insert(0, {root!r})
import bench
ws, rank, _ = bench.dist_setup(argparse.Namespace(impl="reference"))
bench.barrier(ws)
print(json.dumps({{"rank": rank, "ws": ws, "max": bench.max_over_ranks(rank + 0.5, ws)}}))
"""


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _env(**kv):
    env = dict(os.environ)
    env.update({k: str(v) for k, v in kv.items()})
    return env


def test_max_over_ranks_two_gloo_ranks():
    port = _free_port()
    procs = [subprocess.Popen([sys.executable, "-c", _RANK_SCRIPT.format(root=ROOT)],
                              stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True,
                              env=_env(RANK=r, LOCAL_RANK=r, WORLD_SIZE=2,
                                       MASTER_ADDR="127.0.0.1", MASTER_PORT=port))
             for r in range(2)]
    outs = []
    for p in procs:
        out, err = p.communicate(timeout=180)
        assert p.returncode == 0, err[-2000:]
        outs.append(json.loads(out.strip().splitlines()[-1]))
    assert sorted(o["rank"] for o in outs) == [0, 1]
    assert all(o["ws"] == 2 and o["max"] == 1.5 for o in outs)


def test_reference_arm_prints_once_under_two_ranks():
    """Under torchrun the oracle arm runs on rank 0 alone: one JSON line, and
    every rank exits 0."""
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py",
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600,
                       env=_env(MASTER_ADDR="127.0.0.1"))
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [json.loads(l) for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    line = lines[0]
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0
