"""The benchmark's multi-process path on CPU (gloo, world size 2): the
reference arm runs on rank 0 only and prints one JSON line; other ranks exit
0 without work; the max-over-ranks helper returns the largest value."""
import json
import os
import re
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _torchrun(args, timeout=600):
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(_port())] + args
    env = dict(os.environ, OMP_NUM_THREADS="2")
    return subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=timeout, env=env)


def test_dist_max_over_ranks_gloo(tmp_path):
    script = tmp_path / "m.py"
    script.write_text(
        "import os, sys, json\n"
        f"sys.path.insert(0, {ROOT!r})\n"
        "import bench\n"
        "d = bench.Dist(2)\n"
        "v = d.max(1.5 + d.rank)\n"
        "d.barrier()\n"
        "print(json.dumps({'rank': d.rank, 'max': v}), flush=True)\n"
        "d.close()\n")
    r = _torchrun([str(script)])
    assert r.returncode == 0, r.stderr[-2000:]
    # the two ranks share stdout, so their lines may interleave
    vals = [json.loads(m) for m in re.findall(r"\{[^{}]*\}", r.stdout)]
    assert sorted(v["rank"] for v in vals) == [0, 1]
    assert all(v["max"] == 2.5 for v in vals)


@pytest.mark.slow
def test_reference_arm_prints_one_line_from_rank0():
    r = _torchrun(["bench.py", "--impl", "reference", "--gpus", "2", "--steps", "1",
                   "--warmup", "0", "--ref-sample", "2"], timeout=900)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0 and d["cpu_baseline"]["kind"] == "oracle"
    assert d["e2e"]["h2d_bytes_per_step"] == 0
