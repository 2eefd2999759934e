"""bench.py's reference arm (the oracle on the host cores) keeps the one-line
JSON contract, alone and under torch.distributed.run with two ranks (rank 0
prints, the other rank exits without work). CPU only."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def run(cmd, timeout=300):
    env = dict(os.environ, OMP_NUM_THREADS="1", CUDA_VISIBLE_DEVICES="")
    p = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=timeout)
    assert p.returncode == 0, p.stderr[-2000:]
    return [json.loads(l) for l in p.stdout.splitlines() if l.startswith("{")]


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def check_line(j, steps, warmup):
    assert j["impl"] == "reference"
    assert j["unit"] == "tokens/s" and j["higher_is_better"] is True
    assert j["value"] > 0 and j["steps"] == steps and j["warmup"] == warmup
    assert j["metric"] and j["config"]["workload"].startswith("batch-1 decode")
    cb = j["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == j["value"]
    assert str(steps) in cb["sample"]
    e2e = j["e2e"]
    assert e2e["value"] == j["value"] and e2e["unit"] == j["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0
    # ms_per_step is one 40-layer step
    assert j["ms_per_step"] == pytest.approx(1e3 / j["value"], rel=1e-3)


def test_reference_arm_prints_one_json_line():
    lines = run([sys.executable, "bench.py", "--impl", "reference", "--steps", "2", "--warmup", "1"])
    assert len(lines) == 1
    check_line(lines[0], 2, 1)


def test_reference_arm_under_two_ranks_prints_once():
    lines = run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
                 "--master-addr", "127.0.0.1", "--master-port", str(free_port()), "bench.py",
                 "--impl", "reference", "--gpus", "2", "--steps", "2", "--warmup", "1"])
    assert len(lines) == 1
    check_line(lines[0], 2, 1)
