"""The benchmark's reference arm on the host (no GPU): the oracle timed on the
host cores prints one JSON line with the keys the benchmark line carries, and
under a two-rank launch only rank 0 prints while the other rank exits at once.
"""
import json
import os
import socket
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _lines(cmd):
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    return [json.loads(l) for l in r.stdout.splitlines() if l.startswith("{")]


def _check(line, n_gpus):
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e", "gpu_launches"):
        assert k in line, k
    assert line["impl"] == "reference" and line["n_gpus"] == n_gpus and line["steps"] == 1
    assert line["value"] > 0 and line["unit"] == "GB/s" and line["higher_is_better"] is True
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["cpu_baseline"]["value"] == line["value"] == line["e2e"]["value"]
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["gpu_launches"] == 0
    assert "workload" in line["config"]


def test_reference_arm_one_process(built_lib):
    lines = _lines([sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "3"])
    assert len(lines) == 1
    _check(lines[0], 1)


def test_reference_arm_two_ranks_print_once(built_lib):
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    lines = _lines([sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
                    "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl", "reference",
                    "--gpus", "2", "--steps", "1", "--warmup", "3"])
    assert len(lines) == 1
    _check(lines[0], 2)
