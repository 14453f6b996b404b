"""bench.py's reference arm (the CPU oracle timed on a bounded sample): one JSON
line with the contract's keys, for the default workload and the routed and
PTQ1_0 ones. Under torchrun only rank 0 prints it, and every rank exits 0.
Runs on the CPU: the reference arm needs no GPU."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
KEYS = {"impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
        "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"}


def run(args, env=None, timeout=240):
    p = subprocess.run(args, cwd=ROOT, capture_output=True, text=True, timeout=timeout,
                       env={**os.environ, **(env or {})})
    assert p.returncode == 0, p.stderr[-2000:]
    return [json.loads(l) for l in p.stdout.splitlines() if l.startswith("{")]


def check_line(d, workload=None):
    assert KEYS <= set(d), KEYS - set(d)
    assert d["impl"] == "reference" and d["unit"] == "TOPS" and d["higher_is_better"] is True
    assert d["value"] > 0 and d["ms_per_step"] > 0 and d["steps"] == 1 and d["warmup"] >= 3
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    if workload:
        assert d["config"]["workload"] == workload


@pytest.mark.parametrize("workload", [None, "q4k_moe_e8_top2_m512_k4096_n14336", "ptq1_m2048_k5120_n5120"])
def test_reference_arm_line(workload):
    args = [sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "0"]
    if workload:
        args += ["--workload", workload]
    lines = run(args)
    assert len(lines) == 1
    check_line(lines[0], workload)


def test_reference_arm_under_torchrun_prints_once():
    lines = run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
                 "--master-addr", "127.0.0.1", "--master-port", "29531", "bench.py", "--impl", "reference",
                 "--gpus", "2", "--steps", "1", "--warmup", "0"])
    assert len(lines) == 1
    check_line(lines[0])
    assert lines[0]["n_gpus"] == 2
