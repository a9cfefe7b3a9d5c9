"""`bench.py --mode fwd` (the forward without tangents) prints one JSON line
with the bench contract's keys, on a small specified workload."""

import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.parametrize("workload", ["f16_b2h8n512d64_causal", "bf16_b2h8n1024d64_additive"])
def test_bench_fwd_mode_prints_one_contract_line(workload):
    out = subprocess.run([sys.executable, "bench.py", "--mode", "fwd", "--workload", workload,
                          "--steps", "3", "--warmup", "3", "--no-cpu-baseline"],
                         cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    r = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "dtype", "data", "config", "roofline", "clocks",
                "gpu_launches"):
        assert key in r, key
    assert r["mode"] == "fwd" and r["config"]["workload"] == workload
    assert r["value"] > 0 and r["ms_per_step"] > 0 and r["gpu_launches"] == 3
    assert r["roofline"]["bound"] == "tensor" and 0 < r["roofline"]["frac"] < 1.2
