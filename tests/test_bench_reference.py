"""bench.py --impl reference (the oracle timed on the host cores) prints one
JSON line with the contract's keys, for the verify workload and the prefill
GEMM; it needs no GPU."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
KEYS = {"impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
        "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline",
        "e2e"}


@pytest.mark.parametrize("workload,unit", [("q4_attn", "GB/s"), ("fp8_prefill", "TFLOP/s")])
def test_reference_arm_line(workload, unit):
    out = subprocess.run(
        [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", workload,
         "--steps", "1", "--warmup", "3", "--cpu-budget", "0.5"],
        capture_output=True, text=True, check=True, cwd=ROOT, timeout=600)
    lines = [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, out.stdout
    line = json.loads(lines[0])
    assert KEYS <= set(line), KEYS - set(line)
    assert line["impl"] == "reference" and line["unit"] == unit and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["value"] == line["value"]
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
    assert line["dtype"] == "f64" and line["higher_is_better"] is True
