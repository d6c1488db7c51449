"""The benchmark's reference arm (the oracle timed on the host cores) keeps the JSON-line
contract on the CPU: one line with the same metric, unit and config keys as the CUDA arm
of the same workload, and the cpu_baseline / e2e objects describing the run."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
KEYS = {"impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
        "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
        "cpu_baseline", "e2e"}


def _reference_line(workload):
    p = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", workload,
                        "--steps", "3", "--warmup", "3"], cwd=ROOT, capture_output=True, text=True,
                       timeout=600)
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [ln for ln in p.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, p.stdout[-2000:]
    return json.loads(lines[0])


@pytest.mark.parametrize("workload,unit,config_keys", [
    ("tiny_sliding", "steps/s", {"workload", "batch", "hidden", "heads", "head_dim", "context"}),
    ("verify_l16_8k", "blocks/s", {"workload", "tokens", "prior"}),
])
def test_reference_arm_prints_one_contract_line(workload, unit, config_keys):
    d = _reference_line(workload)
    assert KEYS <= set(d), KEYS - set(d)
    assert d["impl"] == "reference" and d["unit"] == unit and d["dtype"] == "f64"
    assert d["steps"] == 3 and d["warmup"] == 3 and d["higher_is_better"] is True
    assert d["value"] > 0 and abs(d["ms_per_step"] * d["value"] - 1e3) < 1e-6 * 1e3
    assert config_keys <= set(d["config"]) and d["config"]["workload"] == workload
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["unit"] == unit
    assert cb["cores"] >= 1 and workload in cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": unit, "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
