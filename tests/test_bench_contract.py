"""The JSON line of bench.py's reference arm (the oracle timed on the host cores), checked on CPU.

The reference arm runs without a GPU, so its line can be checked here key by key: one JSON line on
stdout, with the keys and types the bench contract fixes (throughput value and unit, step counts,
a time-like flag, scaling, the compute dtype, the workload name, the CPU baseline with its core
count and sample, and the end-to-end figure with zero host-device bytes).
"""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def reference_line():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "3"],
                       cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout[-2000:]
    return json.loads(lines[0])


def test_reference_line_has_the_contract_keys(reference_line):
    d = reference_line
    assert d["impl"] == "reference"
    assert isinstance(d["metric"], str) and d["metric"]
    assert d["value"] > 0 and d["unit"] == "GB/s"
    assert d["n_gpus"] == 1 and d["steps"] == 1 and d["warmup"] == 3
    assert d["ms_per_step"] > 0
    assert d["higher_is_better"] is True
    assert d["scaling"] in ("weak", "strong")
    assert d["vs_baseline"] is None
    assert d["dtype"] == "f64"
    assert d["data"].startswith("synthetic")
    assert isinstance(d["config"]["workload"], str) and d["config"]["workload"]
    assert "model" not in d["config"]


def test_reference_line_reports_its_cpu_baseline_and_e2e(reference_line):
    d = reference_line
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["unit"] == d["unit"]
    assert cb["value"] == d["value"]
    assert cb["cores"] >= 1 and cb["sample"]
    one = d["cpu_baseline_1core"]
    assert one["cores"] == 1 and one["value"] > 0
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0
