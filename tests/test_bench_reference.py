"""The reference arm of bench.py (the float64 oracle timed on the host cores)
prints exactly one JSON line carrying the bench contract's keys.

Runs on the CPU: the reference arm needs no GPU.  The smaller causal sink
workload (16K queries, one KV head) and a 3-second oracle budget keep it to
well under a minute.
"""

import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

KEYS = ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
        "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e")


def test_reference_arm_prints_one_contract_line():
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", "causal_sink_16k_1kv",
           "--steps", "1", "--warmup", "3", "--ref-budget", "3"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout[-2000:]
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    for k in KEYS:
        assert k in d, k
    assert d["unit"] == "TFLOP/s" and d["higher_is_better"] is True and d["n_gpus"] == 1
    assert d["steps"] == 1 and d["warmup"] == 3 and d["dtype"] == "f64"
    assert d["value"] > 0 and d["ms_per_step"] > 0
    assert d["config"]["workload"] == "causal_sink_16k_1kv"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1 and cb["sample"]
    assert isinstance(cb["cpu_model"], str) and cb["cpu_model"]
    # the same config dict as the library's arm prints for this workload
    sys.path.insert(0, ROOT)
    import bench
    assert d["config"] == bench.workload_config(bench.WORKLOADS["causal_sink_16k_1kv"])
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0
