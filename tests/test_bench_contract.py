"""bench.py's reference arm runs on the host cores (the fp64 oracle), so its
JSON line can be checked here: one line, the keys the benchmark contract
names, and values consistent with one another."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench(*args, timeout=300):
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT, capture_output=True,
                       text=True, timeout=timeout)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    return json.loads(lines[0])


def test_reference_arm_line():
    line = _bench("--impl", "reference", "--config", "1", "--steps", "2", "--warmup", "3", "--cpu-seconds", "1")
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference"
    assert line["unit"] == "GB/s" and line["higher_is_better"] is True
    assert line["steps"] == 2 and line["warmup"] == 3 and line["n_gpus"] == 1
    assert line["dtype"] == "f64" and line["value"] > 0
    assert line["config"]["workload"].endswith("(config 1)")
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == line["value"] and cb["sample"]
    e2e = line["e2e"]
    assert e2e["value"] == line["value"] and e2e["unit"] == line["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0
    # the time per step and the bandwidth describe the same calls
    assert abs(line["ms_per_step"] * 1e3 - line["us_per_call"]) < 1e-6 * line["us_per_call"]


def test_reference_arm_other_workloads_are_marked_unavailable():
    line = _bench("--impl", "reference", "--workload", "merge")
    assert line["impl"] == "reference" and "unavailable" in line
