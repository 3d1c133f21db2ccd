"""bench.py's host-side contract on CPU: the nearest-rank percentile of the
timing spread, the warm-up rule, and the JSON line of the reference arm (the
f64 oracle timed on the host cores), parsed and checked key by key."""
import json
import os
import subprocess
import sys

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_percentile_nearest_rank():
    xs = [5.0, 1.0, 3.0, 2.0, 4.0]
    assert bench.percentile(xs, 0) == 1.0
    assert bench.percentile(xs, 50) == 3.0
    assert bench.percentile(xs, 100) == 5.0
    assert bench.percentile([7.0], 90) == 7.0
    ys = list(range(101))
    assert bench.percentile(ys, 10) == 10 and bench.percentile(ys, 90) == 90


def test_warmup_below_three_is_refused():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--warmup", "2"],
                       cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode != 0 and "--warmup must be >= 3" in r.stderr


def test_reference_arm_json_line():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--config", "tiny",
                        "--steps", "1", "--warmup", "3"],
                       cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout[-2000:]
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "GB/s" and d["higher_is_better"] is True
    assert d["n_gpus"] == 1 and d["steps"] == 1 and d["warmup"] == 3 and d["value"] > 0
    assert d["scaling"] == "weak" and d["data"] == "synthetic"
    assert d["config"]["workload"] == "tiny"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"]
    assert cb["cores"] >= 1 and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": "GB/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
