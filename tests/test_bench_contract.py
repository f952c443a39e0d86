"""bench.py's reference arm (the fp64 oracle timed on the host cores) prints
one JSON line with the keys the benchmark contract asks for: the same metric,
unit and config as the GPU arm, `impl: reference`, a `cpu_baseline` that
describes the run, and an `e2e` whose value is the line's own with no
host-device bytes.  Runs on CPU in a few seconds."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_json_line():
    out = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1",
                          "--warmup", "3"], cwd=ROOT, capture_output=True, text=True,
                         timeout=300)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference"
    assert d["unit"] == "TFLOP/s" and d["higher_is_better"] is True
    assert d["steps"] == 1 and d["warmup"] == 3 and d["n_gpus"] == 1
    assert d["config"]["workload"] == "longformer_base_fp16_n4096_w256_d0"
    assert d["value"] > 0
    # the line reports the work it timed: value = the step's flops / its time
    fl = d["config"]["flops_per_step"]
    assert d["config"]["slices_per_step"] == 1
    assert abs(fl / (d["ms_per_step"] * 1e-3) / 1e12 - d["value"]) <= 1e-3 * d["value"] + 1e-6
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1
    assert cb["sample"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_warmup_below_three_is_refused():
    out = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1",
                          "--warmup", "2"], cwd=ROOT, capture_output=True, text=True,
                         timeout=120)
    assert out.returncode != 0
    assert "--warmup must be >= 3" in out.stderr
