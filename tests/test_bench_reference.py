"""The bench's reference arm runs the CPU oracle (no GPU): its one JSON line
keeps the bench contract's keys, and its workload and metric are the GPU
arm's."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def run_bench(*args):
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT,
                         capture_output=True, text=True, timeout=600, check=True).stdout
    lines = [l for l in out.splitlines() if l.startswith("{")]
    assert len(lines) == 1, out
    return json.loads(lines[0])


def test_reference_arm_line_on_the_tiny_workload(built_lib):
    d = run_bench("--impl", "reference", "--steps", "2", "--warmup", "0",
                  "--workload", "tiny_ncc_256_t16")
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference"
    assert d["metric"] == "NCC coefficients/s (tiny_ncc_256_t16)"
    assert d["unit"] == "coefficients/s" and d["higher_is_better"] is True
    assert d["steps"] == 2 and d["value"] > 0 and d["ms_per_step"] > 0
    assert d["config"]["workload"] == "tiny_ncc_256_t16"
    assert d["config"]["sample_rows"] == 241          # the whole 241 x 241 map
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["h2d_bytes_per_step"] == 0
