"""The benchmark's reference arm (the CPU oracle on a block sample) and the
host-side helpers run without a GPU and print the contract's JSON line."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_json_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--steps", "2", "--warmup", "1", "--cpu-blocks", "64"],
                         capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr
    line = json.loads(out.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference"
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "config", "cpu_baseline", "e2e"):
        assert k in line, k
    assert line["unit"] == "Gelem/s" and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"
    assert line["config"]["workload"] == "flat6e9"


def test_profiled_traffic_matches_current_kernel_or_is_null():
    sys.path.insert(0, ROOT)
    import bench
    t = bench.profiled_traffic()
    assert t is None or 1.7e11 < t < 1.9e11
