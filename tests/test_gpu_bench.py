"""The benchmark's JSON line on a one-tile case of the 6e9 workload: one
line, every key the line promises, consistent numbers (value = elements /
time, the roofline fraction = achieved / peak, one launch per timed step,
the end-to-end bytes per step of one 7168^2 tile)."""
import json
import os
import subprocess
import sys

import pytest

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_bench_line_schema():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--workload", "flat6e9",
           "--max-elems", str(7168 * 7168), "--steps", "4", "--warmup", "3",
           "--no-cpu-baseline", "--no-aux"]
    out = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.strip().startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data", "config", "roofline", "gpu_launches", "clocks"):
        assert k in d, k
    assert d["n_gpus"] == 1 and d["steps"] == 4 and d["warmup"] == 3
    assert d["higher_is_better"] is True and d["scaling"] == "weak" and d["dtype"] == "f32"
    assert d["config"]["workload"].startswith("flat6e9") and d["config"]["elements"] == 7168 * 7168
    r = d["roofline"]
    for k in ("bound", "achieved", "peak", "unit", "frac", "traffic"):
        assert k in r, k
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and 0 < r["frac"] < 1.5
    assert abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-3
    # the copy recipe re-measured on this machine, beside the recorded peak
    assert r["box_copy_gbs"] > 0 and abs(r["frac_of_box_copy"] - r["achieved"] / r["box_copy_gbs"]) < 1e-3
    assert abs(d["value"] - d["config"]["elements"] / (d["ms_per_step"] / 1e3) / 1e9) < 0.01 * d["value"]
    assert d["gpu_launches"] == d["steps"]
    lo, hi = d["min_max_ms_per_step"]
    assert 0 < lo <= d["median_ms_per_step"] <= hi
    assert {"sm_mhz", "sm_max_mhz", "reasons"} <= set(d["clocks"])
    e = d["e2e"]
    n = 7168 * 7168
    assert e["unit"] == "Gelem/s" and e["value"] > 0 and e["median_step_gelem_s"] > 0
    # grads in; codes + inverse scales + the column-major copy and its grid out
    assert e["h2d_bytes_per_step"] == 4 * n
    assert e["d2h_bytes_per_step"] == 2 * n + 2 * 4 * (n // 16384)
    assert len(e["step_ms"]) == e["steps"] and all(x > 0 for x in e["step_ms"])
    assert {"h2d_gbs", "d2h_gbs", "both_gbs", "bound_gelem_s"} <= set(e["link"])
