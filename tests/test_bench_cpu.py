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


def test_profiled_traffic_matches_current_kernel():
    """The bench's roofline `traffic` comes from the committed ncu summary only
    while the step kernel's sources hash to the captured ones; this holds the
    committed sources and summary together (a kernel change needs a new
    capture, a comment-only edit of the sources breaks the match too)."""
    sys.path.insert(0, ROOT)
    import bench
    t = bench.profiled_traffic()
    assert t is not None, "step kernel sources differ from the profiled ones"
    assert 1.7e11 < t < 1.9e11


def test_prior_moments_match_the_drawn_stand_in():
    """The config timings run the ten moment updates that a step count of 11
    implies; the parity tests draw m, v from the distribution those updates
    give (exp_avg N(0, (0.2150 sigma)^2), exp_avg_sq of mean 0.4013 sigma^2).
    The two must agree: on 64 blocks of N(0, 1e-3) grads the updates' m has
    that spread and v that mean, within a sampling error of ~0.2 %.  Swapped
    betas (v mean 0.651 sigma^2) or a missing (1 - beta) factor fail here."""
    import numpy as np
    import torch
    sys.path.insert(0, ROOT)
    import bench
    from blockwise_fp8_zero_gb300 import workloads
    w = workloads.get("dense_h7168")
    assert w.extra["prior_steps"] == 10 and w.hp["step"] == 11
    nb = 64
    blocks = {"valid_rows": np.full(nb, 128, np.int32), "valid_cols": np.full(nb, 128, np.int32)}
    state = {k: torch.full((nb * 16384,), 7.0) for k in "gmv"}
    bench._prior_moments(w, state, blocks, 10)
    sigma = 1e-3
    m, v = state["m"].double(), state["v"].double()
    assert abs(m.mean().item()) < 0.01 * workloads.M10_STD * sigma
    assert abs(m.std().item() / (workloads.M10_STD * sigma) - 1) < 0.01
    assert abs(v.mean().item() / (workloads.V10_MEAN * sigma * sigma) - 1) < 0.01
    g0 = torch.empty(nb * 16384)
    workloads.fill(g0, "g", w.dists["g"], 0, blocks["valid_rows"], blocks["valid_cols"])
    assert torch.equal(state["g"], g0)          # the timed step's own grad is back


def test_reference_arm_under_torchrun_prints_one_line():
    """Launched as the driver launches N > 1 (torchrun, one process per rank,
    127.0.0.1), the reference arm runs on rank 0 alone: one JSON line with
    n_gpus = 2, and every rank exits 0."""
    import socket
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        port = sk.getsockname()[1]
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "2", "--warmup", "1", "--cpu-blocks", "32"]
    out = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.strip().startswith("{")]
    assert len(lines) == 1, out.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
