#!/usr/bin/env python3
"""Benchmark: fused AdamW + blockwise-E4M3 requant step on one GB300.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload flat6e9]

Default workload: 117 tiles of 7168x7168 FP32 master params (6.01e9 elements,
366,912 blocks of 128x128), step 1000, grads N(0,1e-4) with 0.1 % x100 spikes,
column-major E4M3 copy with the transposed scale grid on.  One step = one pass
of the whole hot path over the shard = one kernel launch.  The state (96 GB)
is far larger than L2 (129 MB), so no L2 flush is needed between steps.

Prints ONE JSON line on rank 0.  Under torchrun (N > 1) every rank runs its own
replica on its own GPU (weak scaling, no collective on the data path); times
are max-reduced across ranks.
"""
from __future__ import annotations

import argparse
import csv
import hashlib
import io
import json
import os
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "optimizer-step Gelem/s and achieved HBM GB/s (% of GB300 peak), 1 GPU"
UNIT = "Gelem/s"
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 8000.0
BLK = 16384
PROFILE_SUMMARY = os.path.join(ROOT, "profiles", "fp8z_step_kernel_flat6e9.md")
KERNEL_SOURCES = ["blockwise_fp8_zero_gb300/csrc/step.cu", "blockwise_fp8_zero_gb300/csrc/fp8z_device.cuh"]


# --------------------------------------------------------------------- env
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs, copy)"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback (6.8 TB/s, earlier GB300 measurement)"


def kernel_hash():
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic():
    """DRAM bytes per launch from the committed ncu summary, if the kernel
    sources still hash to the ones profiled; else None."""
    try:
        txt = open(PROFILE_SUMMARY).read()
    except OSError:
        return None
    vals = {}
    for line in txt.splitlines():
        if ":" in line and line.strip().startswith("- "):
            k, v = line.strip()[2:].split(":", 1)
            vals[k.strip()] = v.strip().strip("`")
    if vals.get("kernel_sources_sha256") != kernel_hash():
        return None
    try:
        return float(vals["dram_bytes_per_full_launch"])
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi sampled every 200 ms while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid=None):
        self.uuid = uuid
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(prefix="fp8z_clocks_", suffix=".csv")
        os.close(fd)
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "200"]
        if self.uuid:
            cmd.insert(1, f"--id={self.uuid}")
        try:
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(cmd, stdout=self.out, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.out.close()

    def summary(self):
        if self.proc is None or not self.path:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = list(csv.reader(io.StringIO(open(self.path).read())))
        os.unlink(self.path)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            r = [x.strip() for x in r]
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1]))
                smax.append(float(r[2]))
            except ValueError:
                continue
            for name, val in zip(names, r[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": max(smax), "samples": len(sm),
                "reasons": sorted(reasons)}


def max_over_ranks(x: float, device=None) -> float:
    """The largest value of x over all ranks (the job's time is the slowest
    rank's); x itself when not running distributed."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def box_copy_gbs(dev, reps=10):
    """The measured-peak recipe on this machine, after the timed region: b.copy_(a)
    over 1 Gi bf16 elements, read + write bytes, best of `reps`, CUDA events.
    Context for the box-to-box spread; the roofline's peak stays the
    driver-written one."""
    import torch
    try:
        a = torch.empty(1 << 30, dtype=torch.bfloat16, device=dev)
        b = torch.empty_like(a)
    except RuntimeError:
        return None
    a.fill_(1.0)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    best = None
    for _ in range(reps + 1):
        ev[0].record()
        b.copy_(a)
        ev[1].record()
        torch.cuda.synchronize(dev)
        ms = ev[0].elapsed_time(ev[1])
        best = ms if best is None else min(best, ms)
    del a, b
    torch.cuda.empty_cache()
    return 2 * (1 << 30) * 2 / (best / 1e3) / 1e9


def host_mem_gb():
    try:
        for line in open("/proc/meminfo"):
            if line.startswith("MemAvailable:"):
                return int(line.split()[1]) / 1e6
    except OSError:
        pass
    return 0.0


# ----------------------------------------------------------- oracle (CPU)
def cpu_oracle_run(w, host, hp_kw, threads, outputs=None):
    """Time the oracle on host arrays (a block sample, updated in place); returns
    seconds.  outputs: a dict that receives the oracle's codes and scales."""
    import oracle
    from concurrent.futures import ThreadPoolExecutor
    ohp = oracle.Hparams.make(**hp_kw)
    nb = host["p"].size // BLK
    q = np.zeros(nb * BLK, np.uint8)
    inv = np.zeros(nb, np.float32)
    per = -(-nb // threads)

    def run(b0):
        b1 = min(nb, b0 + per)
        sl = slice(b0 * BLK, b1 * BLK)
        oracle.adamw_requant_step(host["p"][sl], host["g"][sl], host["m"][sl], host["v"][sl],
                                  q[sl], inv[b0:b1], 0, b1 - b0, ohp)

    t0 = time.perf_counter()
    with ThreadPoolExecutor(threads) as ex:
        list(ex.map(run, range(0, nb, per)))
    secs = time.perf_counter() - t0
    if outputs is not None:
        outputs["q"], outputs["inv"] = q, inv
    return secs


def sample_host_blocks(w, nblocks, seed=0):
    """The workload's distributions, drawn on the host for a block sample
    (the sample is full 128x128 blocks of the same kind as the workload)."""
    import torch
    from blockwise_fp8_zero_gb300 import workloads
    host = {}
    for k in "pgmv":
        t = torch.empty(nblocks * BLK, dtype=torch.float32)
        workloads.fill(t, k, w.dists[k], seed + 17)
        host[k] = t.numpy()
    return host


# --------------------------------------------------------------- our path
def run_ours(args):
    import torch
    from blockwise_fp8_zero_gb300 import build, fp8z, workloads

    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    build.build()
    fp8z.lib()

    w = workloads.get(args.workload, args.split)
    if args.max_elems:
        w = workloads.scaled(w, args.max_elems)
    free, total = torch.cuda.mem_get_info(dev)
    per_elem = 16 + 1 + (1 if w.transposed else 0)
    budget = int((free - (6 << 30)) / per_elem)
    scaled_note = None
    if w.real_elems > budget:
        w = workloads.scaled(w, budget)
        scaled_note = f"scaled to {w.real_elems} elements to fit {free / 1e9:.0f} GB free"

    params, shards, blocks, summ = fp8z.fp8z_plan_shards(w.shapes, w.dp, w.split)
    cap = int(summ["capacity_blocks"])
    real = int(summ["real_elems"])
    state = workloads.make_state(w, blocks, dev, seed=rank)
    q = torch.empty(cap * BLK, dtype=torch.uint8, device=dev)
    inv = torch.empty(cap, dtype=torch.float32, device=dev)
    desc = fp8z.table_to_device(blocks, dev)
    pdev = fp8z.table_to_device(params, dev)
    t_bytes = int(sum(e * r * c for e, r, c in w.shapes))
    t_scales = int(sum(int(p["e"]) * int(p["hb"]) * int(p["wb"]) for p in params))
    wt = torch.empty(t_bytes, dtype=torch.uint8, device=dev) if w.transposed else None
    it = torch.empty(t_scales, dtype=torch.float32, device=dev) if w.transposed else None
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    torch.cuda.synchronize(dev)          # drawn on torch's stream; the steps run on their own
    stream = torch.cuda.Stream(dev)
    step0 = int(w.hp["step"])
    hp_kw = dict(w.hp)

    def one_step(t, s=stream):
        hp = fp8z.hparams(**{**hp_kw, "step": t})
        for sh in shards:      # one launch per shard; flat6e9 has a single shard
            fp8z.fp8z_adamw_requant_step(state["p"], state["g"], state["m"], state["v"], q, inv,
                                         int(sh["blk_begin"]), int(sh["blk_count_real"]), hp,
                                         desc=desc, params=pdev if w.transposed else None,
                                         nparams=len(params) if w.transposed else 0,
                                         w_fp8_t=wt, inv_scale_t=it, dev_status=status, stream=s)

    launches_per_step = len(shards)
    t = step0
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            one_step(t)
            t += 1
    torch.cuda.synchronize(dev)
    if status.item() != 0:
        raise RuntimeError(fp8z.fp8z_status_string(status.item()))

    def barrier():
        if ws > 1:
            import torch.distributed as dist
            dist.barrier(device_ids=[local])

    # ---- timed region: K steps, per-launch CUDA events on the launch stream
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    uuid = None
    try:
        uuid = str(torch.cuda.get_device_properties(dev).uuid)
        if uuid and not uuid.startswith("GPU-"):
            uuid = "GPU-" + uuid
    except Exception:
        uuid = None
    with ClockSampler(uuid) as clocks:
        barrier()
        torch.cuda.synchronize(dev)
        torch.cuda.nvtx.range_push("timed_steps")
        with torch.cuda.stream(stream):
            ev[0].record(stream)
            for i in range(args.steps):
                one_step(t)
                t += 1
                ev[i + 1].record(stream)
        torch.cuda.synchronize(dev)
        torch.cuda.nvtx.range_pop()
        barrier()
    clk = clocks.summary()
    if status.item() != 0:
        raise RuntimeError(fp8z.fp8z_status_string(status.item()))
    per_step_ms = [ev[i].elapsed_time(ev[i + 1]) for i in range(args.steps)]
    total_ms = max_over_ranks(ev[0].elapsed_time(ev[-1]), dev)
    value = real * args.steps * ws / (total_ms / 1e3) / 1e9

    # algorithmic bytes per launch: read g, p, m, v; write p, m, v, codes
    # (+ the column-major copy); plus per block a descriptor and inverse scale(s)
    nblk_run = int(sum(int(s["blk_count_real"]) for s in shards))
    per_block = BLK * (16 + 12 + 1 + (1 if w.transposed else 0)) + 20 + 4 + (4 if w.transposed else 0)
    alg_bytes_step = nblk_run * per_block
    avg_launch_s = (sum(per_step_ms) / len(per_step_ms)) / 1e3 / launches_per_step
    achieved = alg_bytes_step / launches_per_step / avg_launch_s / 1e9
    peak, peak_src = measured_peak()
    traffic = profiled_traffic() if (scaled_note is None and launches_per_step == 1) else None

    def fused(rm, timed):
        """The step with fold-on-read / unfold-on-write, on the row-major grad rm."""
        try:
            w_row = torch.empty(w.real_elems, dtype=torch.uint8, device=dev)
        except RuntimeError:
            return
        maps = fp8z.fp8z_encode_grad_maps([rm], params, device=dev)
        hp = fp8z.hparams(**{**hp_kw, "step": t})
        sh = shards[0]
        timed(lambda: fp8z.fp8z_adamw_requant_step_rowmajor(
            state["p"], state["m"], state["v"], maps, w_row, inv, int(sh["blk_begin"]),
            int(sh["blk_count_real"]), hp, desc, pdev, len(params), w_fp8_t=wt, inv_scale_t=it,
            dev_status=status, stream=stream), alg_bytes_step, "fp8z_adamw_requant_step_rowmajor")
        del w_row

    box_copy = box_copy_gbs(dev)
    torch.cuda.nvtx.range_push("aux_kernels")
    aux = None if (args.no_aux or len(shards) != 1) else time_aux_kernels(
        w, q, inv, params, dev, stream, peak, g=state["g"], fused=fused, no_rowwise=args.no_rowwise,
        max_tokens=args.rowwise_max_tokens)
    torch.cuda.nvtx.range_pop()
    if aux is not None:
        # the MXFP8 output variant of the same step (no column-major copy): codes
        # + one E8M0 byte per 32 elements, no block-wide amax
        try:
            mx = torch.empty(cap * 512, dtype=torch.uint8, device=dev)
            hp_mx = fp8z.hparams(**{**hp_kw, "step": t})
            sh = shards[0]
            ev2 = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
            with torch.cuda.stream(stream):
                run_mx = lambda: fp8z.fp8z_adamw_requant_step_mx(
                    state["p"], state["g"], state["m"], state["v"], q, mx, int(sh["blk_begin"]),
                    int(sh["blk_count_real"]), hp_mx, desc=desc, dev_status=status, stream=stream)
                run_mx()
                ev2[0].record(stream)
                for _ in range(5):
                    run_mx()
                ev2[1].record(stream)
            torch.cuda.synchronize(dev)
            ms_mx = ev2[0].elapsed_time(ev2[1]) / 5
            b_mx = nblk_run * (BLK * 29 + 512 + 20)
            aux["fp8z_adamw_requant_step_mx"] = {"ms": round(ms_mx, 4), "bytes": b_mx,
                                                 "gbs": round(b_mx / ms_mx / 1e6, 1),
                                                 "frac": round(b_mx / ms_mx / 1e6 / peak, 4)}
            del mx
        except RuntimeError:
            pass
    if aux is not None and w.transposed:
        # the same step without the column-major copy: what the copy costs on this machine
        hp_nc = fp8z.hparams(**{**hp_kw, "step": t})
        sh = shards[0]
        ev3 = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        with torch.cuda.stream(stream):
            run_nc = lambda: fp8z.fp8z_adamw_requant_step(
                state["p"], state["g"], state["m"], state["v"], q, inv, int(sh["blk_begin"]),
                int(sh["blk_count_real"]), hp_nc, desc=desc, dev_status=status, stream=stream)
            run_nc()
            ev3[0].record(stream)
            for _ in range(5):
                run_nc()
            ev3[1].record(stream)
        torch.cuda.synchronize(dev)
        ms_nc = ev3[0].elapsed_time(ev3[1]) / 5
        b_nc = nblk_run * (BLK * 29 + 24)
        aux["fp8z_adamw_requant_step_nocopy"] = {"ms": round(ms_nc, 4), "bytes": b_nc,
                                                 "gbs": round(b_nc / ms_nc / 1e6, 1),
                                                 "frac": round(b_nc / ms_nc / 1e6 / peak, 4),
                                                 "column_major_copy_ms": round(avg_launch_s * 1e3 - ms_nc, 4)}
    if aux and "fp8z_adamw_requant_step_rowmajor" in aux:
        aux["unfused_fold_step_unfold_ms"] = round(
            aux["fp8z_fold_f32"]["ms"] + avg_launch_s * 1e3 + aux["fp8z_unfold_e4m3"]["ms"], 4) \
            if "fp8z_unfold_e4m3" in aux else None

    # ---- several shards: the same step as one launch over every block (shard
    # padding included, masked by the descriptors) and the rank-0 shard alone
    shard_timing = None
    if len(shards) > 1:
        def timed_ranges(ranges, reps=5):
            hp_s = fp8z.hparams(**{**hp_kw, "step": t})
            evs = [torch.cuda.Event(enable_timing=True) for _ in range(2)]

            def go():
                for b0, nb in ranges:
                    fp8z.fp8z_adamw_requant_step(
                        state["p"], state["g"], state["m"], state["v"], q, inv, b0, nb, hp_s, desc=desc,
                        params=pdev if w.transposed else None, nparams=len(params) if w.transposed else 0,
                        w_fp8_t=wt, inv_scale_t=it, dev_status=status, stream=stream)
            with torch.cuda.stream(stream):
                go()
                evs[0].record(stream)
                for _ in range(reps):
                    go()
                evs[1].record(stream)
            torch.cuda.synchronize(dev)
            return evs[0].elapsed_time(evs[1]) / reps
        one_ms = timed_ranges([(0, cap)])
        a0, n0 = int(shards[0]["blk_begin"]), int(shards[0]["blk_count_real"])
        r0_ms = timed_ranges([(a0, n0)])
        r0_real = int(np.sum(blocks["valid_rows"][a0:a0 + n0].astype(np.int64)
                             * blocks["valid_cols"][a0:a0 + n0].astype(np.int64)))
        if status.item() != 0:
            raise RuntimeError(fp8z.fp8z_status_string(status.item()))
        shard_timing = {
            "per_shard_launches_ms": round(total_ms / args.steps, 4),
            "all_shards_one_launch_ms": round(one_ms, 4),
            "all_shards_one_launch_gelem_s": round(real / (one_ms / 1e3) / 1e9, 4),
            "rank0_shard_ms": round(r0_ms, 4), "rank0_blocks": n0,
            "rank0_gelem_s": round(r0_real / (r0_ms / 1e3) / 1e9, 4)}

    # ---- end to end through the C ABI with pinned host buffers
    torch.cuda.nvtx.range_push("e2e")
    e2e = None if args.no_e2e else run_e2e(args, w, state, q, inv, wt, it, desc, pdev, params,
                                            shards, hp_kw, t, dev, ws)
    torch.cuda.nvtx.range_pop()

    # ---- the other workloads, after this one's buffers are freed
    configs = None
    if not args.no_configs and w.name == "flat6e9":
        del state, q, inv, wt, it, desc, pdev
        torch.cuda.empty_cache()
        torch.cuda.nvtx.range_push("configs")
        configs = run_configs(args, dev, stream, peak)
        torch.cuda.nvtx.range_pop()

    line = {
        "metric": METRIC, "value": round(value, 4), "unit": UNIT, "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(total_ms / args.steps, 4),
        "median_ms_per_step": round(float(np.median(per_step_ms)), 4),
        "min_max_ms_per_step": [round(min(per_step_ms), 4), round(max(per_step_ms), 4)],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": w.name, "params": len(w.shapes), "elements": real, "blocks": nblk_run,
                   "split": "param-wise" if w.split == 1 else "block-wise",
                   "padding_bytes_fp32_state": int(summ["fold_pad_elems"] + summ["shard_pad_elems"]) * 16,
                   "dp_shards": w.dp, "column_major_copy": w.transposed, "step": step0,
                   "l2": f"state {cap * BLK * 16 / 1e9:.0f} GB >> 129 MB L2: no flush between steps",
                   "launches_per_step": launches_per_step, "scaled": scaled_note,
                   "parallelism": f"{ws} independent replicas, one per GPU" if ws > 1 else "one GPU",
                   "hbm_gbs": round(achieved, 1),
                   "frac_of_nominal_8tbs": round(achieved / NOMINAL_HBM_GBS, 4)},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": traffic,
                     "algorithmic_bytes": alg_bytes_step // launches_per_step,
                     "peak_source": peak_src,
                     "box_copy_gbs": None if box_copy is None else round(box_copy, 1),
                     "frac_of_box_copy": None if box_copy is None else round(achieved / box_copy, 4),
                     "kernel": "fp8z_step_kernel", "kernel_ms": round(avg_launch_s * 1e3, 4)},
        "aux_kernels": aux,
        "shard_timing": shard_timing,
        "configs": configs,
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk,
        "e2e": e2e,
    }
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:      # the host baseline at N = 1 only
        line["cpu_baseline"] = cpu_baseline(w, hp_kw, args, dev=dev)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def time_aux_kernels(w, q, inv, params, dev, stream, peak, reps=5, g=None, fused=None, no_rowwise=False,
                     max_tokens=65536):
    """Dequantize, the standalone column-major transpose, unfold/fold of the
    FP32 grad, the fused row-major step, unfold of the E4M3 codes, and the 1x128
    row-wise kernels (rowwise_study), each timed with CUDA events against its
    algorithmic bytes (dequant: 1 B read + 4 B written per element + 4 B per
    block; transpose: 1 + 1 B per element + 8 B per block; FP32 fold/unfold:
    4 + 4 B per element; byte unfold: 1 + 1 B per element)."""
    import torch
    from blockwise_fp8_zero_gb300 import fp8z
    out = {}
    nblk = inv.numel()
    try:
        buf = torch.empty(nblk * BLK, dtype=torch.float32, device=dev)
    except RuntimeError:
        return None
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    with torch.cuda.stream(stream):
        fp8z.fp8z_dequant(q, inv, nblk, buf, stream=stream)
        ev[0].record(stream)
        for _ in range(reps):
            fp8z.fp8z_dequant(q, inv, nblk, buf, stream=stream)
        ev[1].record(stream)
    torch.cuda.synchronize(dev)
    ms = ev[0].elapsed_time(ev[1]) / reps
    nbytes = nblk * (BLK * 5 + 4)
    out["fp8z_dequant"] = {"ms": round(ms, 4), "bytes": nbytes, "gbs": round(nbytes / ms / 1e6, 1),
                           "frac": round(nbytes / ms / 1e6 / peak, 4)}
    del buf
    pe = params[0]
    E, H, W = int(pe["e"]), int(pe["rows"]), int(pe["cols"])
    nb = E * int(pe["hb"]) * int(pe["wb"])
    t_out = torch.empty(E * W * H, dtype=torch.uint8, device=dev)
    t_inv = torch.empty(nb, dtype=torch.float32, device=dev)
    with torch.cuda.stream(stream):
        fp8z.fp8z_transpose_fp8(q, inv, pe, t_out, t_inv, stream=stream)
        ev[0].record(stream)
        for _ in range(reps):
            fp8z.fp8z_transpose_fp8(q, inv, pe, t_out, t_inv, stream=stream)
        ev[1].record(stream)
    torch.cuda.synchronize(dev)
    ms = ev[0].elapsed_time(ev[1]) / reps
    nbytes = E * H * W * 2 + nb * 8
    out["fp8z_transpose_fp8"] = {"ms": round(ms, 4), "bytes": nbytes, "gbs": round(nbytes / ms / 1e6, 1),
                                 "frac": round(nbytes / ms / 1e6 / peak, 4),
                                 "param": f"{E}x{H}x{W}"}
    del t_out, t_inv

    def timed(fn, nbytes, label):
        with torch.cuda.stream(stream):
            fn()
            ev[0].record(stream)
            for _ in range(reps):
                fn()
            ev[1].record(stream)
        torch.cuda.synchronize(dev)
        ms_ = ev[0].elapsed_time(ev[1]) / reps
        out[label] = {"ms": round(ms_, 4), "bytes": nbytes, "gbs": round(nbytes / ms_ / 1e6, 1),
                      "frac": round(nbytes / ms_ / 1e6 / peak, 4), "param": f"{E}x{H}x{W}"}

    if g is not None and len(params) == 1:
        try:
            rm = torch.empty(E * H * W, dtype=torch.float32, device=dev)
        except RuntimeError:
            return out
        # unfold then fold back: g ends exactly as it started
        timed(lambda: fp8z.fp8z_unfold(g, pe, rm, stream=stream), 8 * E * H * W, "fp8z_unfold_f32")
        timed(lambda: fp8z.fp8z_fold(rm, pe, g, stream=stream), 8 * E * H * W, "fp8z_fold_f32")
        if fused is not None:
            fused(rm, timed)
        del rm
        qb = torch.empty(E * H * W, dtype=torch.uint8, device=dev)
        timed(lambda: fp8z.fp8z_unfold(q, pe, qb, stream=stream), 2 * E * H * W, "fp8z_unfold_e4m3")
        del qb
    if not no_rowwise:
        try:
            out.update(rowwise_study(dev, stream, peak, max_tokens=max_tokens))
        except RuntimeError:
            pass
    return out


def _activation(T, Hd, dev, seed=5):
    """An activation of T tokens x Hd: N(0,1) with 0.1 % outliers x60.  Drawn
    on torch's current stream; the device is synchronized before it is
    returned, so kernels on another stream read it complete."""
    import torch
    gen = torch.Generator(device=dev)
    gen.manual_seed(seed)
    x = torch.randn(T, Hd, generator=gen, device=dev)
    x = torch.where(torch.rand(T, Hd, generator=gen, device=dev) < 1e-3, x * 60, x)
    torch.cuda.synchronize(dev)
    return x


def rowwise_study(dev, stream, peak, reps=5, max_tokens=65536):
    """1x128 row-wise quantization and the two ways to the column-wise layout
    ("FP8-Flow-MoE" §3.1): the scaling-aware transpose, and the naive
    dequantize -> transpose -> quantize, both run from the library's kernels
    (the naive path: fp8z_dequant_rowwise with its transposed output, then
    fp8z_quantize_rowwise; its dequantize and transpose share one pass, which
    can only make it faster).  Timed at T x 7168 activations for several T
    (power-of-two scales, the page's setting for its speed comparison), with
    each kernel's algorithmic bytes: quantize 4 + 1 B per element + 4 B per
    128; scaling-aware transpose 1 + 1 B per element + 8 B per 128; transposed
    dequantize 1 + 4 B per element + 4 B per 128."""
    import torch
    from blockwise_fp8_zero_gb300 import fp8z
    out = {}
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]

    def timed(fn):
        with torch.cuda.stream(stream):
            fn()
            ev[0].record(stream)
            for _ in range(reps):
                fn()
            ev[1].record(stream)
        torch.cuda.synchronize(dev)
        return ev[0].elapsed_time(ev[1]) / reps

    def entry(ms, nbytes, param):
        return {"ms": round(ms, 4), "bytes": nbytes, "gbs": round(nbytes / ms / 1e6, 1),
                "frac": round(nbytes / ms / 1e6 / peak, 4), "param": param}

    Hd = 7168
    sweep = {}
    tokens = [T for T in (4096, 16384, 65536) if T <= max_tokens] or [4096]
    for T in tokens:
        x = _activation(T, Hd, dev)
        n = T * Hd
        qa = torch.empty(T, Hd, dtype=torch.uint8, device=dev)
        sa = torch.empty(T, Hd // 128, device=dev)
        qta = torch.empty(Hd, T, dtype=torch.uint8, device=dev)
        sta = torch.empty(Hd, T // 128, device=dev)
        xt = torch.empty(Hd, T, device=dev)
        ms_q = timed(lambda: fp8z.fp8z_quantize_rowwise(x, True, qa, sa, stream=stream))
        ms_sa = timed(lambda: fp8z.fp8z_transpose_rowwise(qa, sa, qta, sta, stream=stream))
        ms_dt = timed(lambda: fp8z.fp8z_dequant_rowwise(qa, sa, xt, transpose=True, stream=stream))
        ms_qt = timed(lambda: fp8z.fp8z_quantize_rowwise(xt, True, qta, sta, stream=stream))
        param = f"{T}x{Hd} activation"
        if T == tokens[-1]:
            out["fp8z_quantize_rowwise"] = entry(ms_q, 5 * n + 4 * n // 128, param)
            out["fp8z_transpose_rowwise"] = entry(ms_sa, 2 * n + 8 * n // 128, param)
            out["fp8z_dequant_rowwise_transposed"] = entry(ms_dt, 5 * n + 4 * n // 128, param)
        sweep[str(T)] = {"scaling_aware_ms": round(ms_sa, 4),
                         "naive_dequant_transpose_requant_ms": round(ms_dt + ms_qt, 4),
                         "naive_over_scaling_aware": round((ms_dt + ms_qt) / ms_sa, 3)}
        del qa, sa, qta, sta, xt
        if T != tokens[-1]:
            del x
    out["rowwise_transpose_speed"] = {
        "by_tokens": sweep,
        "note": "T x 7168 activations, power-of-two scales; naive = fp8z_dequant_rowwise (transposed "
                "output) + fp8z_quantize_rowwise; the page reports 2-3x for its direct transpose "
                "over dequantize-transpose-quantize (\"FP8-Flow-MoE\" §3.1, Figure 1)"}
    out["naive_dequant_transpose_requant_ms"] = sweep[str(tokens[-1])]["naive_dequant_transpose_requant_ms"]
    out["naive_over_scaling_aware"] = sweep[str(tokens[-1])]["naive_over_scaling_aware"]
    out["rowwise_double_quantization"] = rowwise_error_study(x, stream)
    del x
    return out


def rowwise_error_study(x, stream):
    """The double-quantization error of "FP8-Flow-MoE" §3.1 at the bench's
    activation size, E = Q_col(D(Q_row(X))) - Q_col(X): X is quantized
    row-wise (1x128 tiles), brought to the column-wise layout the naive way
    (dequantize, transpose, quantize again), and compared with quantizing X^T
    column-wise directly; the scaling-aware transpose of Q_row(X) is compared
    with Q_col(X) the same way.  Every quantize, dequantize and transpose here
    is the library's; torch ops only subtract and sum.  Per scale rule:
    frac_codes_differ (codes of the two column-wise tensors), frac_values_differ
    and rel_mean_abs_E = sum|E| / sum|X| on the dequantized values (the two
    sides may carry different scales), for E_naive and for the scaling-aware
    E_sa = SA(Q_row(X)) - Q_col(X); and frac_changed_vs_row_*: the fraction of
    values that moving to the column-wise layout changes from the row-wise
    values D(Q_row(X))^T (the double quantization itself; with power-of-two
    scales the scaling-aware transpose changes only values that underflow)."""
    import torch
    from blockwise_fp8_zero_gb300 import fp8z
    T, Hd = x.shape
    dev = x.device

    def quant(v, pow2):
        q = torch.empty(v.shape, dtype=torch.uint8, device=dev)
        sc = torch.empty(v.shape[0], v.shape[1] // 128, device=dev)
        fp8z.fp8z_quantize_rowwise(v, pow2, q, sc, stream=stream)
        return q, sc

    def dq(q, sc, transpose=False):
        r, c = q.shape
        o = torch.empty((c, r) if transpose else (r, c), device=dev)
        fp8z.fp8z_dequant_rowwise(q, sc, o, transpose=transpose, stream=stream)
        return o

    res = {}
    with torch.cuda.stream(stream):
        xt = x.t().contiguous()
        denom = float(xt.abs().double().sum())
        for name, pow2 in (("pow2_scales", True), ("amax448_scales", False)):
            q_row, s_row = quant(x, pow2)
            q_dir, s_dir = quant(xt, pow2)                          # Q_col(X)
            v_dir = dq(q_dir, s_dir)
            q_nv, s_nv = quant(dq(q_row, s_row, transpose=True), pow2)   # Q_col(D(Q_row(X)))
            q_sa = torch.empty(Hd, T, dtype=torch.uint8, device=dev)
            s_sa = torch.empty(Hd, T // 128, device=dev)
            fp8z.fp8z_transpose_rowwise(q_row, s_row, q_sa, s_sa, stream=stream)
            row = {}
            v_row_t = dq(q_row, s_row, transpose=True)              # D(Q_row(X))^T
            for tag, (q2, s2) in (("naive", (q_nv, s_nv)), ("scaling_aware", (q_sa, s_sa))):
                v2 = dq(q2, s2)
                e = v2 - v_dir
                row[f"frac_codes_differ_{tag}"] = round(float((q2 != q_dir).double().mean()), 6)
                row[f"frac_values_differ_{tag}"] = round(float((e != 0).double().mean()), 6)
                row[f"rel_mean_abs_E_{tag}"] = round(float(e.abs().double().sum()) / denom, 7)
                row[f"frac_changed_vs_row_{tag}"] = round(float((v2 != v_row_t).double().mean()), 6)
                del e, v2
            del v_row_t
            # the row-wise values themselves against X (one quantization)
            row["rel_err_row_layout"] = round(float((dq(q_row, s_row) - x).abs().double().sum()) / denom, 6)
            res[name] = row
            del q_row, s_row, q_dir, s_dir, v_dir, q_nv, s_nv, q_sa, s_sa
    torch.cuda.synchronize()
    res["param"] = f"{T}x{Hd} activation"
    res["note"] = ("E = Q_col(D(Q_row(X))) - Q_col(X) on dequantized values; rel_mean_abs_E = "
                   "sum|E| / sum|X|; *_scaling_aware: the same with the scaling-aware transpose in "
                   "place of the naive path; frac_changed_vs_row_*: values that differ from "
                   "D(Q_row(X))^T")
    return res


def run_e2e(args, w, state, q, inv, wt, it, desc, pdev, params, shards, hp_kw, t, dev, ws):
    """The same step end to end: every step copies the grads in from pinned host
    memory and the E4M3 weights, inverse scales (and the column-major copy with
    its scale grid) back out, pipelined over whole params/experts on three
    streams (copy in, step, copy out).  The FP32 main params and moments stay
    resident in HBM, as in ZeRO-1."""
    import torch
    from blockwise_fp8_zero_gb300 import fp8z
    if len(shards) != 1:
        return None
    # whole-param units (experts of a 3-D bank) so the column-major copy of a
    # unit is one contiguous range
    units = []
    for i, pe in enumerate(params):
        nb_e = int(pe["hb"]) * int(pe["wb"])
        for e in range(int(pe["e"])):
            b0 = int(pe["blk_offset"]) + e * nb_e
            t0 = int(pe["t_offset"]) + e * int(pe["rows"]) * int(pe["cols"])
            s0 = int(pe["t_scale_offset"]) + e * nb_e
            units.append((b0, nb_e, t0, int(pe["rows"]) * int(pe["cols"]), s0))
    nunits = len(units)
    per_unit_host = units[0][1] * BLK * 4 + units[0][1] * BLK * (2 if w.transposed else 1)
    # pinned host buffers: at most half of the host's available memory, shared
    # by every rank of this node
    local_ranks = max(1, int(os.environ.get("LOCAL_WORLD_SIZE", "1")))
    budget = max(1, int((host_mem_gb() * 1e9 * 0.5 / local_ranks) // max(per_unit_host, 1)))
    if budget < nunits:
        units = units[:budget]
    e_blocks = sum(u[1] for u in units)
    b_end = units[-1][0] + units[-1][1]
    g_host = torch.empty(b_end * BLK, dtype=torch.float32, pin_memory=True)
    g_host.copy_(state["g"][: b_end * BLK])
    q_host = torch.empty(b_end * BLK, dtype=torch.uint8, pin_memory=True)
    inv_host = torch.empty(b_end, dtype=torch.float32, pin_memory=True)
    t_end = units[-1][2] + units[-1][3] if w.transposed else 0
    s_end = units[-1][4] + units[-1][1] if w.transposed else 0
    wt_host = torch.empty(t_end, dtype=torch.uint8, pin_memory=True) if w.transposed else None
    it_host = torch.empty(s_end, dtype=torch.float32, pin_memory=True) if w.transposed else None
    s_in, s_run, s_out = (torch.cuda.Stream(dev) for _ in range(3))
    steps = max(3, min(args.steps, 10))
    h2d = e_blocks * BLK * 4
    d2h = e_blocks * BLK + e_blocks * 4 + ((e_blocks * BLK + e_blocks * 4) if w.transposed else 0)

    # the host link as it is on this machine right now: pinned copies of up to 2 GB
    # each way (the device grad gets back its own host copy; the host code
    # buffer is overwritten by the timed steps anyway)
    nb_in = min(g_host.numel(), (2 << 30) // 4)
    nb_out = min(q_host.numel(), 2 << 30)

    def link(fn_in, fn_out):
        torch.cuda.synchronize(dev)
        t_ = time.perf_counter()
        if fn_in:
            with torch.cuda.stream(s_in):
                fn_in()
        if fn_out:
            with torch.cuda.stream(s_out):
                fn_out()
        torch.cuda.synchronize(dev)
        return time.perf_counter() - t_
    cp_in = lambda: state["g"][:nb_in].copy_(g_host[:nb_in], non_blocking=True)
    cp_out = lambda: q_host[:nb_out].copy_(q[:nb_out], non_blocking=True)
    link(cp_in, cp_out)
    # best of three: one sample can catch a transient of the shared host link
    t_in = min(link(cp_in, None) for _ in range(3))
    t_out = min(link(None, cp_out) for _ in range(3))
    t_both = min(link(cp_in, cp_out) for _ in range(3))
    h2d_gbs, d2h_gbs = nb_in * 4 / t_in / 1e9, nb_out / t_out / 1e9
    both_gbs = (nb_in * 4 + nb_out) / t_both / 1e9
    bound_s = max(h2d / (h2d_gbs * 1e9), d2h / (d2h_gbs * 1e9), (h2d + d2h) / (both_gbs * 1e9))

    ran = [None] * len(units)      # kernel done with unit u (its g may be overwritten)
    sent = [None] * len(units)     # outputs of unit u copied out (they may be overwritten)

    def one(tstep):
        hp = fp8z.hparams(**{**hp_kw, "step": tstep})
        for u, (b0, nb, t0, tn, s0) in enumerate(units):
            e_in, e_run, e_out = torch.cuda.Event(), torch.cuda.Event(), torch.cuda.Event()
            if ran[u] is not None:
                s_in.wait_event(ran[u])
            with torch.cuda.stream(s_in):
                state["g"][b0 * BLK:(b0 + nb) * BLK].copy_(g_host[b0 * BLK:(b0 + nb) * BLK], non_blocking=True)
                e_in.record(s_in)
            s_run.wait_event(e_in)
            if sent[u] is not None:
                s_run.wait_event(sent[u])
            fp8z.fp8z_adamw_requant_step(state["p"], state["g"], state["m"], state["v"], q, inv, b0, nb, hp,
                                         desc=desc, params=pdev if w.transposed else None,
                                         nparams=len(params) if w.transposed else 0,
                                         w_fp8_t=wt, inv_scale_t=it, stream=s_run)
            e_run.record(s_run)
            ran[u] = e_run
            s_out.wait_event(e_run)
            with torch.cuda.stream(s_out):
                q_host[b0 * BLK:(b0 + nb) * BLK].copy_(q[b0 * BLK:(b0 + nb) * BLK], non_blocking=True)
                inv_host[b0:b0 + nb].copy_(inv[b0:b0 + nb], non_blocking=True)
                if w.transposed:
                    wt_host[t0:t0 + tn].copy_(wt[t0:t0 + tn], non_blocking=True)
                    it_host[s0:s0 + nb].copy_(it[s0:s0 + nb], non_blocking=True)
                e_out.record(s_out)
            sent[u] = e_out
        # end of this step's work: its last output copy
        done = torch.cuda.Event(enable_timing=True)
        done.record(s_out)
        step_done.append(done)

    step_done = []
    one(t)
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    for i in range(steps):
        one(t + 1 + i)
    torch.cuda.synchronize(dev)
    secs = max_over_ranks(time.perf_counter() - t0, dev)
    real = sum(u[3] for u in units)
    # time between the ends of consecutive steps (the steps overlap, so this is
    # each step's share of the stream, not its latency)
    step_ms = [step_done[i].elapsed_time(step_done[i + 1]) for i in range(len(step_done) - 1)]
    med_ms = float(np.median(step_ms))
    return {"value": round(real * steps * ws / secs / 1e9, 4), "unit": UNIT,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": steps,
            "step_ms": [round(x, 1) for x in step_ms],
            "median_step_gelem_s": round(real * ws / (med_ms / 1e3) / 1e9, 4),
            "link": {"h2d_gbs": round(h2d_gbs, 1), "d2h_gbs": round(d2h_gbs, 1),
                     "both_gbs": round(both_gbs, 1),
                     "bound_gelem_s": round(real * ws / bound_s / 1e9, 2),
                     "note": "pinned copies measured just before the timed steps (best of three); "
                             "the bound is max(in / h2d, out / d2h, (in + out) / both)"},
            "units": f"{len(units)} of {nunits} tiles" if len(units) < nunits else f"all {nunits} tiles",
            "note": "grads in, E4M3 weights + scales out per step; FP32 state resident"}


CONFIG_RUNS = [("single_256x384", None), ("dense_h7168", None), ("moe64", None),
               ("mixed500", 1), ("mixed500", 0)]


def _prior_moments(w, state, blocks, steps=10):
    """m, v of a workload that has run `steps` earlier optimizer steps (ten
    for the step-11 workloads): that many moment updates from zero
    (exp_avg = b1 exp_avg + (1 - b1) g, exp_avg_sq = b2 exp_avg_sq +
    (1 - b2) g^2, the moment half of the AdamW step), each with a fresh grad
    drawn from the workload's own grad distribution, in plain torch ops on the
    tensors' device; the g buffer serves as the scratch and gets the timed
    step's own grad back at the end.  The moments do not depend on the params,
    so the params keep their draw."""
    from blockwise_fp8_zero_gb300 import workloads
    b1, b2 = float(w.hp["beta1"]), float(w.hp["beta2"])
    vr, vc = blocks["valid_rows"], blocks["valid_cols"]
    m, v, g = state["m"], state["v"], state["g"]
    m.zero_()
    v.zero_()
    for k in range(steps):
        workloads.fill(g, "g", w.dists["g"], 101 + k, vr, vc)
        m.mul_(b1).add_(g, alpha=1.0 - b1)
        v.mul_(b2).addcmul_(g, g, value=1.0 - b2)
    workloads.fill(g, "g", w.dists["g"], 0, vr, vc)


def _measure_config(w, dev, stream, peak, reps):
    """One workload of run_configs: plan, draw, time, free (its tensors go out of
    scope on return)."""
    import torch
    from blockwise_fp8_zero_gb300 import fp8z, workloads
    params, shards, blocks, summ = fp8z.fp8z_plan_shards(w.shapes, w.dp, w.split)
    cap = int(summ["capacity_blocks"])
    free, _ = torch.cuda.mem_get_info(dev)
    if cap * BLK * 17 + (4 << 30) > free:
        return {"skipped": f"needs {cap * BLK * 17 / 1e9:.0f} GB, {free / 1e9:.0f} GB free"}
    state = workloads.make_state(w, blocks, dev, seed=0)
    prior = int(w.extra.get("prior_steps", 0))
    if prior > 0:
        _prior_moments(w, state, blocks, prior)
    q = torch.empty(cap * BLK, dtype=torch.uint8, device=dev)
    inv = torch.empty(cap, dtype=torch.float32, device=dev)
    desc = fp8z.table_to_device(blocks, dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    torch.cuda.synchronize(dev)      # drawn on torch's stream; the steps run on their own
    hp = fp8z.hparams(**w.hp)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]

    def timed(ranges):
        def go():
            for b0, nb in ranges:
                fp8z.fp8z_adamw_requant_step(state["p"], state["g"], state["m"], state["v"], q, inv, b0,
                                             nb, hp, desc=desc, dev_status=status, stream=stream)
        with torch.cuda.stream(stream):
            for _ in range(3):
                go()
            ev[0].record(stream)
            for _ in range(reps):
                go()
            ev[1].record(stream)
        torch.cuda.synchronize(dev)
        return ev[0].elapsed_time(ev[1]) / reps

    shard_ranges = [(int(sh["blk_begin"]), int(sh["blk_count_real"])) for sh in shards]
    real = int(summ["real_elems"])
    nreal = int(summ["total_blocks"])
    per_block = BLK * 29 + 24
    ms = timed(shard_ranges)
    entry = {"dp_shards": w.dp, "split": "param-wise" if w.split == 1 else "block-wise",
             "moments": (f"{prior} prior moment updates with fresh grads (plain torch ops)" if prior > 0
                         else "zero (first step)"),
             "params": len(w.shapes), "elements": real, "blocks": nreal, "capacity_blocks": cap,
             "padding_bytes_fp32_state": int(summ["fold_pad_elems"] + summ["shard_pad_elems"]) * 16,
             "fold_pad_elems": int(summ["fold_pad_elems"]),
             "shard_pad_elems": int(summ["shard_pad_elems"]),
             "launches": len(shards), "ms": round(ms, 4),
             "gelem_s": round(real / (ms / 1e3) / 1e9, 4),
             "gbs": round(nreal * per_block / ms / 1e6, 1),
             "frac": round(nreal * per_block / ms / 1e6 / peak, 4)}
    if len(shards) > 1:
        one_ms = timed([(0, cap)])
        a0, n0 = shard_ranges[0]
        r0_ms = timed([(a0, n0)])
        r0_real = int(np.sum(blocks["valid_rows"][a0:a0 + n0].astype(np.int64)
                             * blocks["valid_cols"][a0:a0 + n0].astype(np.int64)))
        entry["shard_timing"] = {
            "per_shard_launches_ms": round(ms, 4),
            "all_shards_one_launch_ms": round(one_ms, 4),
            "all_shards_one_launch_gelem_s": round(real / (one_ms / 1e3) / 1e9, 4),
            "all_shards_one_launch_frac": round(cap * per_block / one_ms / 1e6 / peak, 4),
            "rank0_shard_ms": round(r0_ms, 4), "rank0_blocks": n0,
            "rank0_gelem_s": round(r0_real / (r0_ms / 1e3) / 1e9, 4),
            "rank0_gbs": round(n0 * per_block / r0_ms / 1e6, 1),
            "rank0_frac": round(n0 * per_block / r0_ms / 1e6 / peak, 4)}
    else:
        entry["us"] = round(ms * 1e3, 2)
    if status.item() != 0:
        raise RuntimeError(f"{w.name}: {fp8z.fp8z_status_string(status.item())}")
    return entry


def run_configs(args, dev, stream, peak, reps=10):
    """The step on the other workloads, one after another in this process (each
    freed before the next): per-shard launches (the whole model's step as D
    launches, one per shard), all shards as one launch (shard padding masked by
    the descriptors), and the rank-0 shard alone, the per-rank optimizer step a
    DP rank would run.  Bytes: 29 B per element of every block a launch
    processes (16 read, 13 written) + 24 B per block (descriptor, scale)."""
    import torch
    from blockwise_fp8_zero_gb300 import workloads
    res = {}
    for name, split in CONFIG_RUNS:
        w = workloads.get(name, split)
        key = name if split is None else f"{name}_{'paramwise' if split == 1 else 'blockwise'}"
        try:
            res[key] = _measure_config(w, dev, stream, peak, reps)
        except torch.cuda.OutOfMemoryError as e:
            res[key] = {"skipped": f"out of device memory: {str(e).splitlines()[0][:120]}"}
        torch.cuda.empty_cache()
    res["note"] = ("no column-major copy (only the flat 6e9 workload carries one); the same kernel, "
                   "hyper-parameters of each workload; frac of the measured copy bandwidth")
    return res


def sample_parity(w, hp_kw, host_in, want, dev):
    """The timed kernel on the oracle's block sample: the same inputs go through
    fp8z_adamw_requant_step on the GPU, and every output is compared bit for bit
    with the oracle's (p', m', v' as float bit patterns, NaN equal to NaN; E4M3
    codes, a NaN code equal to either sign's; inverse scales)."""
    import torch
    from blockwise_fp8_zero_gb300 import fp8z
    nb = host_in["p"].size // BLK
    d = {k: torch.from_numpy(host_in[k]).to(dev) for k in "pgmv"}
    q = torch.zeros(nb * BLK, dtype=torch.uint8, device=dev)
    inv = torch.zeros(nb, dtype=torch.float32, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    fp8z.fp8z_adamw_requant_step(d["p"], d["g"], d["m"], d["v"], q, inv, 0, nb,
                                 fp8z.hparams(**{**hp_kw, "step": int(hp_kw["step"])}), dev_status=st)
    torch.cuda.synchronize(dev)
    out = {"blocks": nb, "elements": nb * BLK, "status": int(st.item())}
    for k in "pmv":
        a = d[k].cpu().numpy()
        b = want[k]
        same = (a.view(np.uint32) == b.view(np.uint32)) | (np.isnan(a) & np.isnan(b))
        out[f"{k}_mismatches"] = int((~same).sum())
    qa, qb = q.cpu().numpy(), want["q"]
    out["code_mismatches"] = int((~((qa == qb) | (((qa & 0x7F) == 0x7F) & ((qb & 0x7F) == 0x7F)))).sum())
    out["scale_mismatches"] = int((inv.cpu().numpy().view(np.uint32) != want["inv"].view(np.uint32)).sum())
    out["identical"] = out["status"] == 0 and not any(out[k] for k in
                                                      ("p_mismatches", "m_mismatches", "v_mismatches",
                                                       "code_mismatches", "scale_mismatches"))
    return out


def cpu_baseline(w, hp_kw, args, threads=None, dev=None):
    threads = threads or (os.cpu_count() or 1)
    nblocks = args.cpu_blocks
    host = sample_host_blocks(w, nblocks)
    host_in = {k: v.copy() for k, v in host.items()} if dev is not None else None
    oracle_out = {}
    secs = cpu_oracle_run(w, host, {**hp_kw, "step": int(hp_kw["step"])}, threads, outputs=oracle_out)
    parity = None
    if dev is not None:
        parity = sample_parity(w, hp_kw, host_in, {"p": host["p"], "m": host["m"], "v": host["v"],
                                                  "q": oracle_out["q"], "inv": oracle_out["inv"]}, dev)
        del host_in
    # the same oracle on one core, on the first 1/16 of the sample
    n1 = max(1, nblocks // 16)
    one = {k: v[:n1 * BLK].copy() for k, v in host.items()}
    secs1 = cpu_oracle_run(w, one, {**hp_kw, "step": int(hp_kw["step"])}, 1)
    return {"value": round(nblocks * BLK / secs / 1e9, 6), "unit": UNIT, "cores": threads,
            "kind": "oracle",
            "sample": f"{nblocks} full 128x128 blocks ({nblocks * BLK} elements) of the {w.name} "
                      f"distributions, one oracle step, {threads} threads over block ranges, "
                      f"{secs:.2f} s wall",
            "single_core": {"value": round(n1 * BLK / secs1 / 1e9, 6), "unit": UNIT,
                            "sample": f"{n1} blocks, {secs1:.2f} s wall"},
            "parity_vs_gpu": parity}


def run_reference(args):
    ws, rank, local = dist_env()
    if rank != 0:
        return
    from blockwise_fp8_zero_gb300 import workloads
    import oracle
    oracle.build_oracle()
    w = workloads.get(args.workload)
    threads = os.cpu_count() or 1
    nblocks = args.cpu_blocks
    host = sample_host_blocks(w, nblocks)
    if args.warmup > 0:
        cpu_oracle_run(w, {k: v.copy() for k, v in host.items()}, dict(w.hp), threads)
    secs = 0.0
    for i in range(args.steps):
        secs += cpu_oracle_run(w, host, {**w.hp, "step": int(w.hp["step"]) + i}, threads)
    value = nblocks * BLK * args.steps / secs / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": UNIT,
            "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(secs / args.steps * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": w.name, "sample_blocks": nblocks,
                       "note": "the CPU oracle on a block sample of the workload per step"},
            "cpu_baseline": {"value": round(value, 6), "unit": UNIT, "cores": threads, "kind": "oracle",
                             "sample": f"{nblocks} blocks of {w.name} per step"},
            "e2e": {"value": round(value, 6), "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="flat6e9")
    ap.add_argument("--split", type=int, default=None, choices=[0, 1],
                    help="0 block-wise, 1 param-wise (default: the workload's own)")
    ap.add_argument("--cpu-blocks", type=int, default=24576)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-aux", action="store_true", help="skip the dequant/transpose timings")
    ap.add_argument("--no-configs", action="store_true", help="skip the other workloads' step timings")
    ap.add_argument("--no-rowwise", action="store_true", help="skip the 1x128 row-wise study")
    ap.add_argument("--rowwise-max-tokens", type=int, default=65536,
                    help="largest activation of the row-wise study (4096, 16384 or 65536 tokens)")
    ap.add_argument("--max-elems", type=int, default=0,
                    help="run a smaller workload of the same kind (profiling cases)")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
