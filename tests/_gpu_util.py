"""Helpers for the GPU parity tests: seeded inputs, the CUDA path through the
C ABI, and the oracle run over the same blocks on the host (threads over block
ranges; the oracle's C code releases the GIL)."""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

from blockwise_fp8_zero_gb300 import fp8z, workloads

BLK = fp8z.BLOCK_ELEMS
THREADS = max(1, min(32, os.cpu_count() or 1))


def oracle_hp(oracle, hp):
    return oracle.Hparams(hp.lr, hp.beta1, hp.beta2, hp.eps, hp.weight_decay, hp.step,
                          hp.fp8_max, hp.min_scale, hp.scale_mode, hp.decay_mode)


def oracle_blocks(oracle, hp, p, g, m, v, desc, params=None, wt=None, it=None):
    """Run the oracle step over every block of the host arrays (in place on
    p, m, v).  desc: descriptor of each block (same order) or None.
    Returns (q, inv)."""
    nb = p.size // BLK
    q = np.zeros(nb * BLK, np.uint8)
    inv = np.zeros(nb, np.float32)
    ohp = oracle_hp(oracle, hp)
    step = max(1, -(-nb // THREADS))

    def run(b0):
        b1 = min(nb, b0 + step)
        sl = slice(b0 * BLK, b1 * BLK)
        oracle.adamw_requant_step(p[sl], g[sl], m[sl], v[sl], q[sl], inv[b0:b1], 0, b1 - b0, ohp,
                                  desc=None if desc is None else np.ascontiguousarray(desc[b0:b1]),
                                  params=params, w_fp8_t=wt, inv_scale_t=it)

    with ThreadPoolExecutor(THREADS) as ex:
        list(ex.map(run, range(0, nb, step)))
    return q, inv


class Case:
    """A planned, filled workload on the GPU plus its host copy of the inputs."""

    def __init__(self, shapes, dp=1, split=0, dists=None, seed=0, device="cuda", transposed=False,
                 gen_device="cpu"):
        import torch
        self.shapes = shapes
        self.dp = dp
        self.split = split
        self.params, self.shards, self.blocks, self.summary = fp8z.fp8z_plan_shards(shapes, dp, split)
        self.cap = int(self.summary["capacity_blocks"])
        dists = dists or dict(p=workloads.Dist("normal", 0.02), g=workloads.Dist("normal", 1e-3),
                              m=workloads.Dist("normal", 2e-4),
                              v=workloads.Dist("uniform", 2e-7, 6e-7))
        self.host = {}
        self.dev = {}
        for k in "pgmv":
            t = torch.empty(self.cap * BLK, dtype=torch.float32, device=gen_device)
            workloads.fill(t, k, dists[k], seed, self.blocks["valid_rows"], self.blocks["valid_cols"])
            self.dev[k] = t.to(device)
            self.host[k] = t.cpu().numpy().copy()
        self.w_fp8 = torch.zeros(self.cap * BLK, dtype=torch.uint8, device=device)
        self.inv = torch.zeros(self.cap, dtype=torch.float32, device=device)
        self.desc_dev = fp8z.table_to_device(self.blocks, device)
        self.params_dev = fp8z.table_to_device(self.params, device)
        self.t_bytes = int(sum(e * r * c for e, r, c in shapes))
        self.t_scales = int(sum(int(p["e"]) * int(p["hb"]) * int(p["wb"]) for p in self.params))
        self.transposed = transposed
        if transposed:
            self.wt = torch.zeros(self.t_bytes, dtype=torch.uint8, device=device)
            self.it = torch.zeros(self.t_scales, dtype=torch.float32, device=device)
        else:
            self.wt = self.it = None
        self.status = torch.zeros(1, dtype=torch.int32, device=device)
        self.processed = np.zeros(self.cap, bool)
        self._oracle_plan = None

    def oracle_tables(self, oracle):
        """The oracle's own planner tables (params, blocks) for this layout: the
        oracle's inputs never come from the library."""
        if self._oracle_plan is None:
            op, _, ob, _ = oracle.plan_shards(self.shapes, self.dp, self.split)
            self._oracle_plan = (op, ob)
        return self._oracle_plan

    def step(self, hp, ranges=None, use_desc=True):
        """Run the CUDA step over the given (begin, count) block ranges
        (default: every shard's real range, one launch per shard)."""
        import torch
        if ranges is None:
            ranges = [(int(s["blk_begin"]), int(s["blk_count_real"])) for s in self.shards]
        for b0, nb in ranges:
            self.processed[b0:b0 + nb] = True
            fp8z.fp8z_adamw_requant_step(
                self.dev["p"], self.dev["g"], self.dev["m"], self.dev["v"], self.w_fp8, self.inv,
                b0, nb, hp, desc=self.desc_dev if use_desc else None,
                params=self.params_dev if self.transposed else None,
                nparams=len(self.params) if self.transposed else 0,
                w_fp8_t=self.wt, inv_scale_t=self.it, dev_status=self.status)
        torch.cuda.synchronize()
        assert int(self.status.item()) == 0, fp8z.fp8z_status_string(int(self.status.item()))

    def oracle(self, oracle, hp, use_desc=True):
        """Oracle over all capacity blocks, on the host copy of the inputs."""
        p, g, m, v = (self.host[k].copy() for k in "pgmv")
        wt = np.zeros(self.t_bytes, np.uint8) if self.transposed else None
        it = np.zeros(self.t_scales, np.float32) if self.transposed else None
        op, ob = self.oracle_tables(oracle)
        params = op if self.transposed else None
        desc = ob if use_desc else None
        q, inv = oracle_blocks(oracle, hp, p, g, m, v, desc, params, wt, it)
        return dict(p=p, m=m, v=v, q=q, inv=inv, wt=wt, it=it)

    def results(self):
        out = {k: self.dev[k].cpu().numpy() for k in "pmv"}
        out["q"] = self.w_fp8.cpu().numpy()
        out["inv"] = self.inv.cpu().numpy()
        out["wt"] = self.wt.cpu().numpy() if self.wt is not None else None
        out["it"] = self.it.cpu().numpy() if self.it is not None else None
        return out


def data_mask(blocks):
    return blocks["param"] >= 0


def assert_bitexact(got, want, inv_mask=None):
    """p, m, v, q and inv identical (the build is IEEE div/sqrt, no FMA);
    NaN equal to NaN; an E4M3 NaN code may differ only in its sign bit."""
    for k in ("p", "m", "v"):
        a, b = got[k], want[k]
        same = (a.view(np.uint32) == b.view(np.uint32)) | (np.isnan(a) & np.isnan(b))
        if not np.all(same):
            bad = np.nonzero(~same)[0]
            raise AssertionError(f"{k}: {bad.size} mismatches, first at {bad[:5]}: "
                                 f"{a[bad[:5]]} vs {b[bad[:5]]}")
    qa, qb = got["q"], want["q"]
    nan_codes = ((qa & 0x7F) == 0x7F) & ((qb & 0x7F) == 0x7F)
    ok = (qa == qb) | nan_codes
    if not np.all(ok):
        bad = np.nonzero(~ok)[0]
        raise AssertionError(f"q: {bad.size} mismatches, first at {bad[:5]}: {qa[bad[:5]]} vs {qb[bad[:5]]}")
    ia, ib = got["inv"], want["inv"]
    sel = np.ones(ia.shape, bool) if inv_mask is None else inv_mask
    assert np.array_equal(ia[sel].view(np.uint32), ib[sel].view(np.uint32)), "inv_scale differs"
    if want.get("wt") is not None:
        assert np.array_equal(got["wt"], want["wt"]), "column-major copy differs"
        assert np.array_equal(got["it"].view(np.uint32), want["it"].view(np.uint32)), \
            "transposed scale grid differs"
