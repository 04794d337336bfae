"""Seeded synthetic workloads: shapes, hyper-parameters and input draws.

This module only draws random inputs and zeroes padding; it holds none of the
optimizer's arithmetic and imports neither the CUDA binding nor the oracle, so
tests, the oracle checks and the benchmark can all take their inputs from it.

Workloads (all synthetic; no dataset or checkpoint is involved):
  single_256x384   one 256x384 weight (6 blocks), 1 shard, step 1, m = v = 0
  dense_h7168      hidden-7168 dense layer set: Q, O 7168x7168, KV-down
                   7168x576 (ragged edge blocks), MLP up, gate 7168x18432,
                   down 18432x7168; block-wise split into 8 shards
  moe64            64 experts x (gate, up 2048x7168; down 7168x2048) as three
                   [64, ., .] banks; Student-t(3) grads; 16 shards
  mixed500         500 matrices with rows/cols log-uniform in [128, 18432] in
                   multiples of 64; 16 shards, param-wise or block-wise
  flat6e9          117 tiles of 7168x7168 (6.01e9 elements), step 1000, grads
                   N(0, 1e-4) with 0.1 % of them x100; column-major copy on
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

BLOCK = 128
BLOCK_ELEMS = BLOCK * BLOCK

# Moments after ten prior steps from zero with grads N(0, sigma^2) and
# betas (0.9, 0.95): exp_avg is N(0, (0.2150*sigma)^2) since
# Var = sigma^2 (1-b1)^2 sum_{j<10} b1^(2j); exp_avg_sq has mean
# sigma^2 (1 - b2^10) = 0.4013 sigma^2, drawn here uniform in [0.5, 1.5] x mean.
# Workloads drawn this way carry extra["prior_steps"] = 10, for a caller that
# runs the ten moment updates itself instead.
M10_STD = 0.2150
V10_MEAN = 0.4013


@dataclass
class Dist:
    kind: str                 # normal | uniform | student_t | spiky_normal | zeros
    a: float = 0.0            # std (normal), low (uniform), scale (student_t)
    b: float = 0.0            # high (uniform), dof (student_t)
    frac: float = 0.0         # spiky_normal: fraction multiplied by `mult`
    mult: float = 1.0


@dataclass
class Workload:
    name: str
    shapes: list                      # [(e, rows, cols)]
    dp: int
    split: int                        # 0 block-wise, 1 param-wise
    hp: dict                          # lr, beta1, beta2, eps, weight_decay, step
    dists: dict                       # tensor name -> Dist
    transposed: bool = False
    note: str = ""
    extra: dict = field(default_factory=dict)

    @property
    def real_elems(self) -> int:
        return int(sum(e * r * c for e, r, c in self.shapes))


def _hp(step, lr=1e-4):
    return dict(lr=lr, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1, step=step)


def _ten_prior_steps(sigma):
    return dict(m=Dist("normal", M10_STD * sigma),
                v=Dist("uniform", 0.5 * V10_MEAN * sigma * sigma, 1.5 * V10_MEAN * sigma * sigma))


def mixed500_shapes(n=500, seed=0):
    """(rows, cols) = clamp(64*round(exp(U(ln 128, ln 18432))/64), 128, 18432),
    drawn as one (n, 2) array from numpy default_rng(seed)."""
    rng = np.random.default_rng(seed)
    u = rng.uniform(np.log(128.0), np.log(18432.0), size=(n, 2))
    dims = np.clip(64 * np.round(np.exp(u) / 64), 128, 18432).astype(np.int64)
    return [(1, int(r), int(c)) for r, c in dims]


def get(name: str, split: int | None = None) -> Workload:
    if name == "single_256x384":
        return Workload(name, [(1, 256, 384)], 1, 0, _hp(1),
                        dict(p=Dist("normal", 0.02), g=Dist("normal", 1e-3),
                             m=Dist("zeros"), v=Dist("zeros")))
    if name == "dense_h7168":
        h, f = 7168, 18432
        shapes = [(1, h, h), (1, h, h), (1, h, 576), (1, h, f), (1, h, f), (1, f, h)]
        return Workload(name, shapes, 8, 0, _hp(11),
                        dict(p=Dist("normal", 0.02), g=Dist("normal", 1e-3), **_ten_prior_steps(1e-3)),
                        note="Q, O, KV-down, up, gate, down", extra=dict(prior_steps=10))
    if name == "moe64":
        shapes = [(64, 2048, 7168), (64, 2048, 7168), (64, 7168, 2048)]
        sigma = 1e-3 * np.sqrt(3.0)          # std of 1e-3 * t(3)
        return Workload(name, shapes, 16, 0, _hp(11),
                        dict(p=Dist("normal", 0.02), g=Dist("student_t", 1e-3, 3.0),
                             **_ten_prior_steps(sigma)),
                        note="gate, up, down banks of 64 experts", extra=dict(prior_steps=10))
    if name == "mixed500":
        return Workload(name, mixed500_shapes(), 16, 1 if split is None else split, _hp(11),
                        dict(p=Dist("normal", 0.02), g=Dist("normal", 1e-3), **_ten_prior_steps(1e-3)),
                        extra=dict(prior_steps=10))
    if name == "flat6e9":
        return Workload(name, [(117, 7168, 7168)], 1, 0, _hp(1000),
                        dict(p=Dist("normal", 0.02),
                             g=Dist("spiky_normal", 1e-4, frac=1e-3, mult=100.0),
                             m=Dist("normal", 1e-5), v=Dist("uniform", 0.5e-8, 1.5e-8)),
                        transposed=True, note="117 x 7168^2 = 6,011,486,208 elements")
    raise KeyError(name)


NAMES = ["single_256x384", "dense_h7168", "moe64", "mixed500", "flat6e9"]


def scaled(w: Workload, max_elems: int) -> Workload:
    """A smaller workload of the same kind (for memory-limited runs): keeps the
    first params (and the first experts of 3-D banks) until max_elems."""
    out, tot = [], 0
    for e, r, c in w.shapes:
        per = r * c
        keep = min(e, max(0, (max_elems - tot) // per))
        if keep == 0:
            break
        out.append((keep, r, c))
        tot += keep * per
    return Workload(w.name + "_scaled", out or [w.shapes[0]], w.dp, w.split, dict(w.hp),
                    dict(w.dists), w.transposed, w.note + " (scaled)", dict(w.extra))


# ------------------------------------------------------------------ draws
def _seed(seed, tensor, chunk):
    return (seed * 1_000_003 + {"p": 11, "g": 23, "m": 37, "v": 53}[tensor] * 7919 + chunk) & 0x7FFFFFFF


def _draw(torch, d: Dist, n, gen, device):
    if d.kind == "zeros":
        return torch.zeros(n, dtype=torch.float32, device=device)
    if d.kind == "normal":
        return torch.randn(n, generator=gen, device=device, dtype=torch.float32).mul_(d.a)
    if d.kind == "uniform":
        return torch.rand(n, generator=gen, device=device, dtype=torch.float32).mul_(d.b - d.a).add_(d.a)
    if d.kind == "student_t":
        # t(nu) = z / sqrt(chi2_nu / nu), chi2 with integer nu as a sum of squares
        z = torch.randn(n, generator=gen, device=device, dtype=torch.float32)
        chi = torch.zeros(n, dtype=torch.float32, device=device)
        for _ in range(int(d.b)):
            y = torch.randn(n, generator=gen, device=device, dtype=torch.float32)
            chi.addcmul_(y, y)
        return z.div_(chi.div_(d.b).sqrt_()).mul_(d.a)
    if d.kind == "spiky_normal":
        x = torch.randn(n, generator=gen, device=device, dtype=torch.float32).mul_(d.a)
        hit = torch.rand(n, generator=gen, device=device, dtype=torch.float32) < d.frac
        return torch.where(hit, x * d.mult, x)
    raise ValueError(d.kind)


def fill(out, tensor: str, d: Dist, seed: int, valid_rows=None, valid_cols=None,
         chunk_blocks: int = 4096):
    """Fill a flat float32 torch tensor of nblk*16384 elements (folded layout)
    with i.i.d. draws; elements outside a block's valid rows/cols are zero."""
    import torch
    dev = out.device
    nblk = out.numel() // BLOCK_ELEMS
    view = out.view(nblk, BLOCK, BLOCK)
    for ci, b0 in enumerate(range(0, nblk, chunk_blocks)):
        b1 = min(nblk, b0 + chunk_blocks)
        gen = torch.Generator(device=dev)
        gen.manual_seed(_seed(seed, tensor, ci))
        view[b0:b1] = _draw(torch, d, (b1 - b0) * BLOCK_ELEMS, gen, dev).view(b1 - b0, BLOCK, BLOCK)
    if valid_rows is not None:
        zero_padding(out, valid_rows, valid_cols)
    return out


def zero_padding(out, valid_rows, valid_cols, group: int = 2048):
    """Zero every element (r, c) of block b with r >= valid_rows[b] or c >= valid_cols[b]."""
    import torch
    vr = np.asarray(valid_rows).astype(np.int64)
    vc = np.asarray(valid_cols).astype(np.int64)
    ragged = np.nonzero((vr < BLOCK) | (vc < BLOCK))[0]
    if ragged.size == 0:
        return
    dev = out.device
    view = out.view(-1, BLOCK, BLOCK)
    ar = torch.arange(BLOCK, device=dev)
    for s in range(0, ragged.size, group):
        idx_np = ragged[s:s + group]
        idx = torch.from_numpy(idx_np).to(dev)
        r = torch.from_numpy(vr[idx_np]).to(dev)
        c = torch.from_numpy(vc[idx_np]).to(dev)
        mask = (ar[None, :, None] < r[:, None, None]) & (ar[None, None, :] < c[:, None, None])
        view[idx] = torch.where(mask, view[idx], torch.zeros((), dtype=out.dtype, device=dev))


def make_state(w: Workload, blocks, device, seed: int = 0, capacity_blocks: int | None = None):
    """Allocate and fill p, g, m, v (flat folded float32) for a workload.
    blocks: the planner's block descriptors (numpy, with valid_rows/valid_cols)."""
    import torch
    cap = int(capacity_blocks if capacity_blocks is not None else len(blocks))
    out = {}
    for k in ("p", "g", "m", "v"):
        t = torch.empty(cap * BLOCK_ELEMS, dtype=torch.float32, device=device)
        fill(t, k, w.dists[k], seed, blocks["valid_rows"][:cap], blocks["valid_cols"][:cap])
        out[k] = t
    return out
