"""Whole-step pins for the oracle (CPU only): brute force on tiny tensors,
ragged edges, special blocks, shard-union and layout invariants, and the
column-major copy."""
import numpy as np
import pytest

from _defs import adamw_error_bounds, adamw_fp64, brute_force_encode

BLK = 16384


def _setup(oracle, shapes, dp=1, split=0, seed=0, state=True, spike=None, zero=False):
    params, shards, blocks, summ = oracle.plan_shards(shapes, dp, split)
    cap = int(summ["capacity_blocks"])
    rng = np.random.default_rng(seed)
    bufs = {k: np.zeros(cap * BLK, np.float32) for k in "pgmv"}
    for i, (E, H, W) in enumerate(shapes):
        vals = {
            "p": rng.normal(0, 0.02, (E, H, W)),
            "g": rng.normal(0, 1e-3, (E, H, W)),
            "m": rng.normal(0, 3e-4, (E, H, W)) if state else np.zeros((E, H, W)),
            "v": rng.uniform(0.5, 1.5, (E, H, W)) * 1e-6 if state else np.zeros((E, H, W)),
        }
        if zero:
            vals = {k: np.zeros((E, H, W)) for k in vals}
        if spike is not None and i == 0:
            vals["g"].flat[spike] = 0.5
            vals["p"].flat[spike] = 1.5
        off = int(params[i]["blk_offset"]) * BLK
        n = E * (-(-H // 128)) * (-(-W // 128)) * BLK
        for k in "pgmv":
            bufs[k][off:off + n] = oracle.fold(vals[k].astype(np.float32)).ravel()
    return params, shards, blocks, summ, bufs


def _run(oracle, params, blocks, bufs, hp, b0, nb, transposed=False, t_bytes=None, t_scales=None):
    cap = len(bufs["p"]) // BLK
    q = np.zeros(cap * BLK, np.uint8)
    inv = np.zeros(cap, np.float32)
    out = {k: bufs[k].copy() for k in "pgmv"}
    wt = it = None
    if transposed:
        wt = np.zeros(t_bytes, np.uint8)
        it = np.zeros(t_scales, np.float32)
    oracle.adamw_requant_step(out["p"], out["g"], out["m"], out["v"], q, inv, b0, nb, hp,
                              desc=blocks, params=params, w_fp8_t=wt, inv_scale_t=it)
    return out, q, inv, wt, it


TINY = [[(1, 1, 1)], [(1, 1, 129)], [(1, 129, 1)], [(1, 128, 128)], [(2, 130, 257)],
        [(1, 256, 384)], [(1, 3, 5), (2, 128, 1), (1, 200, 200)]]


@pytest.mark.parametrize("shapes", TINY)
@pytest.mark.parametrize("step", [1, 11])
def test_tiny_brute_force(oracle, shapes, step):
    params, shards, blocks, summ, bufs = _setup(oracle, shapes, state=step > 1, seed=step)
    hp = oracle.Hparams.make(step=step)
    B = int(summ["total_blocks"])
    t_bytes = int(sum(e * h * w for e, h, w in shapes))
    t_scales = int(sum(p["e"] * p["hb"] * p["wb"] for p in params))
    out, q, inv, wt, it = _run(oracle, params, blocks, bufs, hp, 0, B, True, t_bytes, t_scales)
    valid = np.zeros(B * BLK, bool)
    for b in range(B):
        vr, vc = int(blocks[b]["valid_rows"]), int(blocks[b]["valid_cols"])
        m2 = np.zeros((128, 128), bool)
        m2[:vr, :vc] = True
        valid[b * BLK:(b + 1) * BLK] = m2.ravel()
    sl = slice(0, B * BLK)
    # (a) element update against the float64 definition
    pd, md, vd = adamw_fp64(hp, bufs["p"][sl], bufs["g"][sl], bufs["m"][sl], bufs["v"][sl])
    bp, bm, bv = adamw_error_bounds(hp, bufs["p"][sl], bufs["g"][sl], bufs["m"][sl], bufs["v"][sl])
    for got, want, bound in ((out["p"], pd, bp), (out["m"], md, bm), (out["v"], vd, bv)):
        assert np.all(np.abs(got[sl][valid] - want[valid]) <= bound[valid])
        assert not np.any(got[sl][~valid])                     # padding stays zero
    # (b) scale from the page rule, (c) codes by brute force
    for b in range(B):
        blk = out["p"][b * BLK:(b + 1) * BLK]
        amax = np.max(np.abs(blk))
        s = np.float32(1) if amax == 0 else np.float32(448) / amax
        assert inv[b] == np.float32(1) / s
        want_q = brute_force_encode(blk * s)
        want_q[~valid[b * BLK:(b + 1) * BLK]] = 0
        assert np.array_equal(q[b * BLK:(b + 1) * BLK], want_q)
    # (e) column-major copy and transposed scale grid
    for i, (E, H, W) in enumerate(shapes):
        pe = params[i]
        nb = E * int(pe["hb"]) * int(pe["wb"])
        o = int(pe["blk_offset"])
        qq = oracle.unfold(q[o * BLK:(o + nb) * BLK].astype(np.float32).reshape(nb, 128, 128), E, H, W)
        t0 = int(pe["t_offset"])
        assert np.array_equal(wt[t0:t0 + E * H * W].reshape(E, W, H), qq.transpose(0, 2, 1).astype(np.uint8))
        s0 = int(pe["t_scale_offset"])
        grid = inv[o:o + nb].reshape(E, int(pe["hb"]), int(pe["wb"]))
        assert np.array_equal(it[s0:s0 + nb].reshape(E, int(pe["wb"]), int(pe["hb"])), grid.transpose(0, 2, 1))


def test_all_zero_and_spike_blocks(oracle):
    params, shards, blocks, summ, bufs = _setup(oracle, [(1, 256, 256)], zero=True)
    out, q, inv, _, _ = _run(oracle, params, blocks, bufs, oracle.Hparams.make(), 0, 4)
    assert np.all(inv == 1) and not np.any(q) and not np.any(out["p"])
    params, shards, blocks, summ, bufs = _setup(oracle, [(1, 256, 256)], spike=5 * 256 + 9)
    out, q, inv, _, _ = _run(oracle, params, blocks, bufs, oracle.Hparams.make(), 0, 4)
    k = 5 * 128 + 9                                   # block 0, row 5, col 9
    assert q[k] == 0x7E
    # the spike (p = 1.5) sets block 0's scale, ~17x coarser than its neighbours
    assert inv[0] > 10 * inv[1]


@pytest.mark.parametrize("dp", [1, 2, 3, 8, 16])
def test_union_of_shards_equals_unsharded(oracle, dp):
    shapes = [(1, 384, 640), (2, 129, 300), (1, 7, 1000)]
    params, shards, blocks, summ, bufs = _setup(oracle, shapes, dp=dp, seed=dp)
    hp = oracle.Hparams.make(step=3)
    cap = int(summ["capacity_blocks"])
    whole = _run(oracle, params, blocks, bufs, hp, 0, cap)
    out = {k: bufs[k].copy() for k in "pgmv"}
    q = np.zeros(cap * BLK, np.uint8)
    inv = np.zeros(cap, np.float32)
    for s in shards:
        oracle.adamw_requant_step(out["p"], out["g"], out["m"], out["v"], q, inv,
                                  int(s["blk_begin"]), int(s["blk_count_real"]), hp, desc=blocks)
    for k in "pmv":
        assert np.array_equal(out[k], whole[0][k])
    assert np.array_equal(q, whole[1])
    data = np.repeat(blocks["param"] >= 0, 1)
    assert np.array_equal(inv[data], whole[2][data])


def test_paramwise_and_blockwise_give_identical_params(oracle):
    shapes = [(1, 300, 200), (1, 128, 128), (2, 256, 130), (1, 64, 700)]
    hp = oracle.Hparams.make(step=7)
    results = []
    for split in (0, 1):
        params, shards, blocks, summ = oracle.plan_shards(shapes, 3, split)
        cap = int(summ["capacity_blocks"])
        bufs = {k: np.zeros(cap * BLK, np.float32) for k in "pgmv"}
        rng = np.random.default_rng(99)
        per = []
        for i, (E, H, W) in enumerate(shapes):
            off = int(params[i]["blk_offset"]) * BLK
            for k, sd in zip("pgmv", (0.02, 1e-3, 3e-4, 1e-6)):
                x = rng.normal(0, sd, (E, H, W)) if k != "v" else rng.uniform(0.5, 1.5, (E, H, W)) * sd
                f = oracle.fold(x.astype(np.float32)).ravel()
                bufs[k][off:off + f.size] = f
        out, q, inv, _, _ = _run(oracle, params, blocks, bufs, hp, 0, cap)
        for i, (E, H, W) in enumerate(shapes):
            pe = params[i]
            nb = E * int(pe["hb"]) * int(pe["wb"])
            o = int(pe["blk_offset"])
            per.append((oracle.unfold(out["p"][o * BLK:(o + nb) * BLK].reshape(nb, 128, 128), E, H, W),
                        q[o * BLK:(o + nb) * BLK].copy(), inv[o:o + nb].copy()))
        results.append(per)
    for a, b in zip(*results):
        assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1]) and np.array_equal(a[2], b[2])


def test_standalone_transpose_and_involution(oracle):
    shapes = [(2, 300, 260)]
    params, shards, blocks, summ, bufs = _setup(oracle, shapes, seed=4)
    out, q, inv, _, _ = _run(oracle, params, blocks, bufs, oracle.Hparams.make(), 0, int(summ["total_blocks"]))
    t, it = oracle.transpose_fp8(q, inv, params[0])
    E, H, W = shapes[0]
    qq = oracle.unfold(q.astype(np.float32).reshape(-1, 128, 128), E, H, W).astype(np.uint8)
    assert np.array_equal(t, qq.transpose(0, 2, 1))
    # transpose of the transpose: fold the [E,W,H] copy and transpose again
    tp, _, tb, _ = oracle.plan_shards([(E, W, H)], 1, 0)
    tf = oracle.fold(t.astype(np.float32)).ravel().astype(np.uint8)
    back, inv_back = oracle.transpose_fp8(tf, it.ravel().copy(), tp[0])
    assert np.array_equal(back, qq)
    assert np.array_equal(inv_back.ravel(), inv[:E * 3 * 3])
