"""Pins for the oracle's MXFP8 output variant (E8M0 scale per 32 elements of a
block row; "A ZeRO Optimizer Design for Blockwise FP8 Quantization",
"Blockwise quantization" on MXFP8, mhpn.cn "Core scaling strategies in FP8
training" §3.1)."""
import numpy as np

from _defs import brute_force_encode

BLK = 16384


def _state(rng, nblk, spike=True):
    p = rng.normal(0, 0.02, nblk * BLK).astype(np.float32)
    g = rng.normal(0, 1e-3, nblk * BLK).astype(np.float32)
    m = rng.normal(0, 2e-4, nblk * BLK).astype(np.float32)
    v = (rng.uniform(0.5, 1.5, nblk * BLK) * 4e-7).astype(np.float32)
    if spike:
        p[5 * 128 + 40] = 3.0            # block 0, row 5, group 1
        p[BLK:BLK + 128 * 3] *= 1e-6     # block 1, rows 0-2: tiny values
        p[2 * BLK:2 * BLK + 64] = 0.0    # block 2, row 0, groups 0-1: zero ...
        g[2 * BLK:2 * BLK + 64] = 0.0
        m[2 * BLK:2 * BLK + 64] = 0.0
        v[2 * BLK:2 * BLK + 64] = 0.0
    return p, g, m, v


def test_mx_step_definition(oracle):
    rng = np.random.default_rng(0)
    nblk = 3
    p, g, m, v = _state(rng, nblk)
    hp = oracle.Hparams.make(step=4)
    # the AdamW part is the block-scaled step's
    pb, gb, mb, vb = (a.copy() for a in (p, g, m, v))
    oracle.adamw_requant_step(pb, gb, mb, vb, np.zeros(nblk * BLK, np.uint8), np.zeros(nblk, np.float32),
                              0, nblk, hp)
    q = np.zeros(nblk * BLK, np.uint8)
    sc = np.zeros(nblk * 512, np.uint8)
    oracle.adamw_requant_step_mx(p, g, m, v, q, sc, 0, nblk, hp)
    assert np.array_equal(p, pb) and np.array_equal(m, mb) and np.array_equal(v, vb)
    groups = p.reshape(-1, 32)
    amax = np.max(np.abs(groups), axis=1)
    X = 2.0 ** (sc.astype(np.float64) - 127)
    nz = amax > 0
    ratio = amax[nz] / X[nz]
    assert np.all((ratio >= 256) & (ratio < 512))          # the largest element lands in [256, 512)
    assert np.all(sc[~nz] == 127)
    want = brute_force_encode((groups / X[:, None].astype(np.float64)).astype(np.float32).ravel())
    assert np.array_equal(q, want)
    dec = oracle.e4m3_decode(q).reshape(-1, 32) * X[:, None]
    err = np.abs(dec - groups)
    sat = np.abs(groups / X[:, None]) > 448
    # half an E4M3 spacing (<= 16 at the top binade) times the scale, or the saturation gap
    assert np.all(err[~sat] <= 16 * np.broadcast_to(X[:, None], err.shape)[~sat])
    assert np.all(err[sat] <= 64 * np.broadcast_to(X[:, None], err.shape)[sat])


def test_mx_spike_only_moves_its_group(oracle):
    rng = np.random.default_rng(1)
    p, g, m, v = _state(rng, 1, spike=False)
    hp = oracle.Hparams.make(step=2)
    q0 = np.zeros(BLK, np.uint8)
    s0 = np.zeros(512, np.uint8)
    a = [x.copy() for x in (p, g, m, v)]
    oracle.adamw_requant_step_mx(*a, q0, s0, 0, 1, hp)
    p[5 * 128 + 40] = 3.0
    q1 = np.zeros(BLK, np.uint8)
    s1 = np.zeros(512, np.uint8)
    oracle.adamw_requant_step_mx(p, g, m, v, q1, s1, 0, 1, hp)
    changed = np.nonzero(s0 != s1)[0]
    assert list(changed) == [5 * 4 + 1]                    # row 5, group 1 only


def test_mx_infinite_amax(oracle):
    """An infinite p' makes its group's amax +Inf: floor(log2 amax) - 8 is then
    +Inf, clamped to 127 (scale byte 254); the Inf element saturates to the
    +-448 code, the group's finite elements (|p'| << 2^127) round to a signed
    zero, and every other group keeps the finite rule."""
    rng = np.random.default_rng(3)
    p, g, m, v = _state(rng, 1, spike=False)
    p[7 * 128 + 70] = np.inf                 # row 7, group 2
    p[9 * 128 + 3] = -np.inf                 # row 9, group 0
    q = np.zeros(BLK, np.uint8)
    sc = np.zeros(512, np.uint8)
    ref = [x.copy() for x in (p, g, m, v)]
    oracle.adamw_requant_step_mx(p, g, m, v, q, sc, 0, 1, oracle.Hparams.make(step=3))
    assert sc[7 * 4 + 2] == 254 and sc[9 * 4 + 0] == 254
    assert q[7 * 128 + 70] == 0x7E and q[9 * 128 + 3] == 0xFE
    for r, gi in ((7, 2), (9, 0)):
        grp = q[r * 128 + gi * 32:r * 128 + gi * 32 + 32]
        fin = np.isfinite(p[r * 128 + gi * 32:r * 128 + gi * 32 + 32])
        assert np.all((grp[fin] & 0x7F) == 0)
    # the other groups: same bytes as a run without the infinities
    p0, g0, m0, v0 = ref
    p0[7 * 128 + 70] = 0.0
    p0[9 * 128 + 3] = 0.0
    q0 = np.zeros(BLK, np.uint8)
    s0 = np.zeros(512, np.uint8)
    oracle.adamw_requant_step_mx(p0, g0, m0, v0, q0, s0, 0, 1, oracle.Hparams.make(step=3))
    keep = np.ones(512, bool)
    keep[[7 * 4 + 2, 9 * 4 + 0]] = False
    assert np.array_equal(sc[keep], s0[keep])
    assert np.array_equal(q.reshape(512, 32)[keep], q0.reshape(512, 32)[keep])


def test_mx_padding_and_desc(oracle):
    shapes = [(1, 200, 100)]                                # ragged rows and cols
    params, shards, blocks, summ = oracle.plan_shards(shapes, 1, 0)
    rng = np.random.default_rng(2)
    nblk = int(summ["total_blocks"])
    x = {k: oracle.fold(rng.normal(0, s, (1, 200, 100)).astype(np.float32)).ravel()
         for k, s in zip("pgm", (0.02, 1e-3, 2e-4))}
    x["v"] = oracle.fold((rng.uniform(0.5, 1.5, (1, 200, 100)) * 4e-7).astype(np.float32)).ravel()
    q = np.zeros(nblk * BLK, np.uint8)
    sc = np.zeros(nblk * 512, np.uint8)
    oracle.adamw_requant_step_mx(x["p"], x["g"], x["m"], x["v"], q, sc, 0, nblk,
                                 oracle.Hparams.make(step=3), desc=blocks)
    blk1 = q[BLK:2 * BLK].reshape(128, 128)                 # block row 1: 72 valid rows
    assert not np.any(blk1[72:]) and not np.any(blk1[:, 100:])
    s1 = sc[512:1024].reshape(128, 4)
    assert np.all(s1[72:] == 127)                           # padding rows: all-zero groups
    assert np.all(s1[:72, 3] != 127)                        # cols 96..99 of group 3 are real


def test_mx_group_max_above_448_saturates_and_ignores_block_knobs(oracle):
    """The shared exponent is floor(log2 amax) - 8 (the OCP MX rule: the largest
    element's binade is put at E4M3's top binade, [256, 512)).  A group whose
    largest element has significand above 1.75 therefore lands in (448, 512)
    and saturates to the 448 code, up to ~12.5 % low; fp8_max and min_scale,
    the block-scaled step's knobs, do not enter.  lr = 0 keeps p' = p, so the
    group's values are set directly."""
    rng = np.random.default_rng(4)
    p, g, m, v = _state(rng, 1, spike=False)
    row = 3
    grp = p[row * 128 + 32: row * 128 + 64]                # row 3, group 1
    grp[:] = rng.uniform(-1.0, 1.0, 32).astype(np.float32) * 2.0 ** -5
    grp[17] = np.float32(1.9 * 2.0 ** -3)                   # significand 1.9 > 1.75, binade 2^-3
    grp[4] = np.float32(-1.99 * 2.0 ** -4)                  # below the group max
    runs = []
    for kw in (dict(), dict(fp8_max=100.0, min_scale=1e3), dict(fp8_max=448.0, min_scale=0.0, scale_mode=1)):
        hp = oracle.Hparams.make(lr=0.0, weight_decay=0.0, step=5, **kw)
        a = [x.copy() for x in (p, g, m, v)]
        q = np.zeros(BLK, np.uint8)
        sc = np.zeros(512, np.uint8)
        oracle.adamw_requant_step_mx(*a, q, sc, 0, 1, hp)
        assert np.array_equal(a[0], p)                      # lr = 0: p' = p
        runs.append((q, sc))
    q, sc = runs[0]
    assert sc[row * 4 + 1] == 127 + (-3 - 8)                # x = floor(log2(1.9 * 2^-3)) - 8 = -11
    assert q[row * 128 + 32 + 17] == 0x7E                   # 1.9 * 2^8 = 486.4 -> saturates to 448
    assert oracle.e4m3_decode(q[row * 128 + 32 + 17:row * 128 + 32 + 18])[0] * 2.0 ** -11 == 448 * 2.0 ** -11
    # -1.99 * 2^-4 / 2^-11 = -254.72 -> nearest E4M3 (spacing 16 in [256, 512), 8 in [128, 256)): -256
    assert q[row * 128 + 32 + 4] == 0xF8
    for q2, s2 in runs[1:]:
        assert np.array_equal(q2, q) and np.array_equal(s2, sc)
