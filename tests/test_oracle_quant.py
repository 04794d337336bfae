"""Pins for the oracle's per-block scale, quantize and dequantize (CPU only)."""
import os

import numpy as np
import pytest
import torch

from _defs import EPS32, e4m3_quantum

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _step_one_block(oracle, p, g=None, m=None, v=None, hp=None):
    n = p.size
    z = np.zeros(n, np.float32)
    p = p.astype(np.float32).ravel().copy()
    g = z.copy() if g is None else g.astype(np.float32).ravel().copy()
    m = z.copy() if m is None else m.astype(np.float32).ravel().copy()
    v = z.copy() if v is None else v.astype(np.float32).ravel().copy()
    nblk = n // oracle.BLK_ELEMS
    q = np.zeros(n, np.uint8)
    inv = np.zeros(nblk, np.float32)
    hp = hp or oracle.Hparams.make()
    oracle.adamw_requant_step(p, g, m, v, q, inv, 0, nblk, hp)
    return p, q, inv


def test_golden_scale_cases(oracle):
    rows = [l.split() for l in open(os.path.join(GOLDEN, "scale_cases.txt"))
            if l.strip() and not l.startswith("#")]
    assert len(rows) == 8
    for a, s, inv in rows:
        got_s, got_inv = oracle.block_scale(np.float32(float(a)))
        assert got_s == np.float32(float(s)), (a, got_s)
        assert got_inv == np.float32(float(inv)), (a, got_inv)


def test_amax_element_quantizes_to_448(oracle):
    rng = np.random.default_rng(3)
    for trial in range(20):
        x = (rng.standard_t(3, size=oracle.BLK_ELEMS) * 10.0 ** rng.uniform(-6, 3)).astype(np.float32)
        s, inv = oracle.block_scale(np.max(np.abs(x)))
        q = oracle.e4m3_encode(x * s)
        k = np.argmax(np.abs(x))
        assert q[k] == (0xFE if x[k] < 0 else 0x7E)
        assert np.all(np.abs(oracle.e4m3_decode(q)) <= 448)


def test_zero_block_scale_one_and_zero_codes(oracle):
    p = np.zeros(oracle.BLK_ELEMS, np.float32)
    p1, q, inv = _step_one_block(oracle, p)
    assert inv[0] == 1.0 and not np.any(q) and not np.any(p1)


def test_min_scale_floor_saturates(oracle):
    # amax 1e9: 448/amax = 4.48e-7 < 1e-6, the floor binds (mhpn.cn §4.2)
    x = np.float32([1e9, 5e8, 1e8, 1.0])
    s, inv = oracle.block_scale(np.float32(1e9))
    assert s == np.float32(1e-6)
    q = oracle.e4m3_encode(x * s)
    assert q[0] == 0x7E and q[1] == 0x7E           # 1000, 500 -> saturate to 448
    assert oracle.e4m3_decode(q[2]) == 96.0        # 100 -> nearest is 96


def test_dequant_error_bound(oracle):
    rng = np.random.default_rng(11)
    nblk = 6
    p = rng.normal(0, 0.02, nblk * oracle.BLK_ELEMS).astype(np.float32)
    g = rng.normal(0, 1e-3, p.size).astype(np.float32)
    p1, q, inv = _step_one_block(oracle, p, g)
    xh = oracle.dequant(q, inv, nblk)
    y = p1.astype(np.float64) * np.repeat([oracle.block_scale(np.max(np.abs(b)))[0]
                                           for b in p1.reshape(nblk, -1)], oracle.BLK_ELEMS)
    bound = 0.5 * e4m3_quantum(y) * np.repeat(inv.astype(np.float64), oracle.BLK_ELEMS) \
        * (1 + 2 * EPS32) + EPS32 * np.abs(xh) + 1e-45
    assert np.all(np.abs(xh.astype(np.float64) - p1) <= bound)


def test_same_layout_requant_is_idempotent(oracle):
    """Q(D(Q(x))) = Q(x) ("FP8-Flow-MoE" §3.1, same layout, deterministic RtN)."""
    rng = np.random.default_rng(12)
    x = (rng.standard_t(3, size=oracle.BLK_ELEMS) * 1e-3).astype(np.float32)
    s, inv = oracle.block_scale(np.max(np.abs(x)))
    q = oracle.e4m3_encode(x * s)
    xh = (oracle.e4m3_decode(q).astype(np.float32) * inv).astype(np.float32)
    assert np.array_equal(oracle.e4m3_encode(xh * s), q)
    # recomputed amax: the scale may move by an ulp, the codes do not
    s2, inv2 = oracle.block_scale(np.max(np.abs(xh)))
    assert abs(float(s2) - float(s)) <= float(np.spacing(s))
    assert np.array_equal(oracle.e4m3_encode(xh * s2), q)


def test_pow2_scale_and_exponent_shift_is_exact(oracle):
    """With s = 2^T, a layout change is a pure exponent shift: E' = E - D,
    M' = M ("FP8-Flow-MoE" §3.1, power-of-two scales)."""
    for a in [1.0, 0.3, 448.0, 449.0, 1e-3, 3e-7, 7.1e4]:
        s, inv = oracle.block_scale(np.float32(a), scale_mode=1)
        k = np.log2(float(s))
        assert k == np.round(k)                               # power of two
        assert float(s) * np.float32(a) <= 448.0              # no saturation
        assert 2 * float(s) * np.float32(a) > 448.0           # largest such power
        assert float(inv) * float(s) == 1.0
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F and ((c >> 3) & 15) >= 2],
                     dtype=np.uint8)
    vals = oracle.e4m3_decode(codes).astype(np.float32)
    shifted = oracle.e4m3_encode(vals * np.float32(0.5))     # D = 1
    assert np.array_equal(shifted, codes - 8)                 # exponent field - 1, same M
    # back again: the round trip is exact
    assert np.array_equal(oracle.e4m3_encode(oracle.e4m3_decode(shifted).astype(np.float32) * 2),
                          codes)


def test_block_quantize_against_library_cast(oracle):
    """128x128 block quantize as in mhpn.cn §3.2 (scale = 448/amax, clamp to
    ±448), here done with torch ops and torch's E4M3 cast."""
    rng = np.random.default_rng(13)
    H, W = 256, 384
    x = rng.normal(0, 0.02, (H, W)).astype(np.float32)
    x[5, 7] = 0.4     # a spike in block (0, 0)
    t = torch.from_numpy(x)
    want_q = torch.empty((H, W), dtype=torch.uint8)
    want_s = torch.empty((H // 128, W // 128))
    for i in range(0, H, 128):
        for j in range(0, W, 128):
            blk = t[i:i + 128, j:j + 128]
            sc = torch.tensor(448.0) / blk.abs().max()
            want_s[i // 128, j // 128] = sc
            want_q[i:i + 128, j:j + 128] = (blk * sc).clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8)
    blocks = oracle.fold(x).reshape(-1)
    nblk = blocks.size // oracle.BLK_ELEMS
    q = np.zeros(blocks.size, np.uint8)
    inv = np.zeros(nblk, np.float32)
    for b in range(nblk):
        blk = blocks[b * oracle.BLK_ELEMS:(b + 1) * oracle.BLK_ELEMS]
        s, inv[b] = oracle.block_scale(np.max(np.abs(blk)))
        assert s == want_s.reshape(-1)[b].item()
        q[b * oracle.BLK_ELEMS:(b + 1) * oracle.BLK_ELEMS] = oracle.e4m3_encode(blk * s)
    got = oracle.unfold(q.astype(np.float32).reshape(nblk, 128, 128), 1, H, W)[0]
    assert np.array_equal(got.astype(np.uint8), want_q.numpy())
