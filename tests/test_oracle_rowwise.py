"""Pins for the oracle's 1x128 row-wise quantizer and scaling-aware transpose
("FP8-Flow-MoE: A Casting-Free FP8 Recipe without Double Quantization
Error", §3.1), and the double-quantization error the transpose avoids."""
import numpy as np
import pytest

from _defs import brute_force_encode, finite_e4m3_table


def _act(rng, R, C, outliers=True):
    x = rng.normal(0, 1, (R, C)).astype(np.float32)
    if outliers:
        hit = rng.random((R, C)) < 1e-3
        x[hit] *= 60.0
    x[:, :128] *= 1e-3                       # one very small column tile
    return x


@pytest.mark.parametrize("pow2", [True, False])
def test_rowwise_quantizer_definition(oracle, pow2):
    rng = np.random.default_rng(1)
    x = _act(rng, 64, 384)
    x[3, 128:256] = 0.0                       # an all-zero tile
    q, s = oracle.quantize_rowwise(x, pow2=pow2)
    for r in range(64):
        for t in range(3):
            tile = x[r, t * 128:(t + 1) * 128]
            amax = np.max(np.abs(tile))
            sc = s[r, t]
            if amax == 0:
                assert sc == 1.0
            elif pow2:
                k = np.log2(float(sc))
                assert k == np.round(k)                        # a power of two
                assert amax / float(sc) <= 448.0 < amax / (float(sc) / 2)   # the smallest one
            else:
                assert sc == np.float32(amax / np.float32(448.0))
            want = brute_force_encode((tile / sc).astype(np.float32))
            assert np.array_equal(q[r, t * 128:(t + 1) * 128], want)


def test_same_layout_requant_is_idempotent(oracle):
    """Q_row(D(Q_row(X))) = Q_row(X) (the page's same-layout argument, which
    holds the scale fixed).  With power-of-two scales the recomputed scale can
    halve when a tile's largest value rounded down to exactly 224; the values
    are then unchanged and the codes are the same values one exponent up."""
    rng = np.random.default_rng(2)
    x = _act(rng, 128, 512)
    for pow2 in (True, False):
        q, s = oracle.quantize_rowwise(x, pow2=pow2)
        v = oracle.dequant_rowwise(q, s)
        q2, s2 = oracle.quantize_rowwise(v, pow2=pow2)
        assert np.array_equal(oracle.dequant_rowwise(q2, s2), v)
        same = np.repeat(s2 == s, 128, axis=1)
        assert same.mean() > 0.95
        assert np.array_equal(q2[same], q[same])
        if pow2:
            assert np.all(s2[s2 != s] * 2 == s[s2 != s])
            sn, E, M = _fields(q[~same])
            sn2, E2, M2 = _fields(q2[~same])
            nz = E >= 1
            assert np.array_equal(E2[nz], E[nz] + 1) and np.array_equal(M2[nz], M[nz])


def _fields(code):
    code = np.asarray(code, np.int64)
    return (code >> 7) & 1, (code >> 3) & 15, code & 7


def test_transpose_is_an_exponent_shift_with_pow2_scales(oracle):
    """E' = E - D, M' = M, SN' = SN and value preserved, wherever no underflow."""
    rng = np.random.default_rng(3)
    x = _act(rng, 256, 384)
    q, s = oracle.quantize_rowwise(x, pow2=True)
    qt, st = oracle.transpose_rowwise(q, s)
    R, C = q.shape
    v_row = oracle.dequant_rowwise(q, s)                      # exact values of the row layout
    v_col = oracle.dequant_rowwise(qt, st).T
    sn, E, M = _fields(q)
    snt, Et, Mt = _fields(qt.T)
    s_full = np.repeat(s, 128, axis=1)
    st_full = np.repeat(st, 128, axis=1).T
    D = np.log2(st_full.astype(np.float64)) - np.log2(s_full.astype(np.float64))
    assert np.all(D >= 0) and np.all(D == np.round(D))
    normal = (E >= 1) & (E - D >= 1)
    assert normal.mean() > 0.9
    assert np.array_equal(Et[normal], (E - D)[normal].astype(np.int64))
    assert np.array_equal(Mt[normal], M[normal]) and np.array_equal(snt[normal], sn[normal])
    assert np.array_equal(v_col[normal], v_row[normal])
    # every output tile row carries the tile's largest row scale
    for i in range(R // 128):
        for j in range(C // 128):
            assert np.all(st[j * 128:(j + 1) * 128, i] == s[i * 128:(i + 1) * 128, j].max())


@pytest.mark.parametrize("pow2", [True, False])
def test_transpose_matches_definition_including_underflow(oracle, pow2):
    """Each transposed code is the nearest E4M3 value (brute force) to
    decode(q) * (s_r / s'), the ratio rounded once to float32 (a float64
    quotient of two floats rounds to the correctly rounded float quotient) and
    the product once more; with amax/448 scales the ratios are not powers of
    two, so almost every code is re-rounded."""
    rng = np.random.default_rng(4)
    x = _act(rng, 128, 256)
    x[7] *= 1e4                                # one row with a much larger scale
    q, s = oracle.quantize_rowwise(x, pow2=pow2)
    qt, st = oracle.transpose_rowwise(q, s)
    dec = finite_e4m3_table()
    vals = np.where(q & 0x80, -1.0, 1.0) * dec[q & 0x7F]
    ratio = (np.repeat(s, 128, axis=1) / np.repeat(st, 128, axis=1).T).astype(np.float32)
    want = brute_force_encode((vals.astype(np.float32) * ratio).astype(np.float32))
    assert np.array_equal(qt.T, want)


def test_double_quantization_error(oracle):
    """E = Q_col(D(Q_row(X))) - Q_col(X).  With scales amax/448 the naive
    dequantize -> transpose -> requantize path rounds almost every value a
    second time and its error against X exceeds that of quantizing X
    column-wise directly; with power-of-two scales a change of layout only
    moves exponents, so the transposed values equal the row-layout values
    except where they underflow, and the error equals the direct one."""
    rng = np.random.default_rng(5)
    x = _act(rng, 512, 512)
    xt = np.ascontiguousarray(x.T)
    rel = lambda y: np.abs(y - xt).sum() / np.abs(xt).sum()
    # amax/448 scales: the double quantization error
    q, s = oracle.quantize_rowwise(x, pow2=False)
    v_row = oracle.dequant_rowwise(q, s)
    naive = oracle.dequant_rowwise(*oracle.quantize_rowwise(np.ascontiguousarray(v_row.T), pow2=False))
    ref = oracle.dequant_rowwise(*oracle.quantize_rowwise(xt, pow2=False))
    assert np.mean(naive != v_row.T) > 0.5
    assert rel(naive) > 1.2 * rel(ref)
    # power-of-two scales: no second rounding outside underflow
    q, s = oracle.quantize_rowwise(x, pow2=True)
    v_row = oracle.dequant_rowwise(q, s)
    qt, st = oracle.transpose_rowwise(q, s)
    direct = oracle.dequant_rowwise(qt, st)
    naive = oracle.dequant_rowwise(*oracle.quantize_rowwise(np.ascontiguousarray(v_row.T), pow2=True))
    ref = oracle.dequant_rowwise(*oracle.quantize_rowwise(xt, pow2=True))
    moved = direct != v_row.T
    _, E, _ = _fields(q.T)
    D = (np.log2(np.repeat(st, 128, axis=1).astype(np.float64))
         - np.log2(np.repeat(s, 128, axis=1).T.astype(np.float64)))
    assert np.all((E - D)[moved] < 1)                 # only underflowed values move
    assert np.mean(moved) < 0.01 and np.mean(naive != v_row.T) < 0.01
    assert abs(rel(direct) - rel(ref)) < 1e-3 * rel(ref)


def test_infinite_tile_amax_takes_the_clamp(oracle):
    """Power-of-two scales: a tile holding an Inf has amax/448 = Inf, whose
    smallest power of two above it is out of range: the scale is the clamp,
    2^127; the Inf saturates to the +-448 code and the finite values round to
    a signed zero.  Other tiles keep the finite rule."""
    rng = np.random.default_rng(8)
    x = _act(rng, 4, 384, outliers=False)
    x[1, 130] = np.inf
    x[2, 300] = -np.inf
    q, s = oracle.quantize_rowwise(x, pow2=True)
    assert s[1, 1] == np.float32(2.0 ** 127) and s[2, 2] == np.float32(2.0 ** 127)
    assert q[1, 130] == 0x7E and q[2, 300] == 0xFE
    fin = np.isfinite(x[1, 128:256])
    assert np.all((q[1, 128:256][fin] & 0x7F) == 0)
    x0 = x.copy()
    x0[1, 130] = 0.0
    x0[2, 300] = 0.0
    q0, s0 = oracle.quantize_rowwise(x0, pow2=True)
    keep = np.ones_like(s, bool)
    keep[1, 1] = keep[2, 2] = False
    assert np.array_equal(s[keep], s0[keep])
