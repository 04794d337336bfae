"""Pins for the oracle's E4M3 encoder/decoder (CPU only).

The encoder must round to the nearest E4M3 value with ties to the even
mantissa ("FP8-Flow-MoE" §3.1: scaled values are mapped to the nearest discrete
value, deterministic round-to-nearest) and saturate to ±448 (mhpn.cn "Core
scaling strategies in FP8 training" §3.2 clamp).  It is checked against
(i) a brute-force nearest search over the 127 finite non-negative codes decoded
by the page's value formula and (ii) torch's float8_e4m3fn cast (a library
routine) wherever that cast is defined (|x| < 464).
"""
import os

import numpy as np
import pytest
import torch

from _defs import brute_force_encode, finite_e4m3_table as _finite_table

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _interesting_floats():
    t = _finite_table().astype(np.float32)
    mids = ((t[1:].astype(np.float64) + t[:-1]) / 2).astype(np.float32)
    assert np.all(mids.astype(np.float64) == (t[1:].astype(np.float64) + t[:-1]) / 2)
    base = np.concatenate([t, mids, np.float32([448, 456, 460, 463.99997, 464, 470, 480, 1e4,
                                                2.0 ** -10, 2.0 ** -11, 3 * 2.0 ** -11])])
    b = base.view(np.uint32)
    nb = np.concatenate([b, b + 1, b - 1, b + 2, b - 2]).astype(np.uint32)
    nb = nb[nb < 0x7F800000]
    pos = nb.view(np.float32)
    return np.concatenate([pos, -pos])


def test_golden_codes_match_formula(oracle):
    rows = [l.split() for l in open(os.path.join(GOLDEN, "e4m3_codes.txt"))
            if l.strip() and not l.startswith("#")]
    assert len(rows) >= 20
    for code_s, val_s in rows:
        code = int(code_s, 16)
        got = oracle.e4m3_decode(code)
        if val_s == "nan":
            assert np.isnan(got), code_s
        else:
            want = float(val_s)
            assert got == want and np.signbit(got) == np.signbit(want), (code_s, got, want)
            if code not in (0x00, 0x80):
                assert oracle.e4m3_encode(np.float32([want]))[0] == code


def test_decode_table_is_the_formula(oracle):
    dec = oracle.e4m3_decode(np.arange(256))
    table = _finite_table()
    assert np.array_equal(dec[:127], table)
    assert np.array_equal(dec[128:255], -table)
    assert np.isnan(dec[127]) and np.isnan(dec[255])
    assert dec[126] == 448.0


def test_roundtrip_every_finite_code(oracle):
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    vals = oracle.e4m3_decode(codes).astype(np.float32)
    back = oracle.e4m3_encode(vals)
    want = codes.copy()
    assert np.array_equal(back, want)


def test_encode_matches_brute_force_on_midpoints_and_neighbours(oracle):
    x = _interesting_floats()
    assert np.array_equal(oracle.e4m3_encode(x), brute_force_encode(x))


def test_encode_matches_brute_force_on_random_and_coarse_grid(oracle):
    rng = np.random.default_rng(1234)
    rnd = rng.integers(0, 2 ** 32, size=1 << 18, dtype=np.uint64).astype(np.uint32).view(np.float32)
    rnd = rnd[~np.isnan(rnd)]
    logu = (np.exp(rng.uniform(np.log(2.0 ** -12), np.log(600.0), size=1 << 18))
            * rng.choice([-1.0, 1.0], size=1 << 18)).astype(np.float32)
    # every float whose low 16 mantissa bits are zero: all exponents, 7 mantissa bits
    grid = (np.arange(1 << 16, dtype=np.uint32) << 16).view(np.float32)
    grid = grid[~np.isnan(grid)]
    for x in (rnd, logu, grid):
        assert np.array_equal(oracle.e4m3_encode(x), brute_force_encode(x))


def test_encode_full_binade_at_subnormal_boundary(oracle):
    # every float32 in [2^-7, 2^-6): E4M3 subnormals meet normals here
    lo = np.float32(2.0 ** -7).view(np.uint32)
    x = (lo + np.arange(1 << 23, dtype=np.uint32)).view(np.float32)
    sel = x[:: 7]
    assert np.array_equal(oracle.e4m3_encode(sel), brute_force_encode(sel))
    # and all of it against the library cast
    want = torch.from_numpy(x.copy()).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(oracle.e4m3_encode(x), want)


def test_encode_matches_torch_cast_below_464(oracle):
    # stride through every positive finite float below 464, both signs
    top = int(np.float32(464.0).view(np.uint32))
    bits = np.arange(0, top, 97, dtype=np.uint32)
    x = bits.view(np.float32)
    x = np.concatenate([x, -x])
    want = torch.from_numpy(x.copy()).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(oracle.e4m3_encode(x), want)


def test_saturation_inf_nan(oracle):
    x = np.float32([448, 449, 464, 480, 1e30, np.inf, -448, -1e30, -np.inf])
    assert list(oracle.e4m3_encode(x)) == [0x7E] * 6 + [0xFE] * 3
    n = np.float32([np.nan])
    neg_nan = (n.view(np.uint32) | np.uint32(0x80000000)).view(np.float32)
    assert oracle.e4m3_encode(n)[0] == 0x7F
    assert oracle.e4m3_encode(neg_nan)[0] == 0xFF
    assert oracle.e4m3_encode(np.float32([-0.0]))[0] == 0x80
    assert oracle.e4m3_encode(np.float32([2.0 ** -10]))[0] == 0x00   # tie -> even (0)
    assert oracle.e4m3_encode(np.float32([3 * 2.0 ** -10]))[0] == 0x02  # tie 1,2 -> 2


def test_bits_range_matches_array_encode(oracle):
    first = 0x3F000000
    n = 4096
    x = (np.uint32(first) + np.arange(n, dtype=np.uint32)).view(np.float32)
    assert np.array_equal(oracle.e4m3_encode_bits_range(first, n), oracle.e4m3_encode(x))
