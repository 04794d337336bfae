"""Independent definitions used to pin the oracle (tests only).

These are written from the mathematics, not from the oracle's C code:
- E4M3 values from the value formula and a brute-force nearest search;
- the AdamW step in float64, in the textbook bias-corrected form
  m_hat = m'/(1-beta1^t), v_hat = v'/(1-beta2^t),
  p' = p*(1-lr*wd) - lr*m_hat/(sqrt(v_hat)+eps)        (decay before the update)
  p' = (p - lr*m_hat/(sqrt(v_hat)+eps)) * (1-lr*wd)      (decay after the update)
  (lpnh.cn "Model-Optimizer" article §4.3), with every hyper-parameter taken as
  the float32 value the step receives.
"""
import math

import numpy as np

EPS32 = 2.0 ** -24     # unit roundoff of float32


def finite_e4m3_table():
    """Values of codes 0..126 from the "FP8-Flow-MoE" §3.1 value formula."""
    vals = []
    for code in range(127):
        E, M = code >> 3, code & 7
        vals.append(M / 8.0 * 2.0 ** -6 if E == 0 else (1 + M / 8.0) * 2.0 ** (E - 7))
    return np.array(vals, dtype=np.float64)


def brute_force_encode(x):
    """Nearest finite E4M3 code by exhaustive search; ties to the even code."""
    x = np.asarray(x, dtype=np.float32)
    table = finite_e4m3_table()
    bits = x.view(np.uint32)
    sign = ((bits >> 31) << 7).astype(np.uint8)
    # |x| >= 448 is nearest to the largest value, 448, whatever its size; the cap
    # keeps the float64 distances exact (no false ties for huge inputs)
    a = np.minimum(np.abs(x.astype(np.float64)), 1024.0).ravel()
    out = np.empty(a.shape, dtype=np.uint8)
    chunk = 1 << 16
    codes = np.arange(127)
    for s in range(0, a.size, chunk):
        d = np.abs(a[s:s + chunk, None] - table[None, :])
        cand = d == d.min(axis=1, keepdims=True)
        # two candidates only at an exact midpoint: prefer the even code
        score = np.where(cand, (codes & 1)[None, :] * 1000 + codes[None, :], 1 << 30)
        out[s:s + chunk] = np.argmin(score, axis=1).astype(np.uint8)
    out = out.reshape(x.shape) | sign
    nan = np.isnan(x)
    out[nan] = sign[nan] | 0x7F
    return out


def e4m3_quantum(y):
    """Spacing of E4M3 values around |y| (2^-9 in the subnormal range)."""
    a = np.abs(np.asarray(y, dtype=np.float64))
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -20)))
    return np.where(e < -6, 2.0 ** -9, 2.0 ** (e - 3))


def hp_values(hp):
    """float32 hyper-parameters -> float64 values (exactly the float32 ones)."""
    f = lambda x: float(np.float32(x))
    return dict(lr=f(hp.lr), b1=f(hp.beta1), b2=f(hp.beta2), eps=f(hp.eps),
                wd=f(hp.weight_decay), t=int(hp.step), decay_mode=int(hp.decay_mode))


def adamw_fp64(hp, p, g, m, v):
    """The AdamW step in float64 (see module docstring).  Returns (p', m', v')."""
    h = hp_values(hp)
    p, g, m, v = (np.asarray(a, dtype=np.float64) for a in (p, g, m, v))
    m1 = h["b1"] * m + (1.0 - h["b1"]) * g
    v1 = h["b2"] * v + (1.0 - h["b2"]) * g * g
    m_hat = m1 / (1.0 - math.pow(h["b1"], h["t"]))
    v_hat = v1 / (1.0 - math.pow(h["b2"], h["t"]))
    upd = h["lr"] * m_hat / (np.sqrt(v_hat) + h["eps"])
    keep = 1.0 - h["lr"] * h["wd"]
    if h["decay_mode"] == 0:
        p1 = p * keep - upd
    else:
        p1 = (p - upd) * keep
    return p1, m1, v1


def adamw_error_bounds(hp, p, g, m, v):
    """Generous float32 rounding bounds (absolute) for p', m', v' of one step.

    Each float32 operation adds at most one unit roundoff of its result, and
    the scalars carry one rounding each.  A dropped term, a wrong sign or a
    wrong bias correction gives an error of the size of the term itself, far
    beyond these bounds.
    """
    h = hp_values(hp)
    p, g, m, v = (np.asarray(a, dtype=np.float64) for a in (p, g, m, v))
    p1, m1, v1 = adamw_fp64(hp, p, g, m, v)
    bm = 4 * EPS32 * (np.abs(h["b1"] * m) + np.abs((1 - h["b1"]) * g)) + 1e-44
    bv = 4 * EPS32 * (np.abs(h["b2"] * v) + np.abs((1 - h["b2"]) * g * g)) + 1e-44
    bc2 = 1.0 - math.pow(h["b2"], h["t"])
    d = np.sqrt(v1 / bc2) + h["eps"]
    u = m1 / (1.0 - math.pow(h["b1"], h["t"])) / d
    bu = (bm / (1.0 - math.pow(h["b1"], h["t"])) + np.abs(u) * d * 10 * EPS32) / d
    keep = 1.0 - h["lr"] * h["wd"]
    bp = 4 * EPS32 * (np.abs(p * keep) + np.abs(h["lr"] * u)) + h["lr"] * bu * 1.01 + 1e-44
    if h["decay_mode"] == 1:
        bp = bp + 4 * EPS32 * np.abs(p1)
    return bp, bm, bv


def ulp32(x):
    x = np.abs(np.asarray(x, dtype=np.float32))
    return (np.nextafter(x, np.float32(np.inf)) - x).astype(np.float64)
