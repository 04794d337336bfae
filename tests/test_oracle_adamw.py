"""Pins for the oracle's AdamW element step (CPU only).

Checks against: the float64 textbook definition within rounding bounds; the
closed form of the first step; the zero-state/zero-grad special case; and the
torch-op ordering printed in the lpnh.cn "Model-Optimizer" article §4.3 (decay
after the update), evaluated with torch float32 CPU ops (library routines).
"""
import math

import numpy as np
import pytest
import torch

from _defs import EPS32, adamw_error_bounds, adamw_fp64, ulp32


def _draw(rng, n, scale_p=0.02, scale_g=1e-3, state=True):
    p = rng.normal(0, scale_p, n).astype(np.float32)
    g = rng.normal(0, scale_g, n).astype(np.float32)
    if state:
        m = rng.normal(0, scale_g * 0.3, n).astype(np.float32)
        v = (rng.uniform(0.5, 1.5, n) * scale_g ** 2).astype(np.float32)
    else:
        m = np.zeros(n, np.float32)
        v = np.zeros(n, np.float32)
    return p, g, m, v


@pytest.mark.parametrize("step", [1, 2, 11, 1000])
@pytest.mark.parametrize("decay_mode", [0, 1])
def test_adamw_within_fp64_definition(oracle, step, decay_mode):
    rng = np.random.default_rng(step * 10 + decay_mode)
    hp = oracle.Hparams.make(step=step, decay_mode=decay_mode)
    p, g, m, v = _draw(rng, 4000, state=step > 1)
    # a few wild magnitudes and sign mixes
    g[:20] *= 1e4
    m[20:40] = -np.sign(g[20:40]) * np.abs(m[20:40]) * 50
    p[40:60] = rng.normal(0, 30, 20)
    p1, m1, v1 = oracle.adamw_elements(hp, p, g, m, v)
    pd, md, vd = adamw_fp64(hp, p, g, m, v)
    bp, bm, bv = adamw_error_bounds(hp, p, g, m, v)
    assert np.all(np.abs(m1 - md) <= bm)
    assert np.all(np.abs(v1 - vd) <= bv)
    assert np.all(np.abs(p1 - pd) <= bp)


def test_bounds_catch_plausible_mistakes(oracle):
    """The bounds above are tight enough to fail a dropped or mis-signed term."""
    rng = np.random.default_rng(7)
    hp = oracle.Hparams.make(step=11)
    p, g, m, v = _draw(rng, 2000)
    pd, md, vd = adamw_fp64(hp, p, g, m, v)
    bp, bm, bv = adamw_error_bounds(hp, p, g, m, v)
    lr, wd = 1e-4, 0.1
    no_decay = pd + p * lr * wd                        # weight decay dropped
    assert np.any(np.abs(no_decay - pd) > bp)
    hp1 = oracle.Hparams.make(step=11)
    hp1.step = 12                                       # wrong bias-correction step
    pw, _, _ = adamw_fp64(hp1, p, g, m, v)
    assert np.any(np.abs(pw - pd) > bp)
    wrong_m = 0.1 * m + 0.9 * g                         # betas swapped
    assert np.any(np.abs(wrong_m - md) > bm)


def test_first_step_closed_form(oracle):
    """t = 1, m = v = 0: m'/bc1 = g and sqrt(v'/bc2) = |g|, so
    p' = p*(1 - lr*wd) - lr * g / (|g| + eps) (the update is lr*sign(g) up to eps)."""
    rng = np.random.default_rng(0)
    hp = oracle.Hparams.make(step=1)
    p, g, m, v = _draw(rng, 20000, state=False)
    p1, m1, v1 = oracle.adamw_elements(hp, p, g, m, v)
    lr = float(np.float32(1e-4)); wd = float(np.float32(0.1)); eps = float(np.float32(1e-8))
    gd = g.astype(np.float64)
    upd = lr * gd / (np.abs(gd) + eps)
    closed = p.astype(np.float64) * (1 - lr * wd) - upd
    tol = 4 * ulp32(upd) + ulp32(closed) + ulp32(p * (1 - lr * wd))
    assert np.all(np.abs(p1 - closed) <= tol)
    omb1 = np.float32(1.0 - float(np.float32(0.9)))
    assert np.array_equal(m1, omb1 * g)          # m = 0: m' = (1-beta1)*g exactly


def test_zero_grad_zero_state_is_pure_decay(oracle):
    hp = oracle.Hparams.make(step=5)
    p = np.float32([0.5, -0.25, 3.0, 0.0, -0.0])
    z = np.zeros_like(p)
    p1, m1, v1 = oracle.adamw_elements(hp, p, z, z, z)
    decay = np.float32(1.0 - float(np.float32(1e-4)) * float(np.float32(0.1)))
    assert np.array_equal(p1, p * decay)
    assert not np.any(m1) and not np.any(v1)


def _printed_order_torch(p, g, m, v, lr, b1, b2, eps, wd, t):
    """The update in the order the Model-Optimizer article prints it, torch f32."""
    p, g, m, v = (torch.from_numpy(a.copy()) for a in (p, g, m, v))
    m_new = torch.add(torch.mul(m, b1), g, alpha=1 - b1)
    v_new = torch.addcmul(torch.mul(v, b2), g, g, value=1 - b2)
    c1 = 1 - b1 ** t
    c2 = 1 - b2 ** t
    den = torch.add(torch.div(torch.sqrt(v_new), c2 ** 0.5), eps)
    p_new = torch.addcdiv(p, m_new, den, value=-(lr / c1))
    p_new = torch.add(p_new, p_new, alpha=-(lr * wd))
    return p_new.numpy(), m_new.numpy(), v_new.numpy()


@pytest.mark.parametrize("step", [1, 11, 1000])
def test_matches_printed_torch_order_post_decay(oracle, step):
    rng = np.random.default_rng(100 + step)
    hp = oracle.Hparams.make(step=step, decay_mode=1)
    p, g, m, v = _draw(rng, 5000, state=step > 1)
    p1, m1, v1 = oracle.adamw_elements(hp, p, g, m, v)
    f = lambda x: float(np.float32(x))
    pt, mt, vt = _printed_order_torch(p, g, m, v, f(1e-4), f(0.9), f(0.95), f(1e-8), f(0.1), step)
    # operand-relative bounds: m' may cancel (m and g of opposite signs)
    mag_m = np.abs(0.9 * m.astype(np.float64)) + np.abs(0.1 * g.astype(np.float64))
    assert np.all(np.abs(m1 - mt) <= 4 * EPS32 * mag_m + 1e-44)
    assert np.all(np.abs(v1 - vt) <= 2 * ulp32(vt))
    # u differs by a few ulp (divide by sqrt(bc2) vs multiply by its inverse)
    upd = np.abs(p.astype(np.float64) - pt)
    assert np.all(np.abs(p1 - pt) <= 2 * ulp32(pt) + 8 * EPS32 * upd)


def test_pre_and_post_decay_differ_only_by_second_order(oracle):
    rng = np.random.default_rng(5)
    p, g, m, v = _draw(rng, 5000)
    a, _, _ = oracle.adamw_elements(oracle.Hparams.make(step=11, decay_mode=0), p, g, m, v)
    b, _, _ = oracle.adamw_elements(oracle.Hparams.make(step=11, decay_mode=1), p, g, m, v)
    lr, wd = 1e-4, 0.1
    # post - pre = lr*wd*step_size*u: at most lr*wd*|update| plus rounding
    upd = np.abs(a.astype(np.float64) - p * (1 - lr * wd))
    assert np.all(np.abs(a - b) <= lr * wd * upd * 1.01 + 2 * ulp32(a))


def test_scalars_first_step(oracle):
    hp = oracle.Hparams.make(step=1)
    sc = oracle.adamw_scalars(hp)
    b1, b2 = float(np.float32(0.9)), float(np.float32(0.95))
    lr = float(np.float32(1e-4))
    # at t = 1 the bias corrections are exactly 1 - beta
    assert sc[5] == np.float32(lr / (1 - b1))
    assert sc[6] == np.float32(1 / math.sqrt(1 - b2))
    assert sc[2] == np.float32(1 - b1) and sc[3] == np.float32(1 - b2)
