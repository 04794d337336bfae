"""C-ABI library on the host (no GPU): it loads, exports every symbol that
include/*.h declares, its planner matches the oracle's planner table for table,
and argument errors come back as status codes before any device work."""
import ctypes
import glob
import os
import re

import numpy as np
import pytest

from blockwise_fp8_zero_gb300 import fp8z, workloads

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    from blockwise_fp8_zero_gb300 import build
    build.build()
    return fp8z.lib()


def _declared():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        names |= set(re.findall(r"FP8Z_API\s+[\w\s\*]*?\b(fp8z_\w+)\s*\(", open(h).read()))
    return names


def test_exports_every_declared_symbol(L):
    names = _declared()
    assert {"fp8z_plan_shards", "fp8z_adamw_requant_step", "fp8z_dequant",
            "fp8z_transpose_fp8"} <= names
    for n in names:
        assert hasattr(L, n), n
    assert set(fp8z.EXPORTED) <= names


def test_status_strings(L):
    for code in (0, -1, -2, -3, -4, -5, -6, 99):
        assert fp8z.fp8z_status_string(code).startswith("FP8Z")


def _same(a, b):
    assert a.dtype.names == b.dtype.names or len(a.dtype) == len(b.dtype)
    assert a.tobytes() == b.tobytes()


CASES = [
    ([(1, 256, 384)], 1, 0),
    ([(1, 256, 384), (1, 128, 129), (2, 300, 100)], 3, 0),
    ([(1, 256, 384), (1, 128, 129), (2, 300, 100)], 3, 1),
    ([(1, 128, 128)] * 5, 2, 1),
    ([(1, 256, 256), (1, 128, 128)], 4, 1),
    ([(1, 1, 1)], 7, 0),
]


@pytest.mark.parametrize("shapes,dp,split", CASES)
def test_planner_matches_oracle(L, oracle, shapes, dp, split):
    a = fp8z.fp8z_plan_shards(shapes, dp, split)
    b = oracle.plan_shards(shapes, dp, split)
    for x, y in zip(a, b):
        _same(np.atleast_1d(x), np.atleast_1d(y))


@pytest.mark.parametrize("name,split", [("dense_h7168", 0), ("moe64", 0), ("mixed500", 0),
                                        ("mixed500", 1), ("flat6e9", 0)])
def test_planner_matches_oracle_on_workloads(L, oracle, name, split):
    w = workloads.get(name, split)
    a = fp8z.fp8z_plan_shards(w.shapes, w.dp, split)
    b = oracle.plan_shards(w.shapes, w.dp, split)
    for x, y in zip(a, b):
        _same(np.atleast_1d(x), np.atleast_1d(y))


def test_planner_random_layouts(L, oracle):
    rng = np.random.default_rng(2024)
    for trial in range(40):
        n = int(rng.integers(1, 40))
        shapes = [(int(rng.integers(1, 4)), int(rng.integers(1, 1000)), int(rng.integers(1, 1000)))
                  for _ in range(n)]
        dp = int(rng.integers(1, 20))
        split = int(rng.integers(0, 2))
        a = fp8z.fp8z_plan_shards(shapes, dp, split)
        b = oracle.plan_shards(shapes, dp, split)
        for x, y in zip(a, b):
            _same(np.atleast_1d(x), np.atleast_1d(y))


def test_planner_errors(L):
    sh = np.array([(1, 128, 128)], dtype=fp8z.param_shape_dtype)
    pe = np.zeros(1, fp8z.param_entry_dtype)
    sd = np.zeros(4, fp8z.shard_dtype)
    su = np.zeros(1, fp8z.plan_summary_dtype)
    bl = np.zeros(4, fp8z.block_desc_dtype)
    P = lambda a: a.ctypes.data
    assert L.fp8z_plan_shards(P(sh), 1, 0, 0, P(pe), P(sd), None, 0, P(su)) == fp8z.FP8Z_EINVAL
    assert L.fp8z_plan_shards(P(sh), 1, 2, 5, P(pe), P(sd), None, 0, P(su)) == fp8z.FP8Z_EINVAL
    bad = np.array([(1, 0, 128)], dtype=fp8z.param_shape_dtype)
    assert L.fp8z_plan_shards(P(bad), 1, 2, 0, P(pe), P(sd), None, 0, P(su)) == fp8z.FP8Z_EINVAL
    assert L.fp8z_plan_shards(P(sh), 1, 4, 0, P(pe), P(sd), P(bl), 3, P(su)) == fp8z.FP8Z_ENOSPACE
    assert L.fp8z_plan_shards(P(sh), 1, 4, 0, P(pe), P(sd), P(bl), 4, P(su)) == fp8z.FP8Z_OK


# ---- argument checks of the device entry points: every call below returns
# before any CUDA call, so no pointer here is ever dereferenced.
A16, A4 = 0x10000, 0x10004


def _step(L, hp, p=A16, g=A16, m=A16, v=A16, q=A16, inv=A16, cap=4, b0=0, nb=0, desc=None,
          params=None, npar=0, wt=None, wtb=0, it=None, itc=0, status=None):
    return L.fp8z_adamw_requant_step(p, g, m, v, q, inv, cap, b0, nb, desc, params, npar, wt, wtb,
                                     it, itc, ctypes.byref(hp), status, None)


def test_step_argument_errors(L):
    hp = fp8z.hparams()
    assert _step(L, hp) == fp8z.FP8Z_OK                          # nblk == 0: nothing launched
    assert _step(L, hp, p=None) == fp8z.FP8Z_EINVAL
    assert _step(L, hp, g=A4) == fp8z.FP8Z_EALIGN
    assert _step(L, hp, q=A4) == fp8z.FP8Z_EALIGN
    assert _step(L, hp, nb=-1) == fp8z.FP8Z_EINVAL
    assert _step(L, hp, b0=3, nb=2) == fp8z.FP8Z_ENOSPACE
    assert _step(L, hp, b0=5, nb=0) == fp8z.FP8Z_ENOSPACE
    assert _step(L, hp, wt=A16, it=A16, wtb=10, itc=1) == fp8z.FP8Z_EINVAL   # no desc/params
    assert _step(L, hp, wt=A16) == fp8z.FP8Z_EINVAL                          # half of the pair
    for field, bad in [("beta1", 1.0), ("beta2", -0.1), ("eps", 0.0), ("lr", float("nan")),
                       ("fp8_max", 500.0), ("fp8_max", 0.0), ("min_scale", -1.0),
                       ("scale_mode", 7), ("decay_mode", 2), ("step", 0)]:
        h = fp8z.hparams()
        setattr(h, field, bad)
        assert _step(L, h) == fp8z.FP8Z_EINVAL, field


def test_aux_argument_errors(L):
    assert L.fp8z_dequant(None, A16, 1, A16, None, None) == fp8z.FP8Z_EINVAL
    assert L.fp8z_dequant(A4, A16, 1, A16, None, None) == fp8z.FP8Z_EALIGN
    assert L.fp8z_dequant(A16, A16, 1, A16, A16 + 2, None) == fp8z.FP8Z_EALIGN
    assert L.fp8z_dequant(A16, A16, -1, A16, None, None) == fp8z.FP8Z_EINVAL
    assert L.fp8z_dequant(A16, A16, 0, A16, None, None) == fp8z.FP8Z_OK
    ent = np.zeros(1, fp8z.param_entry_dtype)
    ent[0] = (0, 0, 0, 1, 200, 300, 2, 2, 0, 0)                  # wb should be 3
    assert L.fp8z_transpose_fp8(A16, A16, ent.ctypes.data, A16, A16, None, None) == fp8z.FP8Z_EINVAL
    ent[0]["wb"] = 3
    assert L.fp8z_transpose_fp8(A16, A16, ent.ctypes.data, A4, A16, None, None) == fp8z.FP8Z_EALIGN
    assert L.fp8z_transpose_fp8(A16, A16, ent.ctypes.data, A16, A16, A16 + 2, None) == fp8z.FP8Z_EALIGN
    assert L.fp8z_e4m3_encode_bits(0, 6, A16, None) == fp8z.FP8Z_EINVAL
    assert L.fp8z_e4m3_encode_bits(0, 8, A4, None) == fp8z.FP8Z_EALIGN
    assert L.fp8z_e4m3_encode_bits(0, 0, A16, None) == fp8z.FP8Z_OK
    assert L.fp8z_watchdog_selftest(A16, -1, None) == fp8z.FP8Z_EINVAL
    assert L.fp8z_watchdog_selftest(A16, 10 ** 11, None) == fp8z.FP8Z_EINVAL
    assert L.fp8z_watchdog_selftest(None, 1000, None) == fp8z.FP8Z_EINVAL


def test_rowwise_and_mx_argument_errors(L):
    # 1x128 row-wise quantize / transpose: zero rows is an empty call, a row
    # length that is not a multiple of 128 or a bad pow2 flag is refused
    assert L.fp8z_quantize_rowwise(A16, 0, 256, 1, A16, A16, None) == fp8z.FP8Z_OK
    assert L.fp8z_quantize_rowwise(A16, 4, 0, 1, A16, A16, None) == fp8z.FP8Z_OK
    assert L.fp8z_quantize_rowwise(A16, 4, 100, 1, A16, A16, None) == fp8z.FP8Z_EINVAL
    assert L.fp8z_quantize_rowwise(A16, 4, 128, 2, A16, A16, None) == fp8z.FP8Z_EINVAL
    assert L.fp8z_quantize_rowwise(A16, -1, 128, 1, A16, A16, None) == fp8z.FP8Z_EINVAL
    assert L.fp8z_quantize_rowwise(A4, 4, 128, 1, A16, A16, None) == fp8z.FP8Z_EALIGN
    assert L.fp8z_quantize_rowwise(None, 4, 128, 1, A16, A16, None) == fp8z.FP8Z_EINVAL
    assert L.fp8z_transpose_rowwise(A16, A16, 0, 128, A16, A16, None) == fp8z.FP8Z_OK
    assert L.fp8z_transpose_rowwise(A16, A16, 100, 128, A16, A16, None) == fp8z.FP8Z_EINVAL
    assert L.fp8z_transpose_rowwise(A16, A16, 128, 130, A16, A16, None) == fp8z.FP8Z_EINVAL
    assert L.fp8z_transpose_rowwise(A4, A16, 128, 128, A16, A16, None) == fp8z.FP8Z_EALIGN
    assert L.fp8z_dequant_rowwise(A16, A16, 0, 128, 1, A16, None) == fp8z.FP8Z_OK
    assert L.fp8z_dequant_rowwise(A16, A16, 4, 100, 0, A16, None) == fp8z.FP8Z_EINVAL
    assert L.fp8z_dequant_rowwise(A16, A16, 100, 128, 1, A16, None) == fp8z.FP8Z_EINVAL   # rows % 128
    assert L.fp8z_dequant_rowwise(A16, A16, 4, 128, 2, A16, None) == fp8z.FP8Z_EINVAL
    assert L.fp8z_dequant_rowwise(A16, A16, 4, 128, 0, A4, None) == fp8z.FP8Z_EALIGN
    # MXFP8 step: same state checks as the block-scaled step, its own scale output
    hp = fp8z.hparams()
    mx = lambda **k: L.fp8z_adamw_requant_step_mx(
        k.get("p", A16), A16, A16, A16, k.get("q", A16), k.get("s", A16), 4, k.get("b0", 0),
        k.get("nb", 0), None, ctypes.byref(k.get("hp", hp)), None, None)
    assert mx() == fp8z.FP8Z_OK                                  # nblk == 0: nothing launched
    assert mx(s=A16 + 1) == fp8z.FP8Z_OK                         # E8M0 bytes need no alignment
    assert mx(s=None) == fp8z.FP8Z_EINVAL
    assert mx(p=None) == fp8z.FP8Z_EINVAL
    assert mx(q=A4) == fp8z.FP8Z_EALIGN
    assert mx(b0=3, nb=2) == fp8z.FP8Z_ENOSPACE
    bad = fp8z.hparams()
    bad.eps = 0.0
    assert mx(hp=bad) == fp8z.FP8Z_EINVAL


def test_wait_limit_knob(L):
    """The process-wide limit of the bounded device waits: host only, checked
    range, 0 restores the 2 s default."""
    default = 2_000_000_000
    assert fp8z.fp8z_get_wait_limit_ns() == default
    try:
        fp8z.fp8z_set_wait_limit_ns(300)
        assert fp8z.fp8z_get_wait_limit_ns() == 300
        assert L.fp8z_set_wait_limit_ns(-1) == fp8z.FP8Z_EINVAL
        assert L.fp8z_set_wait_limit_ns(10 ** 10 + 1) == fp8z.FP8Z_EINVAL
        assert fp8z.fp8z_get_wait_limit_ns() == 300            # a refused value changes nothing
        fp8z.fp8z_set_wait_limit_ns(10 ** 10)
        assert fp8z.fp8z_get_wait_limit_ns() == 10 ** 10
    finally:
        fp8z.fp8z_set_wait_limit_ns(0)
    assert fp8z.fp8z_get_wait_limit_ns() == default


def test_bindings_refuse_short_tables():
    """A descriptor or param table shorter than the launch reads is refused by
    the binding before any pointer is taken (CPU tensors: the size check comes
    first, so no device is needed)."""
    torch = pytest.importorskip("torch")
    cap = 4
    f = lambda n, dt=torch.float32: torch.zeros(n, dtype=dt)
    p, g, m, v = (f(cap * fp8z.BLOCK_ELEMS) for _ in range(4))
    q = f(cap * fp8z.BLOCK_ELEMS, torch.uint8)
    inv = f(cap)
    hp = fp8z.hparams()
    short_desc = f(cap * 20 - 1, torch.uint8)
    with pytest.raises(ValueError, match="desc"):
        fp8z.fp8z_adamw_requant_step(p, g, m, v, q, inv, 0, 1, hp, desc=short_desc)
    with pytest.raises(ValueError, match="params"):
        fp8z.fp8z_adamw_requant_step(p, g, m, v, q, inv, 0, 1, hp, desc=f(cap * 20, torch.uint8),
                                     params=f(64 * 2 - 1, torch.uint8), nparams=2,
                                     w_fp8_t=f(16, torch.uint8), inv_scale_t=f(4))
    with pytest.raises(ValueError, match="desc"):
        fp8z.fp8z_adamw_requant_step_mx(p, g, m, v, q, f(cap * 512, torch.uint8), 0, 1, hp,
                                        desc=short_desc)
    maps = f(128, torch.uint8)
    with pytest.raises(ValueError, match="desc"):
        fp8z.fp8z_adamw_requant_step_rowmajor(p, m, v, maps, f(16, torch.uint8), inv, 0, 1, hp,
                                              short_desc, f(64, torch.uint8), 1)
    with pytest.raises(ValueError, match="params"):
        fp8z.fp8z_adamw_requant_step_rowmajor(p, m, v, maps, f(16, torch.uint8), inv, 0, 1, hp,
                                              f(cap * 20, torch.uint8), f(63, torch.uint8), 1)
    ent = np.zeros(1, fp8z.param_entry_dtype)
    ent[0] = (2, 0, 0, 1, 128, 128, 1, 1, 0, 0)                  # blocks 2 .. 2 of a 3-block buffer
    with pytest.raises(ValueError, match="inv_scale"):
        fp8z.fp8z_transpose_fp8(f(3 * fp8z.BLOCK_ELEMS, torch.uint8), f(2), ent[0],
                                f(128 * 128, torch.uint8), f(1))
