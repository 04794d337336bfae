"""CPU oracle for the blockwise-FP8 ZeRO-1 optimizer step -- TEST INFRASTRUCTURE.

Plain, slow, single-threaded C (``fp8z_oracle.c``) behind a ctypes wrapper.
Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference
arm of ``bench.py`` may import this package.  It shares no code with the CUDA
library (``blockwise_fp8_zero_gb300``) and never imports it.

Every array argument is a numpy array on the host.  Struct dtypes below mirror
the C structs in ``fp8z_oracle.c`` (their own definitions, written for the
oracle).
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from .build import build_oracle, oracle_lib_path

__all__ = [
    "PARAM_SHAPE", "PARAM_ENTRY", "SHARD", "BLOCK_DESC", "PLAN_SUMMARY",
    "Hparams", "e4m3_encode", "e4m3_encode_bits_range", "e4m3_decode",
    "adamw_scalars", "adamw_elements", "block_scale", "adamw_requant_step",
    "dequant", "transpose_fp8", "fold", "unfold", "plan_shards", "BLK", "BLK_ELEMS",
    "quantize_rowwise", "transpose_rowwise", "dequant_rowwise", "adamw_requant_step_mx",
]

BLK = 128
BLK_ELEMS = BLK * BLK

PARAM_SHAPE = np.dtype([("e", "<i8"), ("rows", "<i8"), ("cols", "<i8")])
PARAM_ENTRY = np.dtype([
    ("blk_offset", "<i8"), ("t_offset", "<i8"), ("t_scale_offset", "<i8"),
    ("e", "<i8"), ("rows", "<i8"), ("cols", "<i8"),
    ("hb", "<i4"), ("wb", "<i4"), ("bucket", "<i4"), ("reserved", "<i4"),
])
SHARD = np.dtype([("blk_begin", "<i8"), ("blk_count_real", "<i8"), ("blk_capacity", "<i8")])
BLOCK_DESC = np.dtype([
    ("param", "<i4"), ("e", "<i4"), ("brow", "<i4"), ("bcol", "<i4"),
    ("valid_rows", "<u2"), ("valid_cols", "<u2"),
])
PLAN_SUMMARY = np.dtype([
    ("real_elems", "<i8"), ("total_blocks", "<i8"), ("fold_pad_elems", "<i8"),
    ("shard_pad_elems", "<i8"), ("capacity_blocks", "<i8"), ("naive_straddled_blocks", "<i8"),
])
assert PARAM_ENTRY.itemsize == 64 and BLOCK_DESC.itemsize == 20


class Hparams(ctypes.Structure):
    """AdamW + quantizer hyper-parameters (same field order as the C struct)."""

    _fields_ = [
        ("lr", ctypes.c_float), ("beta1", ctypes.c_float), ("beta2", ctypes.c_float),
        ("eps", ctypes.c_float), ("weight_decay", ctypes.c_float),
        ("step", ctypes.c_int64),
        ("fp8_max", ctypes.c_float), ("min_scale", ctypes.c_float),
        ("scale_mode", ctypes.c_int32), ("decay_mode", ctypes.c_int32),
    ]

    @classmethod
    def make(cls, lr=1e-4, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1, step=1,
             fp8_max=448.0, min_scale=1e-6, scale_mode=0, decay_mode=0):
        return cls(lr, beta1, beta2, eps, weight_decay, step, fp8_max, min_scale,
                   scale_mode, decay_mode)


_lib = None


def _load():
    global _lib
    if _lib is None:
        path = oracle_lib_path()
        if not os.path.exists(path):
            build_oracle()
        lib = ctypes.CDLL(path)
        P = ctypes.c_void_p
        i64, i32, u32 = ctypes.c_int64, ctypes.c_int32, ctypes.c_uint32
        lib.fp8z_ref_e4m3_decode.argtypes = [ctypes.c_uint8]
        lib.fp8z_ref_e4m3_decode.restype = ctypes.c_double
        lib.fp8z_ref_e4m3_encode_array.argtypes = [P, i64, P]
        lib.fp8z_ref_e4m3_encode_bits_range.argtypes = [u32, i64, P]
        lib.fp8z_ref_adamw_scalars.argtypes = [ctypes.POINTER(Hparams), P]
        lib.fp8z_ref_adamw_element.argtypes = [P, ctypes.c_int] + [ctypes.c_float] * 4 + [P, P, P]
        lib.fp8z_ref_block_scale.argtypes = [ctypes.c_float, ctypes.c_float, ctypes.c_float,
                                             ctypes.c_int, P]
        lib.fp8z_ref_block_scale.restype = ctypes.c_float
        lib.fp8z_ref_adamw_requant_step.argtypes = [P, P, P, P, P, P, i64, i64, P, P, P, P,
                                                    ctypes.POINTER(Hparams)]
        lib.fp8z_ref_adamw_requant_step.restype = ctypes.c_int
        lib.fp8z_ref_dequant.argtypes = [P, P, i64, P]
        lib.fp8z_ref_transpose_fp8.argtypes = [P, P, P, P, P]
        lib.fp8z_ref_fold.argtypes = [P, i64, i64, i64, P]
        lib.fp8z_ref_unfold.argtypes = [P, i64, i64, i64, P]
        lib.fp8z_ref_plan_shards.argtypes = [P, i32, i32, i32, P, P, P, i64, P]
        lib.fp8z_ref_adamw_requant_step_mx.argtypes = [P, P, P, P, P, P, i64, i64, P,
                                                       ctypes.POINTER(Hparams)]
        lib.fp8z_ref_adamw_requant_step_mx.restype = ctypes.c_int
        lib.fp8z_ref_quantize_rowwise.argtypes = [P, i64, i64, ctypes.c_int, P, P]
        lib.fp8z_ref_transpose_rowwise.argtypes = [P, P, i64, i64, P, P]
        lib.fp8z_ref_dequant_rowwise.argtypes = [P, P, i64, i64, P]
        lib.fp8z_ref_plan_shards.restype = ctypes.c_int
        _lib = lib
    return _lib


def _ptr(a):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data


def e4m3_encode(x):
    x = np.ascontiguousarray(x, dtype=np.float32)
    q = np.empty(x.shape, dtype=np.uint8)
    _load().fp8z_ref_e4m3_encode_array(_ptr(x), x.size, _ptr(q))
    return q


def e4m3_encode_bits_range(first, n, out=None):
    q = np.empty(n, dtype=np.uint8) if out is None else out
    _load().fp8z_ref_e4m3_encode_bits_range(first, n, _ptr(q))
    return q


def e4m3_decode(q):
    """Exact decoded value (float64) of each code; NaN for 0x7F/0xFF."""
    lib = _load()
    table = np.array([lib.fp8z_ref_e4m3_decode(c) for c in range(256)], dtype=np.float64)
    return table[np.asarray(q, dtype=np.uint8)]


def adamw_scalars(hp):
    out = np.zeros(9, dtype=np.float32)
    _load().fp8z_ref_adamw_scalars(ctypes.byref(hp), _ptr(out))
    return out


def adamw_elements(hp, p, g, m, v):
    """Element-wise AdamW on 1-D float32 arrays (no quantization)."""
    lib = _load()
    sc = adamw_scalars(hp)
    p1, m1, v1 = (np.empty_like(np.asarray(a, np.float32)) for a in (p, m, v))
    o = [ctypes.c_float() for _ in range(3)]
    for i in range(len(p)):
        lib.fp8z_ref_adamw_element(_ptr(sc), hp.decay_mode, float(p[i]), float(g[i]),
                                   float(m[i]), float(v[i]),
                                   ctypes.byref(o[0]), ctypes.byref(o[1]), ctypes.byref(o[2]))
        p1[i], m1[i], v1[i] = o[0].value, o[1].value, o[2].value
    return p1, m1, v1


def block_scale(amax, fp8_max=448.0, min_scale=1e-6, scale_mode=0):
    inv = ctypes.c_float()
    s = _load().fp8z_ref_block_scale(amax, fp8_max, min_scale, scale_mode, ctypes.byref(inv))
    return np.float32(s), np.float32(inv.value)


def adamw_requant_step(p, g, m, v, w_fp8, inv_scale, blk_begin, nblk, hp,
                       desc=None, params=None, w_fp8_t=None, inv_scale_t=None):
    """In place on p, m, v; writes w_fp8 / inv_scale (and the optional copies)."""
    for a in (p, g, m, v):
        assert a.dtype == np.float32
    rc = _load().fp8z_ref_adamw_requant_step(
        _ptr(p), _ptr(g), _ptr(m), _ptr(v), _ptr(w_fp8), _ptr(inv_scale),
        blk_begin, nblk, _ptr(desc), _ptr(params), _ptr(w_fp8_t), _ptr(inv_scale_t),
        ctypes.byref(hp))
    if rc != 0:
        raise ValueError(f"oracle step failed: {rc}")


def adamw_requant_step_mx(p, g, m, v, w_fp8, mx_scale, blk_begin, nblk, hp, desc=None):
    """MXFP8 output variant: in place on p, m, v; writes codes and E8M0 scales
    ([nblk, 128, 4] bytes, one per 32 elements of a block row)."""
    rc = _load().fp8z_ref_adamw_requant_step_mx(
        _ptr(p), _ptr(g), _ptr(m), _ptr(v), _ptr(w_fp8), _ptr(mx_scale), blk_begin, nblk,
        _ptr(desc), ctypes.byref(hp))
    if rc != 0:
        raise ValueError(f"oracle mx step failed: {rc}")


def dequant(w_fp8, inv_scale, nblk):
    out = np.empty(nblk * BLK_ELEMS, dtype=np.float32)
    _load().fp8z_ref_dequant(_ptr(w_fp8), _ptr(inv_scale), nblk, _ptr(out))
    return out


def transpose_fp8(w_fp8, inv_scale, entry):
    """entry: one PARAM_ENTRY record.  Returns ([E,W,H] bytes, [E,Wb,Hb] inv)."""
    ent = np.array([entry], dtype=PARAM_ENTRY)
    E, H, W = int(entry["e"]), int(entry["rows"]), int(entry["cols"])
    out = np.zeros((E, W, H), dtype=np.uint8)
    inv_t = np.zeros((E, int(entry["wb"]), int(entry["hb"])), dtype=np.float32)
    _load().fp8z_ref_transpose_fp8(_ptr(w_fp8), _ptr(inv_scale), _ptr(ent), _ptr(out), _ptr(inv_t))
    return out, inv_t


def fold(w):
    """[E,H,W] (or [H,W]) float32 -> folded [nblk,128,128] with zero padding."""
    w = np.ascontiguousarray(w, dtype=np.float32)
    if w.ndim == 2:
        w = w[None]
    E, H, W = w.shape
    nb = E * (-(-H // BLK)) * (-(-W // BLK))
    out = np.empty((nb, BLK, BLK), dtype=np.float32)
    _load().fp8z_ref_fold(_ptr(w), E, H, W, _ptr(out))
    return out


def unfold(blocks, E, H, W):
    blocks = np.ascontiguousarray(blocks, dtype=np.float32)
    out = np.empty((E, H, W), dtype=np.float32)
    _load().fp8z_ref_unfold(_ptr(blocks), E, H, W, _ptr(out))
    return out


def quantize_rowwise(x, pow2=True):
    """[R, C] float32 (C % 128 == 0) -> (codes [R, C], scales [R, C/128]); 1x128 tiles."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    R, C = x.shape
    q = np.empty((R, C), np.uint8)
    s = np.empty((R, C // BLK), np.float32)
    _load().fp8z_ref_quantize_rowwise(_ptr(x), R, C, int(pow2), _ptr(q), _ptr(s))
    return q, s


def transpose_rowwise(q, s):
    """Row-wise codes/scales of [R, C] -> column-wise codes [C, R], scales [C, R/128]."""
    q = np.ascontiguousarray(q, dtype=np.uint8)
    s = np.ascontiguousarray(s, dtype=np.float32)
    R, C = q.shape
    qt = np.empty((C, R), np.uint8)
    st = np.empty((C, R // BLK), np.float32)
    _load().fp8z_ref_transpose_rowwise(_ptr(q), _ptr(s), R, C, _ptr(qt), _ptr(st))
    return qt, st


def dequant_rowwise(q, s):
    q = np.ascontiguousarray(q, dtype=np.uint8)
    s = np.ascontiguousarray(s, dtype=np.float32)
    R, C = q.shape
    x = np.empty((R, C), np.float32)
    _load().fp8z_ref_dequant_rowwise(_ptr(q), _ptr(s), R, C, _ptr(x))
    return x


def plan_shards(shapes, dp, split, with_blocks=True):
    """shapes: list of (e, rows, cols).  Returns (params, shards, blocks|None, summary)."""
    sh = np.array([tuple(int(x) for x in s) for s in shapes], dtype=PARAM_SHAPE)
    n = len(sh)
    params = np.zeros(max(n, 1), dtype=PARAM_ENTRY)
    shards = np.zeros(dp, dtype=SHARD)
    summ = np.zeros(1, dtype=PLAN_SUMMARY)
    lib = _load()
    rc = lib.fp8z_ref_plan_shards(_ptr(sh) if n else None, n, dp, split, _ptr(params),
                                  _ptr(shards), None, 0, _ptr(summ))
    if rc != 0:
        raise ValueError(f"oracle planner failed: {rc}")
    blocks = None
    if with_blocks:
        cap = int(summ["capacity_blocks"][0])
        blocks = np.zeros(max(cap, 1), dtype=BLOCK_DESC)
        rc = lib.fp8z_ref_plan_shards(_ptr(sh) if n else None, n, dp, split, _ptr(params),
                                      _ptr(shards), _ptr(blocks), cap, _ptr(summ))
        if rc != 0:
            raise ValueError(f"oracle planner failed: {rc}")
        blocks = blocks[:cap]
    return params[:n], shards, blocks, summ[0]
