"""Thin ctypes binding of libfp8z.so (include/fp8z.h), same names as the C ABI.

Argument marshalling only: every step of the optimizer path runs in the CUDA
kernels of libfp8z.so.  Device buffers are torch CUDA tensors (PyTorch is used
for device memory and streams); planner tables are numpy arrays.  A non-zero
status raises Fp8zError.  There is no fallback: if the library is missing or
was not built, loading fails loudly.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libfp8z.so")

BLOCK = 128
BLOCK_ELEMS = BLOCK * BLOCK
STATIC_GRAD_MAPS = 1024      # FP8Z_STATIC_GRAD_MAPS: params the no-allocation row-major step takes

FP8Z_OK, FP8Z_EINVAL, FP8Z_EALIGN, FP8Z_ENOSPACE = 0, -1, -2, -3
FP8Z_ECUDA, FP8Z_ETIMEOUT, FP8Z_EUNSUPPORTED = -4, -5, -6
FP8Z_SPLIT_BLOCKWISE, FP8Z_SPLIT_PARAMWISE = 0, 1
FP8Z_SCALE_EXACT, FP8Z_SCALE_POW2 = 0, 1
FP8Z_DECAY_PRE, FP8Z_DECAY_POST = 0, 1

# numpy views of the ABI structs (include/fp8z.h)
param_shape_dtype = np.dtype([("e", "<i8"), ("rows", "<i8"), ("cols", "<i8")])
param_entry_dtype = np.dtype([
    ("blk_offset", "<i8"), ("t_offset", "<i8"), ("t_scale_offset", "<i8"),
    ("e", "<i8"), ("rows", "<i8"), ("cols", "<i8"),
    ("hb", "<i4"), ("wb", "<i4"), ("bucket", "<i4"), ("reserved", "<i4"),
])
shard_dtype = np.dtype([("blk_begin", "<i8"), ("blk_count_real", "<i8"), ("blk_capacity", "<i8")])
block_desc_dtype = np.dtype([
    ("param", "<i4"), ("e", "<i4"), ("brow", "<i4"), ("bcol", "<i4"),
    ("valid_rows", "<u2"), ("valid_cols", "<u2"),
])
plan_summary_dtype = np.dtype([
    ("real_elems", "<i8"), ("total_blocks", "<i8"), ("fold_pad_elems", "<i8"),
    ("shard_pad_elems", "<i8"), ("capacity_blocks", "<i8"), ("naive_straddled_blocks", "<i8"),
])
assert param_entry_dtype.itemsize == 64 and block_desc_dtype.itemsize == 20

EXPORTED = ("fp8z_plan_shards", "fp8z_adamw_requant_step", "fp8z_adamw_requant_step_rowmajor",
            "fp8z_adamw_requant_step_mx", "fp8z_adamw_requant_step_rowmajor_static",
            "fp8z_encode_grad_maps", "fp8z_dequant",
            "fp8z_transpose_fp8", "fp8z_fold", "fp8z_unfold", "fp8z_quantize_rowwise",
            "fp8z_transpose_rowwise", "fp8z_dequant_rowwise", "fp8z_e4m3_encode_bits",
            "fp8z_watchdog_selftest", "fp8z_set_wait_limit_ns", "fp8z_get_wait_limit_ns",
            "fp8z_status_string")


class fp8z_adamw_hparams(ctypes.Structure):
    _fields_ = [
        ("lr", ctypes.c_float), ("beta1", ctypes.c_float), ("beta2", ctypes.c_float),
        ("eps", ctypes.c_float), ("weight_decay", ctypes.c_float), ("step", ctypes.c_int64),
        ("fp8_max", ctypes.c_float), ("min_scale", ctypes.c_float),
        ("scale_mode", ctypes.c_int32), ("decay_mode", ctypes.c_int32),
    ]


assert ctypes.sizeof(fp8z_adamw_hparams) == 48


def hparams(lr=1e-4, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1, step=1,
            fp8_max=448.0, min_scale=1e-6, scale_mode=FP8Z_SCALE_EXACT,
            decay_mode=FP8Z_DECAY_PRE) -> fp8z_adamw_hparams:
    return fp8z_adamw_hparams(lr, beta1, beta2, eps, weight_decay, step, fp8_max, min_scale,
                              scale_mode, decay_mode)


class Fp8zError(RuntimeError):
    def __init__(self, fn, status):
        self.status = status
        super().__init__(f"{fn}: {fp8z_status_string(status)} ({status})")


_lib = None


def lib():
    """Load libfp8z.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: build it with "
                              "`python -c 'import __graft_entry__ as g; g.build()'`")
        L = ctypes.CDLL(LIB_PATH)
        P, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32
        L.fp8z_plan_shards.argtypes = [P, i32, i32, i32, P, P, P, i64, P]
        L.fp8z_adamw_requant_step.argtypes = [P, P, P, P, P, P, i64, i64, i64, P, P, i32,
                                              P, i64, P, i64,
                                              ctypes.POINTER(fp8z_adamw_hparams), P, P]
        L.fp8z_adamw_requant_step_rowmajor.argtypes = [P, P, P, P, P, i64, P, i64, i64, i64, P, P, i32,
                                                       P, i64, P, i64,
                                                       ctypes.POINTER(fp8z_adamw_hparams), P, P]
        L.fp8z_encode_grad_maps.argtypes = [P, P, i32, P]
        L.fp8z_adamw_requant_step_rowmajor_static.argtypes = [P, P, P, P, P, P, i64, P, i64, i64, i64, P,
                                                              P, i32, P, i64, P, i64,
                                                              ctypes.POINTER(fp8z_adamw_hparams), P, P]
        L.fp8z_adamw_requant_step_mx.argtypes = [P, P, P, P, P, P, i64, i64, i64, P,
                                                 ctypes.POINTER(fp8z_adamw_hparams), P, P]
        L.fp8z_dequant.argtypes = [P, P, i64, P, P, P]
        L.fp8z_transpose_fp8.argtypes = [P, P, P, P, P, P, P]
        L.fp8z_fold.argtypes = [P, i32, P, P, P, P]
        L.fp8z_unfold.argtypes = [P, i32, P, P, P, P]
        L.fp8z_quantize_rowwise.argtypes = [P, i64, i64, i32, P, P, P]
        L.fp8z_transpose_rowwise.argtypes = [P, P, i64, i64, P, P, P]
        L.fp8z_dequant_rowwise.argtypes = [P, P, i64, i64, i32, P, P]
        L.fp8z_e4m3_encode_bits.argtypes = [ctypes.c_uint32, i64, P, P]
        L.fp8z_watchdog_selftest.argtypes = [P, i64, P]
        L.fp8z_set_wait_limit_ns.argtypes = [i64]
        L.fp8z_get_wait_limit_ns.argtypes = []
        L.fp8z_status_string.argtypes = [ctypes.c_int]
        L.fp8z_status_string.restype = ctypes.c_char_p
        for name in EXPORTED:
            if name != "fp8z_status_string":
                getattr(L, name).restype = ctypes.c_int
        L.fp8z_get_wait_limit_ns.restype = i64
        _lib = L
    return _lib


def fp8z_status_string(status: int) -> str:
    return lib().fp8z_status_string(int(status)).decode()


def _check(fn, rc):
    if rc != FP8Z_OK:
        raise Fp8zError(fn, rc)


def _dptr(t, dtype=None, name="tensor"):
    """Device pointer of a contiguous CUDA tensor on the current device (None
    -> NULL).  The library launches on the current device, so a tensor of
    another GPU is refused here rather than read through a foreign pointer."""
    if t is None:
        return None
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    import torch
    cur = torch.cuda.current_device()
    if t.device.index is not None and t.device.index != cur:
        raise ValueError(f"{name} is on {t.device}, but the current device is cuda:{cur}")
    return t.data_ptr()


DESC_BYTES = block_desc_dtype.itemsize       # 20
ENTRY_BYTES = param_entry_dtype.itemsize     # 64


def _check_tables(cap, desc, params, nparams):
    """The kernels read desc[b] for every block b < capacity and params[i] for
    i < nparams: a shorter table would be read past its end on the device, so
    it is refused here, before any launch."""
    if desc is not None and desc.numel() * desc.element_size() < cap * DESC_BYTES:
        raise ValueError(f"desc holds {desc.numel() * desc.element_size()} bytes, "
                         f"{cap} blocks need {cap * DESC_BYTES}")
    if params is not None and params.numel() * params.element_size() < int(nparams) * ENTRY_BYTES:
        raise ValueError(f"params holds {params.numel() * params.element_size()} bytes, "
                         f"{int(nparams)} entries need {int(nparams) * ENTRY_BYTES}")


def _stream_handle(stream):
    import torch
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


# ---------------------------------------------------------------- planner
def fp8z_plan_shards(shapes, dp, split=FP8Z_SPLIT_BLOCKWISE, with_blocks=True):
    """shapes: iterable of (e, rows, cols).  Returns (params, shards, blocks, summary)
    as numpy structured arrays (blocks None when with_blocks is False)."""
    sh = np.array([tuple(int(x) for x in s) for s in shapes], dtype=param_shape_dtype)
    n = len(sh)
    params = np.zeros(max(n, 1), dtype=param_entry_dtype)
    shards = np.zeros(max(int(dp), 1), dtype=shard_dtype)
    summ = np.zeros(1, dtype=plan_summary_dtype)
    L = lib()
    rc = L.fp8z_plan_shards(sh.ctypes.data if n else None, n, int(dp), int(split),
                            params.ctypes.data, shards.ctypes.data, None, 0, summ.ctypes.data)
    _check("fp8z_plan_shards", rc)
    blocks = None
    if with_blocks:
        cap = int(summ["capacity_blocks"][0])
        blocks = np.zeros(max(cap, 1), dtype=block_desc_dtype)
        rc = L.fp8z_plan_shards(sh.ctypes.data if n else None, n, int(dp), int(split),
                                params.ctypes.data, shards.ctypes.data, blocks.ctypes.data,
                                cap, summ.ctypes.data)
        _check("fp8z_plan_shards", rc)
        blocks = blocks[:cap]
    return params[:n], shards[:int(dp)], blocks, summ[0]


def table_to_device(arr, device="cuda"):
    """Copy a planner table (numpy structured array) into a CUDA byte tensor."""
    import torch
    raw = np.ascontiguousarray(arr).view(np.uint8).reshape(-1)
    return torch.from_numpy(raw.copy()).to(device)


# ------------------------------------------------------------------ device
def fp8z_adamw_requant_step(p, g, m, v, w_fp8, inv_scale, blk_begin, nblk, hp,
                            desc=None, params=None, nparams=0, w_fp8_t=None,
                            inv_scale_t=None, dev_status=None, stream=None):
    """Fused AdamW + blockwise E4M3 requant of blocks [blk_begin, blk_begin+nblk).

    p, g, m, v: float32 CUDA tensors of capacity*16384 elements; w_fp8 uint8 of
    the same count; inv_scale float32 [capacity]; desc / params: CUDA byte
    tensors from table_to_device (or None); w_fp8_t uint8, inv_scale_t float32
    (optional column-major copy); dev_status int32 CUDA tensor (or None).
    """
    import torch
    cap = p.numel() // BLOCK_ELEMS
    for t, name in ((g, "g"), (m, "m"), (v, "v"), (w_fp8, "w_fp8")):
        if t.numel() != p.numel():
            raise ValueError(f"{name} must have as many elements as p")
    if inv_scale.numel() < cap:
        raise ValueError("inv_scale must hold one scale per block")
    _check_tables(cap, desc, params, nparams)
    rc = lib().fp8z_adamw_requant_step(
        _dptr(p, torch.float32, "p"), _dptr(g, torch.float32, "g"),
        _dptr(m, torch.float32, "m"), _dptr(v, torch.float32, "v"),
        _dptr(w_fp8, torch.uint8, "w_fp8"), _dptr(inv_scale, torch.float32, "inv_scale"),
        cap, int(blk_begin), int(nblk),
        _dptr(desc, torch.uint8, "desc"), _dptr(params, torch.uint8, "params"), int(nparams),
        _dptr(w_fp8_t, torch.uint8, "w_fp8_t"), 0 if w_fp8_t is None else w_fp8_t.numel(),
        _dptr(inv_scale_t, torch.float32, "inv_scale_t"),
        0 if inv_scale_t is None else inv_scale_t.numel(),
        ctypes.byref(hp), _dptr(dev_status, torch.int32, "dev_status"), _stream_handle(stream))
    _check("fp8z_adamw_requant_step", rc)


def fp8z_adamw_requant_step_mx(p, g, m, v, w_fp8, mx_scale, blk_begin, nblk, hp, desc=None,
                               dev_status=None, stream=None):
    """MXFP8 output: E4M3 codes in w_fp8 and one E8M0 byte per 32 elements of a
    block row in mx_scale (uint8, capacity*512)."""
    import torch
    cap = p.numel() // BLOCK_ELEMS
    for t, name in ((g, "g"), (m, "m"), (v, "v"), (w_fp8, "w_fp8")):
        if t.numel() != p.numel():
            raise ValueError(f"{name} must have as many elements as p")
    if mx_scale.numel() < cap * (BLOCK_ELEMS // 32):
        raise ValueError("mx_scale must hold 512 bytes per block")
    _check_tables(cap, desc, None, 0)
    rc = lib().fp8z_adamw_requant_step_mx(
        _dptr(p, torch.float32, "p"), _dptr(g, torch.float32, "g"), _dptr(m, torch.float32, "m"),
        _dptr(v, torch.float32, "v"), _dptr(w_fp8, torch.uint8, "w_fp8"),
        _dptr(mx_scale, torch.uint8, "mx_scale"), cap, int(blk_begin), int(nblk),
        _dptr(desc, torch.uint8, "desc"), ctypes.byref(hp), _dptr(dev_status, torch.int32, "dev_status"),
        _stream_handle(stream))
    _check("fp8z_adamw_requant_step_mx", rc)


def fp8z_encode_grad_maps(grads, params, device="cuda"):
    """Tensor maps over each param's row-major FP32 grad (torch CUDA tensors of
    shape [e, rows, cols] or flat), returned as a CUDA byte tensor to pass as
    g_maps.  The grads must stay alive while the maps are used."""
    import torch
    n = len(params)
    if len(grads) != n:
        raise ValueError("one grad per param")
    for gt, pe in zip(grads, params):
        if gt.dtype != torch.float32 or gt.numel() < int(pe["e"]) * int(pe["rows"]) * int(pe["cols"]):
            raise ValueError("grad must be float32 and hold the whole param")
    ptrs = (ctypes.c_void_p * n)(*[_dptr(gt, torch.float32, "grad") for gt in grads])
    raw = np.zeros(n * 128 + 64, dtype=np.uint8)
    off = (-raw.ctypes.data) % 64
    host = raw[off:off + n * 128]
    ent = np.ascontiguousarray(params, dtype=param_entry_dtype)
    rc = lib().fp8z_encode_grad_maps(ptrs, ent.ctypes.data, n, host.ctypes.data)
    _check("fp8z_encode_grad_maps", rc)
    return torch.from_numpy(host.copy()).to(device)


def fp8z_adamw_requant_step_rowmajor(p, m, v, g_maps, w_row, inv_scale, blk_begin, nblk, hp,
                                     desc, params, nparams, w_fp8_t=None, inv_scale_t=None,
                                     dev_status=None, stream=None):
    """The fused step reading row-major grads (through g_maps) and writing the
    E4M3 weights row-major into w_row (each param at its t_offset)."""
    import torch
    cap = p.numel() // BLOCK_ELEMS
    for t, name in ((m, "m"), (v, "v")):
        if t.numel() != p.numel():
            raise ValueError(f"{name} must have as many elements as p")
    if inv_scale.numel() < cap:
        raise ValueError("inv_scale must hold one scale per block")
    if g_maps.numel() < nparams * 128:
        raise ValueError("g_maps must hold one 128-byte map per param")
    if desc is None or params is None:
        raise ValueError("the row-major step needs desc and params")
    _check_tables(cap, desc, params, nparams)
    rc = lib().fp8z_adamw_requant_step_rowmajor(
        _dptr(p, torch.float32, "p"), _dptr(m, torch.float32, "m"), _dptr(v, torch.float32, "v"),
        _dptr(g_maps, torch.uint8, "g_maps"), _dptr(w_row, torch.uint8, "w_row"), w_row.numel(),
        _dptr(inv_scale, torch.float32, "inv_scale"), cap, int(blk_begin), int(nblk),
        _dptr(desc, torch.uint8, "desc"), _dptr(params, torch.uint8, "params"), int(nparams),
        _dptr(w_fp8_t, torch.uint8, "w_fp8_t"), 0 if w_fp8_t is None else w_fp8_t.numel(),
        _dptr(inv_scale_t, torch.float32, "inv_scale_t"),
        0 if inv_scale_t is None else inv_scale_t.numel(),
        ctypes.byref(hp), _dptr(dev_status, torch.int32, "dev_status"), _stream_handle(stream))
    _check("fp8z_adamw_requant_step_rowmajor", rc)


def fp8z_adamw_requant_step_rowmajor_static(p, m, v, grads, params_host, w_row, inv_scale, blk_begin,
                                            nblk, hp, desc, params, nparams, w_fp8_t=None,
                                            inv_scale_t=None, dev_status=None, stream=None):
    """The row-major step for callers that cannot allocate device memory: the
    grad tensor maps go into an array inside the library instead of a
    caller-allocated g_maps buffer.  grads: one row-major float32 CUDA tensor
    per param; params_host: the planner's param table (numpy, host)."""
    import torch
    cap = p.numel() // BLOCK_ELEMS
    for t, name in ((m, "m"), (v, "v")):
        if t.numel() != p.numel():
            raise ValueError(f"{name} must have as many elements as p")
    if inv_scale.numel() < cap:
        raise ValueError("inv_scale must hold one scale per block")
    if desc is None or params is None:
        raise ValueError("the row-major step needs desc and params")
    _check_tables(cap, desc, params, nparams)
    ent = np.ascontiguousarray(params_host, dtype=param_entry_dtype)
    if len(grads) != int(nparams) or len(ent) != int(nparams):
        raise ValueError("one grad and one host param entry per param")
    if int(nparams) > STATIC_GRAD_MAPS:
        raise ValueError(f"{int(nparams)} params: the library's map array holds at most "
                         f"{STATIC_GRAD_MAPS}; use fp8z_adamw_requant_step_rowmajor with a g_maps buffer")
    for gt, pe in zip(grads, ent):
        if gt.dtype != torch.float32 or gt.numel() < int(pe["e"]) * int(pe["rows"]) * int(pe["cols"]):
            raise ValueError("grad must be float32 and hold the whole param")
    ptrs = (ctypes.c_void_p * len(grads))(*[_dptr(gt, torch.float32, "grad") for gt in grads])
    rc = lib().fp8z_adamw_requant_step_rowmajor_static(
        _dptr(p, torch.float32, "p"), _dptr(m, torch.float32, "m"), _dptr(v, torch.float32, "v"),
        ptrs, ent.ctypes.data, _dptr(w_row, torch.uint8, "w_row"), w_row.numel(),
        _dptr(inv_scale, torch.float32, "inv_scale"), cap, int(blk_begin), int(nblk),
        _dptr(desc, torch.uint8, "desc"), _dptr(params, torch.uint8, "params"), int(nparams),
        _dptr(w_fp8_t, torch.uint8, "w_fp8_t"), 0 if w_fp8_t is None else w_fp8_t.numel(),
        _dptr(inv_scale_t, torch.float32, "inv_scale_t"),
        0 if inv_scale_t is None else inv_scale_t.numel(),
        ctypes.byref(hp), _dptr(dev_status, torch.int32, "dev_status"), _stream_handle(stream))
    _check("fp8z_adamw_requant_step_rowmajor_static", rc)


def fp8z_dequant(w_fp8, inv_scale, nblk, out, dev_status=None, stream=None):
    import torch
    if w_fp8.numel() < nblk * BLOCK_ELEMS or out.numel() < nblk * BLOCK_ELEMS or inv_scale.numel() < nblk:
        raise ValueError("buffers smaller than nblk blocks")
    rc = lib().fp8z_dequant(_dptr(w_fp8, torch.uint8, "w_fp8"),
                            _dptr(inv_scale, torch.float32, "inv_scale"), int(nblk),
                            _dptr(out, torch.float32, "out"), _dptr(dev_status, torch.int32, "dev_status"),
                            _stream_handle(stream))
    _check("fp8z_dequant", rc)


def fp8z_transpose_fp8(w_fp8, inv_scale, entry, out, inv_scale_t, dev_status=None, stream=None):
    """entry: one param_entry_dtype record (host).  out: uint8 [E, W, H];
    inv_scale_t: float32 [E, Wb, Hb]; dev_status: optional int32 device word."""
    import torch
    ent = np.array([entry], dtype=param_entry_dtype)
    E, H, W = int(entry["e"]), int(entry["rows"]), int(entry["cols"])
    nb = E * int(entry["hb"]) * int(entry["wb"])
    if out.numel() < E * H * W or inv_scale_t.numel() < nb:
        raise ValueError("output buffers too small")
    if w_fp8.numel() < (int(entry["blk_offset"]) + nb) * BLOCK_ELEMS:
        raise ValueError("w_fp8 does not hold the param's blocks")
    if inv_scale.numel() < int(entry["blk_offset"]) + nb:
        raise ValueError("inv_scale does not hold the param's scales")
    rc = lib().fp8z_transpose_fp8(_dptr(w_fp8, torch.uint8, "w_fp8"),
                                  _dptr(inv_scale, torch.float32, "inv_scale"), ent.ctypes.data,
                                  _dptr(out, torch.uint8, "out"),
                                  _dptr(inv_scale_t, torch.float32, "inv_scale_t"),
                                  _dptr(dev_status, torch.int32, "dev_status"), _stream_handle(stream))
    _check("fp8z_transpose_fp8", rc)


def _entry_checks(entry, folded, rowmajor):
    E, H, W = int(entry["e"]), int(entry["rows"]), int(entry["cols"])
    nb = E * int(entry["hb"]) * int(entry["wb"])
    if rowmajor.numel() < E * H * W:
        raise ValueError("row-major tensor smaller than the param")
    if folded.numel() < (int(entry["blk_offset"]) + nb) * BLOCK_ELEMS:
        raise ValueError("folded buffer does not hold the param's blocks")
    if folded.dtype != rowmajor.dtype or folded.element_size() not in (1, 4):
        raise ValueError("fold/unfold: both tensors float32 or both uint8")


def fp8z_fold(src, entry, blocks, dev_status=None, stream=None):
    """Row-major [E, rows, cols] -> the param's 128x128 blocks in the folded buffer."""
    import torch
    _entry_checks(entry, blocks, src)
    ent = np.array([entry], dtype=param_entry_dtype)
    rc = lib().fp8z_fold(_dptr(src, None, "src"), src.element_size(), ent.ctypes.data,
                         _dptr(blocks, None, "blocks"), _dptr(dev_status, torch.int32, "dev_status"),
                         _stream_handle(stream))
    _check("fp8z_fold", rc)


def fp8z_unfold(blocks, entry, dst, dev_status=None, stream=None):
    """The param's 128x128 blocks in the folded buffer -> row-major [E, rows, cols]."""
    import torch
    _entry_checks(entry, blocks, dst)
    ent = np.array([entry], dtype=param_entry_dtype)
    rc = lib().fp8z_unfold(_dptr(blocks, None, "blocks"), blocks.element_size(), ent.ctypes.data,
                           _dptr(dst, None, "dst"), _dptr(dev_status, torch.int32, "dev_status"),
                           _stream_handle(stream))
    _check("fp8z_unfold", rc)


def fp8z_quantize_rowwise(x, pow2, q, s, stream=None):
    """x: float32 [rows, cols] -> q uint8 [rows, cols], s float32 [rows, cols/128]."""
    import torch
    rows, cols = x.shape
    if q.numel() < rows * cols or s.numel() < rows * (cols // BLOCK):
        raise ValueError("output buffers too small")
    rc = lib().fp8z_quantize_rowwise(_dptr(x, torch.float32, "x"), rows, cols, int(bool(pow2)),
                                     _dptr(q, torch.uint8, "q"), _dptr(s, torch.float32, "s"),
                                     _stream_handle(stream))
    _check("fp8z_quantize_rowwise", rc)


def fp8z_transpose_rowwise(q, s, q_t, s_t, stream=None):
    """Row-wise q [rows, cols], s [rows, cols/128] -> column-wise q_t [cols, rows], s_t [cols, rows/128]."""
    import torch
    rows, cols = q.shape
    if q_t.numel() < rows * cols or s_t.numel() < cols * (rows // BLOCK) or s.numel() < rows * (cols // BLOCK):
        raise ValueError("buffers too small")
    rc = lib().fp8z_transpose_rowwise(_dptr(q, torch.uint8, "q"), _dptr(s, torch.float32, "s"), rows, cols,
                                      _dptr(q_t, torch.uint8, "q_t"), _dptr(s_t, torch.float32, "s_t"),
                                      _stream_handle(stream))
    _check("fp8z_transpose_rowwise", rc)


def fp8z_dequant_rowwise(q, s, out, transpose=False, stream=None):
    """Row-wise codes q [rows, cols] and scales s [rows, cols/128] -> float32 out
    [rows, cols], or [cols, rows] when transpose is set."""
    import torch
    rows, cols = q.shape
    if out.numel() < rows * cols or s.numel() < rows * (cols // BLOCK):
        raise ValueError("buffers too small")
    rc = lib().fp8z_dequant_rowwise(_dptr(q, torch.uint8, "q"), _dptr(s, torch.float32, "s"), rows, cols,
                                    int(bool(transpose)), _dptr(out, torch.float32, "out"),
                                    _stream_handle(stream))
    _check("fp8z_dequant_rowwise", rc)


def fp8z_e4m3_encode_bits(first_bits, n, out, stream=None):
    import torch
    if out.numel() < n:
        raise ValueError("out too small")
    rc = lib().fp8z_e4m3_encode_bits(int(first_bits) & 0xFFFFFFFF, int(n),
                                     _dptr(out, torch.uint8, "out"), _stream_handle(stream))
    _check("fp8z_e4m3_encode_bits", rc)


def fp8z_watchdog_selftest(dev_status, timeout_ns, stream=None):
    import torch
    rc = lib().fp8z_watchdog_selftest(_dptr(dev_status, torch.int32, "dev_status"),
                                      int(timeout_ns), _stream_handle(stream))
    _check("fp8z_watchdog_selftest", rc)


def fp8z_set_wait_limit_ns(ns):
    """Limit (ns) of every bounded device wait in later launches; 0 restores 2 s."""
    _check("fp8z_set_wait_limit_ns", lib().fp8z_set_wait_limit_ns(int(ns)))


def fp8z_get_wait_limit_ns():
    return int(lib().fp8z_get_wait_limit_ns())
