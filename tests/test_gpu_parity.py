"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle,
element by element on the same seeded inputs.

The library is built with IEEE division and square root and no FMA
contraction, and applies the same per-element operation order, so the bar is
bit-exact: FP32 p', m', v', inverse scales, E4M3 codes (an E4M3 NaN code may
differ only in its sign bit), the column-major copy and its scale grid.
"""
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from blockwise_fp8_zero_gb300 import fp8z, workloads  # noqa: E402

from _gpu_util import Case, assert_bitexact, oracle_blocks  # noqa: E402

pytestmark = pytest.mark.gpu
BLK = fp8z.BLOCK_ELEMS


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from blockwise_fp8_zero_gb300 import build
    build.build()
    fp8z.lib()


def test_e4m3_cast_all_2_32_inputs(oracle):
    """The kernel's float->E4M3 cast on every float32 bit pattern."""
    chunk = 1 << 28
    out = torch.empty(chunk, dtype=torch.uint8, device="cuda")
    want = np.empty(chunk, np.uint8)
    threads = max(1, min(32, os.cpu_count() or 1))
    sub = chunk // threads
    with ThreadPoolExecutor(threads) as ex:
        for first in range(0, 1 << 32, chunk):
            fp8z.fp8z_e4m3_encode_bits(first, chunk, out)
            list(ex.map(lambda i: oracle.e4m3_encode_bits_range(
                first + i * sub, sub, want[i * sub:(i + 1) * sub]), range(threads)))
            got = out.cpu().numpy()
            # NaN inputs: both sides must give a NaN code; the sign bit is free
            bits = np.arange(chunk, dtype=np.uint32) + np.uint32(first)
            nan_in = ((bits & 0x7F800000) == 0x7F800000) & ((bits & 0x7FFFFF) != 0)
            ok = (got == want) | (nan_in & ((got & 0x7F) == 0x7F))
            assert np.all(ok), f"chunk {first:#x}: {np.count_nonzero(~ok)} mismatches"


def test_single_256x384_step1(oracle):
    """One 256x384 weight, one shard, step 1, m = v = 0 (the small workload)."""
    w = workloads.get("single_256x384")
    c = Case(w.shapes, w.dp, w.split, dists=w.dists, seed=0)
    hp = fp8z.hparams(**w.hp)
    c.step(hp)
    assert_bitexact(c.results(), c.oracle(oracle, hp), c.processed)


TINY = [[(1, 1, 1)], [(1, 1, 129)], [(1, 129, 1)], [(1, 128, 128)], [(2, 130, 257)],
        [(1, 3, 5), (2, 128, 1), (1, 200, 200)], [(1, 7168, 576)], [(3, 384, 640)]]


@pytest.mark.parametrize("shapes", TINY)
@pytest.mark.parametrize("transposed", [False, True])
def test_ragged_shapes(oracle, shapes, transposed):
    c = Case(shapes, dp=1, seed=len(shapes), transposed=transposed)
    hp = fp8z.hparams(step=11)
    c.step(hp)
    assert_bitexact(c.results(), c.oracle(oracle, hp), c.processed)


# Larger shards with the column-major copy, fully checked: whole expert
# matrices with more block columns than CTAs (several blocks per CTA), a wide
# ragged param (hb = 3, wb = 201), whole params per param-wise bucket, and
# block-wise shards that cut an expert matrix.
@pytest.mark.parametrize("shapes,dp,split", [([(4, 1024, 5120)], 1, 0), ([(1, 256, 38400)], 1, 0),
                                             ([(2, 512, 10240), (2, 512, 10240)], 2, 1),
                                             ([(1, 300, 25700)], 1, 0), ([(1, 256, 38400)], 3, 0)])
def test_larger_shards_with_copy(oracle, shapes, dp, split):
    c = Case(shapes, dp=dp, split=split, seed=dp + len(shapes), transposed=True)
    hp = fp8z.hparams(step=4)
    c.step(hp)
    assert_bitexact(c.results(), c.oracle(oracle, hp), c.processed)


@pytest.mark.parametrize("kw", [dict(step=1), dict(step=1000), dict(decay_mode=1, step=5),
                                dict(scale_mode=1, step=3), dict(lr=3e-3, weight_decay=0.0, step=2),
                                dict(beta1=0.0, beta2=0.0, step=7), dict(min_scale=1e3, step=2)])
def test_hyperparameter_variants(oracle, kw):
    c = Case([(1, 300, 520), (2, 128, 256)], dp=2, seed=3, transposed=True)
    hp = fp8z.hparams(**kw)
    c.step(hp)
    assert_bitexact(c.results(), c.oracle(oracle, hp), c.processed)


def test_no_descriptor_full_blocks(oracle):
    c = Case([(4, 256, 256)], dp=1, seed=9)
    hp = fp8z.hparams(step=4)
    c.step(hp, use_desc=False)
    assert_bitexact(c.results(), c.oracle(oracle, hp, use_desc=False), c.processed)


def test_special_blocks(oracle):
    """All-zero block, a spike, tiny and huge values, NaN and Inf grads."""
    c = Case([(1, 128, 128 * 6)], dp=1, seed=5)
    for k in "pgmv":
        x = c.host[k].reshape(6, BLK)
        x[0] = 0.0                                      # all-zero block
        if k == "p":
            x[1, 77] = 3.0                              # spike
            x[2] *= 1e-30                               # tiny block values
            x[3] *= 1e11                                # amax > 448e6: the 1e-6 floor binds
        if k == "g":
            x[4, 5] = np.nan
            x[4, 6] = np.inf
            x[5, 9] = -np.inf
        c.dev[k].copy_(torch.from_numpy(c.host[k]))
    hp = fp8z.hparams(step=2)
    c.step(hp)
    assert_bitexact(c.results(), c.oracle(oracle, hp), c.processed)


def _random_hparams(rng):
    return dict(lr=float(10 ** rng.uniform(-7, -1)), beta1=float(rng.choice([0.0, rng.uniform(0, 0.99)])),
                beta2=float(rng.choice([0.0, rng.uniform(0, 0.9999)])), eps=float(10 ** rng.uniform(-12, -2)),
                weight_decay=float(rng.choice([0.0, rng.uniform(0, 1)])),
                step=int(10 ** rng.uniform(0, 6)), scale_mode=int(rng.integers(0, 2)),
                decay_mode=int(rng.integers(0, 2)),
                fp8_max=float(rng.choice([448.0, 240.0, 1.0 + rng.uniform(0, 447)])),
                min_scale=float(rng.choice([0.0, 1e-6, rng.uniform(0, 1e3)])))


@pytest.mark.parametrize("seed", range(24))
def test_hyperparameter_sweep(oracle, seed):
    """Seeded random hyper-parameters (every field the step reads, both scale
    and decay modes, steps up to 1e6) on a ragged two-param, two-shard layout
    with the column-major copy: the same bits as the oracle."""
    rng = np.random.default_rng(1000 + seed)
    c = Case([(1, 200, 300), (2, 130, 129)], dp=2, seed=seed, transposed=True)
    hp = fp8z.hparams(**_random_hparams(rng))
    c.step(hp)
    assert_bitexact(c.results(), c.oracle(oracle, hp), c.processed)


@pytest.mark.parametrize("scale_mode", [0, 1])
def test_extreme_magnitudes(oracle, scale_mode):
    """State and grads log-uniform over [1e-42, 1e38] with random signs (v kept
    >= 0), exact zeros mixed in: subnormal operands, g*g overflowing to Inf,
    quotients overflowing, blocks whose amax is subnormal or near FLT_MAX."""
    c = Case([(1, 256, 640)], dp=1, seed=9, transposed=True)
    rng = np.random.default_rng(77 + scale_mode)
    for k in "pgmv":
        n = c.host[k].size
        mag = 10.0 ** rng.uniform(-42, 38, n)
        x = (mag * rng.choice([-1.0, 1.0], n)).astype(np.float32)
        x[rng.random(n) < 0.02] = 0.0
        if k == "v":
            x = np.abs(x)
        c.host[k][:] = x
        c.dev[k].copy_(torch.from_numpy(c.host[k]))
    hp = fp8z.hparams(step=7, scale_mode=scale_mode)
    c.step(hp)
    assert_bitexact(c.results(), c.oracle(oracle, hp), c.processed)


def test_shard_launches_equal_one_launch(oracle):
    shapes = [(1, 640, 384), (2, 200, 300), (1, 128, 1000)]
    hp = fp8z.hparams(step=6)
    a = Case(shapes, dp=5, seed=2, transposed=True)
    a.step(hp)
    b = Case(shapes, dp=5, seed=2, transposed=True)
    b.step(hp, ranges=[(0, b.cap)])
    ra, rb = a.results(), b.results()
    for k in ("p", "m", "v", "q", "wt", "it"):
        assert np.array_equal(ra[k], rb[k]), k
    data = a.blocks["param"] >= 0
    assert np.array_equal(ra["inv"][data], rb["inv"][data])
    assert_bitexact(ra, a.oracle(oracle, hp), a.processed)


def test_repeated_steps(oracle):
    c = Case([(1, 256, 512)], dp=2, seed=8)
    ohost = {k: c.host[k].copy() for k in "pgmv"}
    for t in (1, 2, 3):
        hp = fp8z.hparams(step=t)
        c.step(hp)
        want = c.oracle(oracle, hp)
        assert_bitexact(c.results(), want, c.processed)
        for k in "pmv":
            c.host[k] = want[k]
    assert not np.array_equal(ohost["p"], c.host["p"])


def test_paramwise_equals_blockwise_per_param(oracle):
    shapes = [(1, 300, 200), (1, 128, 128), (2, 256, 130), (1, 64, 700)]
    hp = fp8z.hparams(step=7)
    res = []
    for split in (0, 1):
        c = Case(shapes, dp=3, split=split, seed=0)
        # same values per param in both layouts: fill by param from one host draw
        rng = np.random.default_rng(1)
        for k, sd in zip("pgmv", (0.02, 1e-3, 3e-4, 1e-6)):
            flat = np.zeros(c.cap * BLK, np.float32)
            for i, (E, H, W) in enumerate(shapes):
                x = rng.normal(0, sd, (E, H, W)) if k != "v" else rng.uniform(0.5, 1.5, (E, H, W)) * sd
                f = oracle.fold(x.astype(np.float32)).ravel()
                o = int(c.params[i]["blk_offset"]) * BLK
                flat[o:o + f.size] = f
            c.host[k] = flat
            c.dev[k].copy_(torch.from_numpy(flat))
        c.step(hp)
        r = c.results()
        assert_bitexact(r, c.oracle(oracle, hp), c.processed)
        per = []
        for i, (E, H, W) in enumerate(shapes):
            o = int(c.params[i]["blk_offset"])
            nb = E * int(c.params[i]["hb"]) * int(c.params[i]["wb"])
            per.append((r["p"][o * BLK:(o + nb) * BLK], r["q"][o * BLK:(o + nb) * BLK], r["inv"][o:o + nb]))
        res.append(per)
    for a, b in zip(*res):
        for x, y in zip(a, b):
            assert np.array_equal(x, y)


def test_dense_h7168_full(oracle):
    """Dense hidden-7168 layer set, 8 shards (one launch each), every block."""
    w = workloads.get("dense_h7168")
    params, shards, blocks, summ = fp8z.fp8z_plan_shards(w.shapes, w.dp, w.split)
    cap = int(summ["capacity_blocks"])
    dev = workloads.make_state(w, blocks, "cuda", seed=0)
    host = {k: dev[k].cpu().numpy() for k in "pgmv"}
    q = torch.zeros(cap * BLK, dtype=torch.uint8, device="cuda")
    inv = torch.zeros(cap, dtype=torch.float32, device="cuda")
    desc = fp8z.table_to_device(blocks)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    hp = fp8z.hparams(**w.hp)
    for s in shards:
        fp8z.fp8z_adamw_requant_step(dev["p"], dev["g"], dev["m"], dev["v"], q, inv,
                                     int(s["blk_begin"]), int(s["blk_count_real"]), hp,
                                     desc=desc, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    d = oracle.plan_shards(w.shapes, w.dp, w.split)[2]       # the oracle's own plan
    qo, invo = oracle_blocks(oracle, hp, host["p"], host["g"], host["m"], host["v"], d)
    got = dict(p=dev["p"].cpu().numpy(), m=dev["m"].cpu().numpy(), v=dev["v"].cpu().numpy(),
               q=q.cpu().numpy(), inv=inv.cpu().numpy())
    assert_bitexact(got, dict(p=host["p"], m=host["m"], v=host["v"], q=qo, inv=invo))


def test_dequant(oracle):
    # codes and scales of a step, made by the oracle and uploaded: no input of
    # the oracle comes from the library
    c = Case([(1, 384, 640)], dp=1, seed=4)
    ref = c.oracle(oracle, fp8z.hparams(step=2))
    out = torch.empty(c.cap * BLK, dtype=torch.float32, device="cuda")
    fp8z.fp8z_dequant(torch.from_numpy(ref["q"]).cuda(), torch.from_numpy(ref["inv"]).cuda(), c.cap, out)
    torch.cuda.synchronize()
    want = oracle.dequant(ref["q"], ref["inv"], c.cap)
    assert np.array_equal(out.cpu().numpy().view(np.uint32), want.view(np.uint32))


@pytest.mark.parametrize("nblk", [1, 153, 2000])
def test_dequant_every_code(oracle, nblk):
    # every finite code and its negation, spread over many blocks per persistent
    # CTA, each block with its own inverse scale (powers of two and not)
    rng = np.random.default_rng(nblk)
    codes = rng.integers(0, 256, nblk * BLK, dtype=np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x00                      # NaN codes: never produced by the step
    codes[:254] = [c for c in range(256) if (c & 0x7F) != 0x7F]
    inv = (rng.uniform(0.5, 2.0, nblk) * 2.0 ** rng.integers(-20, 20, nblk)).astype(np.float32)
    inv[::3] = 2.0 ** rng.integers(-30, 30, inv[::3].size).astype(np.float32)
    out = torch.full((nblk * BLK,), float("nan"), dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    fp8z.fp8z_dequant(torch.from_numpy(codes).cuda(), torch.from_numpy(inv).cuda(), nblk, out, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    want = oracle.dequant(codes, inv, nblk)
    assert np.array_equal(out.cpu().numpy().view(np.uint32), want.view(np.uint32))


# rows a multiple of 16 take the TMA kernel (ragged edges clipped by the
# tensor-map store, several blocks per persistent CTA), the rest the plain one
@pytest.mark.parametrize("shape", [(1, 384, 640), (2, 300, 260), (1, 129, 1), (3, 7168 // 28, 576),
                                   (2, 272, 200), (1, 16, 16), (8, 1024, 1152), (40, 512, 512),
                                   (3, 1040, 7)])
def test_standalone_transpose(oracle, shape):
    # the codes and scales of a step, made by the oracle, go to both sides
    c = Case([shape], dp=1, seed=6)
    ref = c.oracle(oracle, fp8z.hparams(step=3))
    E, H, W = shape
    pe = c.params[0]
    out = torch.full((E * W * H,), 0xA5, dtype=torch.uint8, device="cuda")
    it = torch.zeros(E * int(pe["wb"]) * int(pe["hb"]), dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    fp8z.fp8z_transpose_fp8(torch.from_numpy(ref["q"]).cuda(), torch.from_numpy(ref["inv"]).cuda(), pe, out,
                            it, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0, fp8z.fp8z_status_string(st.item())
    ent = c.oracle_tables(oracle)[0][0]
    wt, wit = oracle.transpose_fp8(ref["q"], ref["inv"], ent)
    assert np.array_equal(out.cpu().numpy(), wt.ravel())
    assert np.array_equal(it.cpu().numpy(), wit.ravel())


def test_watchdog_reports_timeout_and_context_survives(oracle):
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    fp8z.fp8z_watchdog_selftest(st, 20_000_000)         # 20 ms
    torch.cuda.synchronize()
    assert st.item() == fp8z.FP8Z_ETIMEOUT
    # the context is still usable
    c = Case([(1, 128, 256)], dp=1, seed=1)
    hp = fp8z.hparams(step=1)
    c.step(hp)
    assert_bitexact(c.results(), c.oracle(oracle, hp), c.processed)


def test_bad_descriptor_is_reported_not_written(oracle):
    c = Case([(1, 256, 256)], dp=1, seed=2, transposed=True)
    bad = c.blocks.copy()
    bad["param"][1] = 7                                 # no such param
    bad["bcol"][2] = 99                                 # outside the param
    c.desc_dev = fp8z.table_to_device(bad)
    hp = fp8z.hparams(step=1)
    fp8z.fp8z_adamw_requant_step(c.dev["p"], c.dev["g"], c.dev["m"], c.dev["v"], c.w_fp8, c.inv,
                                 0, c.cap, hp, desc=c.desc_dev, params=c.params_dev, nparams=1,
                                 w_fp8_t=c.wt, inv_scale_t=c.it, dev_status=c.status)
    torch.cuda.synchronize()
    assert c.status.item() == fp8z.FP8Z_EINVAL
    # main outputs are still right (the descriptors only gate the copy)
    r = c.results()
    c.transposed = False
    want = c.oracle(oracle, hp)
    for k in ("p", "m", "v", "q"):
        assert np.array_equal(r[k], want[k]), k


def test_checkpoint_resume_is_bit_identical(oracle):
    """The step keeps no state between calls: saving p, m, v to the host after
    step t and resuming from the saved copy gives the same step t+1 as an
    uninterrupted run."""
    shapes = [(1, 384, 520), (2, 128, 200)]
    a = Case(shapes, dp=2, seed=11, transposed=True)
    for t in (1, 2, 3):
        a.step(fp8z.hparams(step=t))
    b = Case(shapes, dp=2, seed=11, transposed=True)
    for t in (1, 2):
        b.step(fp8z.hparams(step=t))
    saved = {k: b.dev[k].cpu().numpy().copy() for k in "pmv"}
    c = Case(shapes, dp=2, seed=11, transposed=True)          # fresh buffers, same grads
    for k in "pmv":
        c.dev[k].copy_(torch.from_numpy(saved[k]))
    c.step(fp8z.hparams(step=3))
    ra, rc = a.results(), c.results()
    for k in ("p", "m", "v", "q", "wt", "it"):
        assert np.array_equal(ra[k], rc[k]), k


@pytest.mark.parametrize("shapes", [[(1, 256, 384)], [(2, 130, 257)], [(1, 200, 100), (1, 7, 1000)]])
def test_mxfp8_step(oracle, shapes):
    """MXFP8 output variant against the oracle, bit for bit (codes, E8M0 bytes, state)."""
    c = Case(shapes, dp=2, seed=17)
    # a spike, tiny values and a zero group
    x = c.host["p"].reshape(-1, 32)
    x[3, 5] = 4.0
    x[10] *= 1e-7
    for k in "pgmv":
        c.host[k].reshape(-1, 32)[20] = 0.0
        c.dev[k].copy_(torch.from_numpy(c.host[k]))
    hp = fp8z.hparams(step=6)
    mx = torch.zeros(c.cap * 512, dtype=torch.uint8, device="cuda")
    for s in c.shards:
        fp8z.fp8z_adamw_requant_step_mx(c.dev["p"], c.dev["g"], c.dev["m"], c.dev["v"], c.w_fp8, mx,
                                        int(s["blk_begin"]), int(s["blk_count_real"]), hp,
                                        desc=c.desc_dev, dev_status=c.status)
    torch.cuda.synchronize()
    assert c.status.item() == 0
    p, g, m, v = (c.host[k].copy() for k in "pgmv")
    q = np.zeros(c.cap * BLK, np.uint8)
    sc = np.zeros(c.cap * 512, np.uint8)
    oracle.adamw_requant_step_mx(p, g, m, v, q, sc, 0, int(c.summary["total_blocks"]),
                                 oracle.Hparams.make(step=6),
                                 desc=c.oracle_tables(oracle)[1])
    for k, want in (("p", p), ("m", m), ("v", v)):
        assert np.array_equal(c.dev[k].cpu().numpy().view(np.uint32), want.view(np.uint32)), k
    assert np.array_equal(c.w_fp8.cpu().numpy(), q)
    data = np.repeat(c.blocks["param"] >= 0, 512)
    assert np.array_equal(mx.cpu().numpy()[data], sc[data])


@pytest.mark.parametrize("step", [1, 50])
def test_mxfp8_extreme_magnitudes(oracle, step):
    """The MXFP8 step on state and grads spread over [1e-42, 1e38] (zeros mixed
    in): groups whose amax is subnormal, near FLT_MAX or zero; bit for bit."""
    c = Case([(1, 256, 384)], dp=1, seed=23)
    rng = np.random.default_rng(step)
    for k in "pgmv":
        n = c.host[k].size
        x = (10.0 ** rng.uniform(-42, 38, n) * rng.choice([-1.0, 1.0], n)).astype(np.float32)
        x[rng.random(n) < 0.02] = 0.0
        c.host[k][:] = np.abs(x) if k == "v" else x
        c.dev[k].copy_(torch.from_numpy(c.host[k]))
    hp = fp8z.hparams(step=step)
    mx = torch.zeros(c.cap * 512, dtype=torch.uint8, device="cuda")
    fp8z.fp8z_adamw_requant_step_mx(c.dev["p"], c.dev["g"], c.dev["m"], c.dev["v"], c.w_fp8, mx, 0, c.cap, hp,
                                    desc=c.desc_dev, dev_status=c.status)
    torch.cuda.synchronize()
    assert c.status.item() == 0
    p, g, m, v = (c.host[k].copy() for k in "pgmv")
    q = np.zeros(c.cap * BLK, np.uint8)
    sc = np.zeros(c.cap * 512, np.uint8)
    oracle.adamw_requant_step_mx(p, g, m, v, q, sc, 0, c.cap, oracle.Hparams.make(step=step),
                                 desc=c.oracle_tables(oracle)[1])
    for k, want in (("p", p), ("m", m), ("v", v)):
        a = c.dev[k].cpu().numpy()
        assert np.all((a.view(np.uint32) == want.view(np.uint32)) | (np.isnan(a) & np.isnan(want))), k
    qa = c.w_fp8.cpu().numpy()
    assert np.all((qa == q) | (((qa & 0x7F) == 0x7F) & ((q & 0x7F) == 0x7F)))
    assert np.array_equal(mx.cpu().numpy(), sc)


@pytest.mark.parametrize("seed", range(4))
def test_mxfp8_hyperparameters(oracle, seed):
    """The MXFP8 step under random hyper-parameters (the AdamW fields and both
    decay modes) on a ragged two-shard layout: bit for bit."""
    rng = np.random.default_rng(900 + seed)
    kw = _random_hparams(rng)
    c = Case([(1, 200, 300), (2, 130, 129)], dp=2, seed=seed)
    hp = fp8z.hparams(**kw)
    mx = torch.zeros(c.cap * 512, dtype=torch.uint8, device="cuda")
    for s in c.shards:
        fp8z.fp8z_adamw_requant_step_mx(c.dev["p"], c.dev["g"], c.dev["m"], c.dev["v"], c.w_fp8, mx,
                                        int(s["blk_begin"]), int(s["blk_count_real"]), hp,
                                        desc=c.desc_dev, dev_status=c.status)
    torch.cuda.synchronize()
    assert c.status.item() == 0
    p, g, m, v = (c.host[k].copy() for k in "pgmv")
    q = np.zeros(c.cap * BLK, np.uint8)
    sc = np.zeros(c.cap * 512, np.uint8)
    oracle.adamw_requant_step_mx(p, g, m, v, q, sc, 0, int(c.summary["total_blocks"]),
                                 oracle.Hparams.make(**kw),
                                 desc=c.oracle_tables(oracle)[1])
    for k, want in (("p", p), ("m", m), ("v", v)):
        assert np.array_equal(c.dev[k].cpu().numpy().view(np.uint32), want.view(np.uint32)), k
    assert np.array_equal(c.w_fp8.cpu().numpy(), q)
    data = np.repeat(c.blocks["param"] >= 0, 512)
    assert np.array_equal(mx.cpu().numpy()[data], sc[data])
