"""The fused row-major step (fold-on-read of the grad through TMA tensor maps,
unfold-on-write of the E4M3 weights) against the oracle: the oracle folds the
row-major grad, runs its step on the folded state, and unfolds its codes.
Same bit-exact bar as the folded step."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from blockwise_fp8_zero_gb300 import fp8z, workloads  # noqa: E402

from _gpu_util import oracle_blocks  # noqa: E402

pytestmark = pytest.mark.gpu
BLK = fp8z.BLOCK_ELEMS


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from blockwise_fp8_zero_gb300 import build
    build.build()
    fp8z.lib()


def run_case(oracle, shapes, dp, split=0, transposed=False, step=5, seed=0, bad_desc=False, hp_kw=None):
    params, shards, blocks, summ = fp8z.fp8z_plan_shards(shapes, dp, split)
    cap = int(summ["capacity_blocks"])
    dev = torch.device("cuda")
    state = {}
    for k, d in zip("pmv", (workloads.Dist("normal", 0.02), workloads.Dist("normal", 2e-4),
                            workloads.Dist("uniform", 1e-7, 4e-7))):
        t = torch.empty(cap * BLK)
        workloads.fill(t, k, d, seed, blocks["valid_rows"], blocks["valid_cols"])
        state[k] = t
    gen = torch.Generator().manual_seed(seed + 1)
    grads = [torch.randn(s, generator=gen) * 1e-3 for s in shapes]
    # host copies for the oracle, grad folded by the oracle's own fold
    host = {k: state[k].numpy().copy() for k in "pmv"}
    g_fold = np.zeros(cap * BLK, np.float32)
    for i, gt in enumerate(grads):
        o = int(params[i]["blk_offset"]) * BLK
        f = oracle.fold(gt.numpy()).ravel()
        g_fold[o:o + f.size] = f
    d = {k: state[k].to(dev) for k in "pmv"}
    gd = [gt.to(dev) for gt in grads]
    maps = fp8z.fp8z_encode_grad_maps(gd, params)
    t_bytes = int(sum(e * r * c for e, r, c in shapes))
    t_scales = int(sum(int(p["e"]) * int(p["hb"]) * int(p["wb"]) for p in params))
    w_row = torch.zeros(t_bytes, dtype=torch.uint8, device=dev)
    inv = torch.zeros(cap, device=dev)
    wt = torch.zeros(t_bytes, dtype=torch.uint8, device=dev) if transposed else None
    it = torch.zeros(t_scales, device=dev) if transposed else None
    bl = blocks.copy()
    if bad_desc:
        bl["param"][0] = len(shapes) + 3
    desc = fp8z.table_to_device(bl)
    pdev = fp8z.table_to_device(params)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    hp = fp8z.hparams(**(hp_kw or {"step": step}))
    for s in shards:
        fp8z.fp8z_adamw_requant_step_rowmajor(d["p"], d["m"], d["v"], maps, w_row, inv,
                                              int(s["blk_begin"]), int(s["blk_count_real"]), hp,
                                              desc, pdev, len(params), w_fp8_t=wt, inv_scale_t=it,
                                              dev_status=st)
    torch.cuda.synchronize()
    if bad_desc:
        return st.item()
    assert st.item() == 0, fp8z.fp8z_status_string(st.item())
    wt_o = np.zeros(t_bytes, np.uint8) if transposed else None
    it_o = np.zeros(t_scales, np.float32) if transposed else None
    o_params, _, o_blocks, _ = oracle.plan_shards(shapes, dp, split)    # the oracle's own plan
    q_o, inv_o = oracle_blocks(oracle, hp, host["p"], g_fold, host["m"], host["v"], o_blocks,
                               o_params if transposed else None, wt_o, it_o)
    for k in "pmv":
        assert np.array_equal(d[k].cpu().numpy().view(np.uint32), host[k].view(np.uint32)), k
    data = blocks["param"] >= 0
    assert np.array_equal(inv.cpu().numpy()[data], inv_o[data])
    want_row = np.zeros(t_bytes, np.uint8)
    for i, (E, H, W) in enumerate(shapes):
        pe = params[i]
        o = int(pe["blk_offset"])
        nb = E * int(pe["hb"]) * int(pe["wb"])
        qq = oracle.unfold(q_o[o * BLK:(o + nb) * BLK].astype(np.float32).reshape(nb, 128, 128), E, H, W)
        t0 = int(pe["t_offset"])
        want_row[t0:t0 + E * H * W] = qq.astype(np.uint8).ravel()
    assert np.array_equal(w_row.cpu().numpy(), want_row)
    if transposed:
        assert np.array_equal(wt.cpu().numpy(), wt_o)
        assert np.array_equal(it.cpu().numpy(), it_o)


@pytest.mark.parametrize("shapes", [[(1, 256, 384)], [(2, 300, 260)], [(1, 129, 4)], [(3, 7, 1000)],
                                    [(1, 7168, 576)], [(1, 300, 200), (2, 128, 640), (1, 64, 64)]])
@pytest.mark.parametrize("transposed", [False, True])
def test_rowmajor_step(oracle, shapes, transposed):
    run_case(oracle, shapes, dp=1, transposed=transposed, seed=len(shapes))


@pytest.mark.parametrize("shapes", [[(1, 130, 65536)], [(1, 65541, 136)], [(512, 16, 16)]])
def test_rowmajor_step_extreme_shapes(oracle, shapes):
    # a 256 KB grad row pitch, 513 block rows, 512 one-block experts
    run_case(oracle, shapes, dp=1, transposed=True, seed=11)


@pytest.mark.parametrize("seed", range(6))
def test_rowmajor_step_hyperparameters(oracle, seed):
    # random hyper-parameters (every field the step reads) on a ragged layout
    rng = np.random.default_rng(500 + seed)
    hp_kw = dict(lr=float(10 ** rng.uniform(-7, -1)), beta1=float(rng.uniform(0, 0.99)),
                 beta2=float(rng.uniform(0, 0.9999)), eps=float(10 ** rng.uniform(-12, -2)),
                 weight_decay=float(rng.uniform(0, 1)), step=int(10 ** rng.uniform(0, 6)),
                 scale_mode=int(rng.integers(0, 2)), decay_mode=int(rng.integers(0, 2)),
                 fp8_max=float(rng.choice([448.0, 1.0 + rng.uniform(0, 447)])),
                 min_scale=float(rng.choice([0.0, 1e-6, rng.uniform(0, 1e3)])))
    run_case(oracle, [(1, 300, 200), (2, 128, 260)], dp=2, transposed=True, seed=seed, hp_kw=hp_kw)


@pytest.mark.parametrize("split", [0, 1])
def test_rowmajor_step_sharded(oracle, split):
    run_case(oracle, [(1, 640, 384), (2, 200, 300), (1, 128, 1000), (1, 1000, 128)], dp=3,
             split=split, transposed=True, step=9)


def test_rowmajor_bad_descriptor_reported(oracle):
    assert run_case(oracle, [(1, 256, 256)], dp=1, bad_desc=True) == fp8z.FP8Z_EINVAL


# grads whose row pitch is not a multiple of 16 bytes (cols % 4 != 0) are read
# with plain loads; mixed with tensor-map params in one launch
UNALIGNED = [(1, 300, 1), (1, 256, 384), (2, 129, 7), (1, 200, 130), (1, 130, 1001), (1, 64, 64)]


@pytest.mark.parametrize("transposed", [False, True])
@pytest.mark.parametrize("dp,split", [(1, 0), (3, 0), (4, 1)])
def test_rowmajor_step_unaligned_rows(oracle, transposed, dp, split):
    run_case(oracle, UNALIGNED, dp=dp, split=split, transposed=transposed, seed=dp + 7)


def test_rowmajor_step_unaligned_rows_pow2_post_decay(oracle):
    run_case(oracle, [(3, 7, 1001), (1, 1000, 129)], dp=2, transposed=True, seed=3,
             hp_kw=dict(step=20, scale_mode=1, decay_mode=1))


def test_encode_grad_maps_alignment_rules():
    # a tensor-map grad must start on 16 bytes; a plain-load grad on 4
    params, _, _, _ = fp8z.fp8z_plan_shards([(1, 128, 132)], 1, 0, with_blocks=False)
    g = torch.zeros(128 * 132 + 1, device="cuda")
    with pytest.raises(fp8z.Fp8zError):
        fp8z.fp8z_encode_grad_maps([g[1:]], params)
    params, _, _, _ = fp8z.fp8z_plan_shards([(1, 128, 130)], 1, 0, with_blocks=False)
    fp8z.fp8z_encode_grad_maps([g[1:1 + 128 * 130]], params)


@pytest.mark.parametrize("enc_cols,run_cols", [(130, 132), (132, 130)])
def test_rowmajor_slot_of_another_shape_is_reported(enc_cols, run_cols):
    """Slots encoded for one shape used with a param table of another: a record
    where a tensor map belongs, or the reverse, gives grad 0 and FP8Z_EINVAL
    (the kernel reads neither through a slot that does not match)."""
    dev = torch.device("cuda")
    p_enc, _, _, _ = fp8z.fp8z_plan_shards([(1, 256, enc_cols)], 1, 0, with_blocks=False)
    g = torch.randn(256 * max(enc_cols, run_cols), device=dev)
    maps = fp8z.fp8z_encode_grad_maps([g], p_enc)
    params, shards, blocks, summ = fp8z.fp8z_plan_shards([(1, 256, run_cols)], 1, 0)
    cap = int(summ["capacity_blocks"])
    p, m, v = (torch.zeros(cap * BLK, device=dev) for _ in range(3))
    w_row = torch.zeros(256 * run_cols, dtype=torch.uint8, device=dev)
    inv = torch.zeros(cap, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    fp8z.fp8z_adamw_requant_step_rowmajor(p, m, v, maps, w_row, inv, 0, cap, fp8z.hparams(),
                                          fp8z.table_to_device(blocks), fp8z.table_to_device(params), 1,
                                          dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == fp8z.FP8Z_EINVAL
    assert int(m.count_nonzero()) == 0          # grad 0 and m 0: m stays 0
