"""Full-size workloads on the GPU, checked against the oracle on sampled
blocks (blocks are independent, so a block computed alone by the oracle is
the exact expected value): every ragged edge block (14,635 in the 500-matrix
workload), the first and last block of every shard, and a seeded random
sample of 1500.  Same bit-exact bar as the small
cases.  The 6e9-element workload runs in the launch configuration the
benchmark times (one launch over all blocks, column-major copy on)."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from blockwise_fp8_zero_gb300 import fp8z, workloads  # noqa: E402

from _gpu_util import assert_bitexact, oracle_blocks  # noqa: E402

pytestmark = pytest.mark.gpu
BLK = fp8z.BLOCK_ELEMS
CHUNK = 2048


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from blockwise_fp8_zero_gb300 import build
    build.build()
    fp8z.lib()
    yield
    torch.cuda.empty_cache()


def _sample(blocks, shards, n_random=1500, seed=0):
    data = np.nonzero(blocks["param"] >= 0)[0]
    rng = np.random.default_rng(seed)
    pick = set(rng.choice(data, size=min(n_random, data.size), replace=False).tolist())
    ragged = np.nonzero((blocks["param"] >= 0) & ((blocks["valid_rows"] < 128) | (blocks["valid_cols"] < 128)))[0]
    pick |= set(ragged.tolist())
    for s in shards:
        if s["blk_count_real"] > 0:
            pick.add(int(s["blk_begin"]))
            pick.add(int(s["blk_begin"] + s["blk_count_real"] - 1))
    return np.array(sorted(pick), dtype=np.int64)


def _gather(t, idx, width):
    it = torch.from_numpy(idx).to(t.device)
    return t.view(-1, width)[it].cpu().numpy().reshape(-1)


def run_sampled(oracle, w, one_launch=False):
    params, shards, blocks, summ = fp8z.fp8z_plan_shards(w.shapes, w.dp, w.split)
    cap = int(summ["capacity_blocks"])
    need = cap * BLK * (16 + 1) + (w.real_elems if w.transposed else 0)
    free, _ = torch.cuda.mem_get_info()
    if need > free - (4 << 30):
        pytest.skip(f"needs {need / 1e9:.0f} GB, {free / 1e9:.0f} GB free")
    dev = torch.device("cuda")
    state = workloads.make_state(w, blocks, dev, seed=0)
    q = torch.zeros(cap * BLK, dtype=torch.uint8, device=dev)
    inv = torch.zeros(cap, dtype=torch.float32, device=dev)
    desc = fp8z.table_to_device(blocks, dev)
    pdev = fp8z.table_to_device(params, dev)
    t_scales = int(sum(int(p["e"]) * int(p["hb"]) * int(p["wb"]) for p in params))
    wt = torch.zeros(w.real_elems, dtype=torch.uint8, device=dev) if w.transposed else None
    it = torch.zeros(t_scales, dtype=torch.float32, device=dev) if w.transposed else None
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    idx = _sample(blocks, shards)
    pre = {k: _gather(state[k], idx, BLK) for k in "pgmv"}
    hp = fp8z.hparams(**w.hp)
    ranges = [(0, cap)] if one_launch else [(int(s["blk_begin"]), int(s["blk_count_real"])) for s in shards]
    for b0, nb in ranges:
        fp8z.fp8z_adamw_requant_step(state["p"], state["g"], state["m"], state["v"], q, inv, b0, nb, hp,
                                     desc=desc, params=pdev if w.transposed else None,
                                     nparams=len(params) if w.transposed else 0,
                                     w_fp8_t=wt, inv_scale_t=it, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0, fp8z.fp8z_status_string(st.item())
    # checked in chunks of blocks, so the host holds the inputs of the sample
    # (gathered before the step) and one chunk of outputs at a time
    o_blocks = oracle.plan_shards(w.shapes, w.dp, w.split)[2]      # the oracle's own plan
    for c0 in range(0, idx.size, CHUNK):
        ii = idx[c0:c0 + CHUNK]
        got = {k: _gather(state[k], ii, BLK) for k in "pmv"}
        got["q"] = _gather(q, ii, BLK)
        got["inv"] = inv[torch.from_numpy(ii).to(dev)].cpu().numpy()
        d = np.ascontiguousarray(o_blocks[ii])
        sl = slice(c0 * BLK, (c0 + ii.size) * BLK)
        pc = {k: pre[k][sl] for k in "pgmv"}
        qc, invc = oracle_blocks(oracle, hp, pc["p"], pc["g"], pc["m"], pc["v"], d)
        assert_bitexact(got, dict(p=pc["p"], m=pc["m"], v=pc["v"], q=qc, inv=invc))
        if c0 == 0:
            qo, invo = qc, invc
        del got
    if w.transposed:
        # the column-major copy of each sampled block is its oracle tile, transposed
        for j, b in enumerate(idx[:400]):
            bd = blocks[b]
            pe = params[int(bd["param"])]
            H, W = int(pe["rows"]), int(pe["cols"])
            vr, vc = int(bd["valid_rows"]), int(bd["valid_cols"])
            base = int(pe["t_offset"]) + int(bd["e"]) * W * H
            mat = wt[base:base + W * H].view(W, H)
            r0, c0 = int(bd["brow"]) * 128, int(bd["bcol"]) * 128
            tile = mat[c0:c0 + vc, r0:r0 + vr].cpu().numpy()
            want = qo[j * BLK:(j + 1) * BLK].reshape(128, 128)[:vr, :vc].T
            assert np.array_equal(tile, want), int(b)
            s_idx = int(pe["t_scale_offset"]) + int(bd["e"]) * int(pe["wb"]) * int(pe["hb"]) \
                + int(bd["bcol"]) * int(pe["hb"]) + int(bd["brow"])
            assert it[s_idx].item() == invo[j]
    del state, q, inv, wt, it
    torch.cuda.empty_cache()
    return summ


def test_moe64_full(oracle):
    """64-expert bank (2.8e9 elements), Student-t grads, 16 shard launches."""
    run_sampled(oracle, workloads.get("moe64"))


@pytest.mark.parametrize("split", [0, 1])
def test_mixed500_full(oracle, split):
    """500 mixed ragged matrices at 16 shards, block-wise and param-wise."""
    summ = run_sampled(oracle, workloads.get("mixed500", split))
    assert summ["total_blocks"] > 400000


def test_flat6e9_full_bench_launch(oracle):
    """117 x 7168^2 with the column-major copy, one launch over all blocks."""
    run_sampled(oracle, workloads.get("flat6e9"), one_launch=True)
