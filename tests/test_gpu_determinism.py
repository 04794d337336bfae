"""Run-to-run identity of the three step variants: the same inputs stepped five
times give the same bytes every time.  A race between the consumers' reads of
a ring slot and its refill, or between the column-major tile's staging and read
out, would show here as differences that come and go (the parity tests compare
one run with the oracle).  Two 2048x7168 expert matrices and a ragged
7168x576 weight: about 40 blocks per CTA, so every ring slot is reused many
times."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from blockwise_fp8_zero_gb300 import fp8z, workloads  # noqa: E402

pytestmark = pytest.mark.gpu
BLK = fp8z.BLOCK_ELEMS
SHAPES = [(2, 2048, 7168), (1, 7168, 576), (3, 1024, 2048)]
RUNS = 5


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from blockwise_fp8_zero_gb300 import build
    build.build()
    fp8z.lib()


def _inputs(params, blocks, cap):
    dists = dict(p=workloads.Dist("normal", 0.02), g=workloads.Dist("normal", 1e-3),
                 m=workloads.Dist("normal", 2e-4), v=workloads.Dist("uniform", 1e-7, 4e-7))
    out = {}
    for k in "pgmv":
        t = torch.empty(cap * BLK)
        workloads.fill(t, k, dists[k], 11, blocks["valid_rows"], blocks["valid_cols"])
        out[k] = t.cuda()
    return out


@pytest.mark.parametrize("variant", ["block_scaled_with_copy", "mxfp8", "rowmajor_with_copy"])
def test_runs_are_bit_identical(variant):
    params, shards, blocks, summ = fp8z.fp8z_plan_shards(SHAPES, 1, 0)
    cap = int(summ["capacity_blocks"])
    base = _inputs(params, blocks, cap)
    desc = fp8z.table_to_device(blocks)
    pdev = fp8z.table_to_device(params)
    t_bytes = int(sum(e * r * c for e, r, c in SHAPES))
    t_scales = int(sum(int(p["e"]) * int(p["hb"]) * int(p["wb"]) for p in params))
    hp = fp8z.hparams(step=9)
    grads_rm = None
    if variant == "rowmajor_with_copy":
        # the same grads in each param's row-major layout
        grads_rm = []
        for i, (e, r, c) in enumerate(SHAPES):
            g = torch.empty(e * r * c, device="cuda")
            fp8z.fp8z_unfold(base["g"], params[i], g)
            grads_rm.append(g)
        maps = fp8z.fp8z_encode_grad_maps(grads_rm, params)
    first = None
    for rep in range(RUNS):
        s = {k: v.clone() for k, v in base.items()}
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        inv = torch.zeros(cap, device="cuda")
        if variant == "block_scaled_with_copy":
            q = torch.zeros(cap * BLK, dtype=torch.uint8, device="cuda")
            wt = torch.zeros(t_bytes, dtype=torch.uint8, device="cuda")
            it = torch.zeros(t_scales, device="cuda")
            fp8z.fp8z_adamw_requant_step(s["p"], s["g"], s["m"], s["v"], q, inv, 0, cap, hp, desc=desc,
                                         params=pdev, nparams=len(params), w_fp8_t=wt, inv_scale_t=it,
                                         dev_status=st)
            outs = [q, inv, wt, it]
        elif variant == "mxfp8":
            q = torch.zeros(cap * BLK, dtype=torch.uint8, device="cuda")
            mx = torch.zeros(cap * 512, dtype=torch.uint8, device="cuda")
            fp8z.fp8z_adamw_requant_step_mx(s["p"], s["g"], s["m"], s["v"], q, mx, 0, cap, hp, desc=desc,
                                            dev_status=st)
            outs = [q, mx]
        else:
            w_row = torch.zeros(t_bytes, dtype=torch.uint8, device="cuda")
            wt = torch.zeros(t_bytes, dtype=torch.uint8, device="cuda")
            it = torch.zeros(t_scales, device="cuda")
            fp8z.fp8z_adamw_requant_step_rowmajor(s["p"], s["m"], s["v"], maps, w_row, inv, 0, cap, hp, desc,
                                                  pdev, len(params), w_fp8_t=wt, inv_scale_t=it, dev_status=st)
            outs = [w_row, inv, wt, it]
        torch.cuda.synchronize()
        assert st.item() == 0, fp8z.fp8z_status_string(st.item())
        got = [x.view(torch.uint8).cpu().numpy() for x in [s["p"], s["m"], s["v"]] + outs]
        if first is None:
            first = got
        else:
            for a, b in zip(first, got):
                assert np.array_equal(a, b), f"run {rep} differs from run 0 in {np.count_nonzero(a != b)} bytes"
