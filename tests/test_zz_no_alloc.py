"""The row-major step for callers that cannot allocate device memory.

fp8z_adamw_requant_step_rowmajor_static keeps the grad tensor maps in an
array inside the library instead of the g_maps buffer that
fp8z_adamw_requant_step_rowmajor reads, so a caller that may not call
cudaMalloc at step time (code inside another framework's step that only owns
the tensors it was handed, or code that must not stall the device) can still
run the fused row-major step.  Here it is called through the C ABI twice in a
row, each time beside the allocating entry point on a copy of the same state,
and every output must be identical (the bar of the other parity tests: bit
for bit).  The second call uses new grad tensors, so the array's maps must be
replaced, not reused.  This file is collected last on purpose."""
import ctypes

import numpy as np
import pytest

from blockwise_fp8_zero_gb300 import fp8z, workloads

BLK = fp8z.BLOCK_ELEMS
SHAPES = [(1, 300, 260), (2, 200, 384), (1, 128, 1000)]
DP = 2


def test_refuses_more_params_than_the_array_holds():
    """More params than the library's array holds is refused before any device
    work (no pointer below is dereferenced)."""
    from blockwise_fp8_zero_gb300 import build
    build.build()
    L = fp8z.lib()
    n = 1025
    assert L.fp8z_adamw_requant_step_rowmajor_static(
        0x10000, 0x10000, 0x10000, 0x10000, 0x10000, 0x10000, 16, 0x10000, 4, 0, 1, 0x10000, 0x10000, n,
        None, 0, None, 0, ctypes.byref(fp8z.hparams()), None, None) == fp8z.FP8Z_ENOSPACE


@pytest.mark.gpu
def test_static_maps_step_matches_allocating_step_twice():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from blockwise_fp8_zero_gb300 import build
    build.build()
    fp8z.lib()
    dev = torch.device("cuda")
    params, shards, blocks, summ = fp8z.fp8z_plan_shards(SHAPES, DP, 0)
    cap = int(summ["capacity_blocks"])
    t_bytes = int(sum(e * r * c for e, r, c in SHAPES))
    t_scales = int(sum(int(p["e"]) * int(p["hb"]) * int(p["wb"]) for p in params))
    desc = fp8z.table_to_device(blocks, dev)
    pdev = fp8z.table_to_device(params, dev)

    state = {}
    for k, d in zip("pmv", (workloads.Dist("normal", 0.02), workloads.Dist("normal", 2e-4),
                            workloads.Dist("uniform", 1e-7, 4e-7))):
        t = torch.empty(cap * BLK)
        workloads.fill(t, k, d, 21, blocks["valid_rows"], blocks["valid_cols"])
        state[k] = t

    def outputs():
        return dict(w_row=torch.zeros(t_bytes, dtype=torch.uint8, device=dev),
                    inv=torch.zeros(cap, device=dev),
                    wt=torch.zeros(t_bytes, dtype=torch.uint8, device=dev),
                    it=torch.zeros(t_scales, device=dev),
                    st=torch.zeros(1, dtype=torch.int32, device=dev))

    ref = {k: state[k].to(dev) for k in "pmv"}          # the allocating entry point's state
    new = {k: state[k].to(dev) for k in "pmv"}          # the static entry point's state
    ref_out, new_out = outputs(), outputs()
    data = blocks["param"] >= 0

    for call, seed in enumerate((31, 47)):
        gen = torch.Generator().manual_seed(seed)
        grads = [(torch.randn(s, generator=gen) * 1e-3).to(dev) for s in SHAPES]   # fresh tensors
        hp = fp8z.hparams(step=7 + call)
        maps = fp8z.fp8z_encode_grad_maps(grads, params)
        for s in shards:
            b0, nb = int(s["blk_begin"]), int(s["blk_count_real"])
            fp8z.fp8z_adamw_requant_step_rowmajor(
                ref["p"], ref["m"], ref["v"], maps, ref_out["w_row"], ref_out["inv"], b0, nb, hp, desc, pdev,
                len(params), w_fp8_t=ref_out["wt"], inv_scale_t=ref_out["it"], dev_status=ref_out["st"])
            fp8z.fp8z_adamw_requant_step_rowmajor_static(
                new["p"], new["m"], new["v"], grads, params, new_out["w_row"], new_out["inv"], b0, nb, hp,
                desc, pdev, len(params), w_fp8_t=new_out["wt"], inv_scale_t=new_out["it"],
                dev_status=new_out["st"])
        torch.cuda.synchronize()
        assert int(ref_out["st"].item()) == 0 and int(new_out["st"].item()) == 0, call
        for k in "pmv":
            a, b = new[k].cpu().numpy(), ref[k].cpu().numpy()
            assert np.array_equal(a.view(np.uint32), b.view(np.uint32)), (call, k)
        assert torch.equal(new_out["w_row"], ref_out["w_row"]), call
        assert np.array_equal(new_out["inv"].cpu().numpy()[data].view(np.uint32),
                              ref_out["inv"].cpu().numpy()[data].view(np.uint32)), call
        assert torch.equal(new_out["wt"], ref_out["wt"]), call
        assert np.array_equal(new_out["it"].cpu().numpy().view(np.uint32),
                              ref_out["it"].cpu().numpy().view(np.uint32)), call
        # the step did run: the codes are not all zero
        assert int(new_out["w_row"].count_nonzero()) > t_bytes // 2, call
        del grads, maps


@pytest.mark.gpu
def test_static_maps_step_with_plain_load_grads():
    """Grads whose row pitch is not a multiple of 16 bytes are described by
    plain records instead of tensor maps; the library's array holds those
    too.  Mixed with tensor-map params, one call, against the allocating
    entry point."""
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from blockwise_fp8_zero_gb300 import build
    build.build()
    fp8z.lib()
    dev = torch.device("cuda")
    shapes = [(1, 300, 130), (1, 256, 384), (2, 129, 7)]
    params, shards, blocks, summ = fp8z.fp8z_plan_shards(shapes, 1, 0)
    cap = int(summ["capacity_blocks"])
    t_bytes = int(sum(e * r * c for e, r, c in shapes))
    desc = fp8z.table_to_device(blocks, dev)
    pdev = fp8z.table_to_device(params, dev)
    state = {}
    for k, d in zip("pmv", (workloads.Dist("normal", 0.02), workloads.Dist("normal", 2e-4),
                            workloads.Dist("uniform", 1e-7, 4e-7))):
        t = torch.empty(cap * BLK)
        workloads.fill(t, k, d, 5, blocks["valid_rows"], blocks["valid_cols"])
        state[k] = t
    gen = torch.Generator().manual_seed(9)
    grads = [(torch.randn(s, generator=gen) * 1e-3).to(dev) for s in shapes]
    hp = fp8z.hparams(step=3)
    runs = []
    for static in (False, True):
        st = {k: state[k].to(dev) for k in "pmv"}
        w_row = torch.zeros(t_bytes, dtype=torch.uint8, device=dev)
        inv = torch.zeros(cap, device=dev)
        status = torch.zeros(1, dtype=torch.int32, device=dev)
        if static:
            fp8z.fp8z_adamw_requant_step_rowmajor_static(st["p"], st["m"], st["v"], grads, params, w_row, inv, 0,
                                                        cap, hp, desc, pdev, len(params), dev_status=status)
        else:
            maps = fp8z.fp8z_encode_grad_maps(grads, params)
            fp8z.fp8z_adamw_requant_step_rowmajor(st["p"], st["m"], st["v"], maps, w_row, inv, 0, cap, hp, desc,
                                                  pdev, len(params), dev_status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        runs.append((st, w_row, inv))
    (a, wa, ia), (b, wb, ib) = runs
    for k in "pmv":
        assert np.array_equal(a[k].cpu().numpy().view(np.uint32), b[k].cpu().numpy().view(np.uint32)), k
    assert torch.equal(wa, wb)
    data = blocks["param"] >= 0
    assert np.array_equal(ia.cpu().numpy()[data].view(np.uint32), ib.cpu().numpy()[data].view(np.uint32))
    assert int(wb.count_nonzero()) > t_bytes // 2
