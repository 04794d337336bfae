"""The library keeps no shared mutable state between calls: the planner gives
the same tables when many host threads call it at once (CPU), and shard steps
launched at the same time from several host threads, each on its own stream,
give the oracle's results bit for bit (GPU).  The only process-wide state is
the per-device caches of launch attributes, filled with atomics."""
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest

from blockwise_fp8_zero_gb300 import fp8z, workloads


@pytest.fixture(scope="module")
def L():
    from blockwise_fp8_zero_gb300 import build
    build.build()
    return fp8z.lib()


def test_planner_from_many_threads(L):
    w = workloads.get("mixed500", 1)
    want = fp8z.fp8z_plan_shards(w.shapes, w.dp, 1)

    def plan(i):
        split = i % 2
        return split, fp8z.fp8z_plan_shards(w.shapes, w.dp, split)

    want0 = fp8z.fp8z_plan_shards(w.shapes, w.dp, 0)
    with ThreadPoolExecutor(8) as ex:
        for split, got in ex.map(plan, range(32)):
            ref = want if split == 1 else want0
            for x, y in zip(got, ref):
                assert np.array_equal(np.atleast_1d(x), np.atleast_1d(y))


@pytest.mark.gpu
@pytest.mark.parametrize("transposed", [False, True])
def test_shards_on_concurrent_streams(L, oracle, transposed):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from _gpu_util import Case, assert_bitexact

    # 8 block-wise shards that cut expert matrices and a ragged param
    c = Case([(3, 640, 1152), (1, 7168, 576), (2, 200, 300)], dp=8, seed=17, transposed=transposed)
    hp = fp8z.hparams(step=11)
    streams = [torch.cuda.Stream() for _ in c.shards]
    torch.cuda.synchronize()

    def launch(i):
        s = c.shards[i]
        b0, nb = int(s["blk_begin"]), int(s["blk_count_real"])
        c.processed[b0:b0 + nb] = True
        return fp8z.fp8z_adamw_requant_step(
            c.dev["p"], c.dev["g"], c.dev["m"], c.dev["v"], c.w_fp8, c.inv, b0, nb, hp,
            desc=c.desc_dev, params=c.params_dev if transposed else None,
            nparams=len(c.params) if transposed else 0, w_fp8_t=c.wt, inv_scale_t=c.it,
            dev_status=c.status, stream=streams[i])

    with ThreadPoolExecutor(len(streams)) as ex:
        list(ex.map(launch, range(len(streams))))
    torch.cuda.synchronize()
    assert int(c.status.item()) == 0, fp8z.fp8z_status_string(int(c.status.item()))
    assert_bitexact(c.results(), c.oracle(oracle, hp), c.processed)
