"""The kernels' own bounded waits, made to run out.

Every barrier wait of the step (block-scaled with the column-major copy,
row-major, MXFP8), of dequant, of the TMA transpose and of the TMA fold /
unfold gives up after a limit, reports FP8Z_ETIMEOUT in *dev_status, lets the
copies it still has in flight land, and returns.  Here the limit is cut to
1 ns, so that every real wait of a launch of about 2,000 blocks that finds its
barrier still incomplete gives up (a few hundred nanoseconds proved too long
to be sure of it: a block the previous kernel left in L2 can land sooner).
No barrier is left unarmed and nothing faults: the copies all land, only the
waiting stops early.  Afterwards the limit is restored
and a normal step on the same context must still match the oracle bit for
bit.  The pages print no failure handling; this covers the library's own
watchdog."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from blockwise_fp8_zero_gb300 import fp8z, workloads  # noqa: E402

from _gpu_util import Case, assert_bitexact  # noqa: E402

pytestmark = pytest.mark.gpu
BLK = fp8z.BLOCK_ELEMS
SHORT_NS = 1             # every wait that finds its barrier incomplete gives up
TRIES = 5


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from blockwise_fp8_zero_gb300 import build
    build.build()
    fp8z.lib()


@pytest.fixture
def short_waits():
    fp8z.fp8z_set_wait_limit_ns(SHORT_NS)
    try:
        yield
    finally:
        fp8z.fp8z_set_wait_limit_ns(0)


def times_out(launch):
    """Run launch(status) up to TRIES times with a fresh status word; True once
    a launch reports FP8Z_ETIMEOUT.  Any other non-zero status fails."""
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    for _ in range(TRIES):
        st.zero_()
        launch(st)
        torch.cuda.synchronize()
        code = int(st.item())
        if code == fp8z.FP8Z_ETIMEOUT:
            return True
        assert code == 0, fp8z.fp8z_status_string(code)
    return False


SHAPE = (1, 40 * 128, 50 * 128)          # 2,000 blocks, one param


@pytest.fixture(scope="module")
def case():
    return Case([SHAPE], dp=1, seed=3, transposed=True, gen_device="cuda")


def test_step_with_copy_times_out(case, short_waits):
    hp = fp8z.hparams(step=4)
    c = case

    def launch(st):
        fp8z.fp8z_adamw_requant_step(c.dev["p"], c.dev["g"], c.dev["m"], c.dev["v"], c.w_fp8, c.inv, 0,
                                     c.cap, hp, desc=c.desc_dev, params=c.params_dev, nparams=1,
                                     w_fp8_t=c.wt, inv_scale_t=c.it, dev_status=st)
    assert times_out(launch)


def test_mx_step_times_out(case, short_waits):
    hp = fp8z.hparams(step=4)
    c = case
    mx = torch.zeros(c.cap * 512, dtype=torch.uint8, device="cuda")

    def launch(st):
        fp8z.fp8z_adamw_requant_step_mx(c.dev["p"], c.dev["g"], c.dev["m"], c.dev["v"], c.w_fp8, mx, 0,
                                        c.cap, hp, desc=c.desc_dev, dev_status=st)
    assert times_out(launch)


def test_rowmajor_step_times_out(case, short_waits):
    hp = fp8z.hparams(step=4)
    c = case
    g = torch.randn(SHAPE, device="cuda") * 1e-3
    maps = fp8z.fp8z_encode_grad_maps([g], c.params)
    w_row = torch.zeros(c.t_bytes, dtype=torch.uint8, device="cuda")

    def launch(st):
        fp8z.fp8z_adamw_requant_step_rowmajor(c.dev["p"], c.dev["m"], c.dev["v"], maps, w_row, c.inv, 0,
                                              c.cap, hp, c.desc_dev, c.params_dev, 1, w_fp8_t=c.wt,
                                              inv_scale_t=c.it, dev_status=st)
    assert times_out(launch)


def test_dequant_times_out(case, short_waits):
    c = case
    out = torch.empty(c.cap * BLK, device="cuda")
    assert times_out(lambda st: fp8z.fp8z_dequant(c.w_fp8, c.inv, c.cap, out, dev_status=st))


def test_tma_transpose_times_out(case, short_waits):
    c = case
    pe = c.params[0]
    assert int(pe["rows"]) % 16 == 0           # the TMA kernel, not the one-CTA-per-block one
    out = torch.empty(c.t_bytes, dtype=torch.uint8, device="cuda")
    inv_t = torch.empty(c.cap, device="cuda")
    assert times_out(lambda st: fp8z.fp8z_transpose_fp8(c.w_fp8, c.inv, pe, out, inv_t, dev_status=st))


@pytest.mark.parametrize("dtype", [torch.float32, torch.uint8])
def test_tma_fold_unfold_times_out(case, short_waits, dtype):
    c = case
    pe = c.params[0]
    n = c.cap * BLK
    blocks = torch.zeros(n, dtype=dtype, device="cuda")
    rm = torch.zeros(n, dtype=dtype, device="cuda")
    assert times_out(lambda st: fp8z.fp8z_unfold(blocks, pe, rm, dev_status=st))
    assert times_out(lambda st: fp8z.fp8z_fold(rm, pe, blocks, dev_status=st))


def test_normal_step_after_timeouts_is_exact(oracle):
    """The limit back at its default, the context that saw every timeout above
    still runs a step that matches the oracle bit for bit."""
    assert fp8z.fp8z_get_wait_limit_ns() == 2_000_000_000
    c = Case([(1, 300, 700), (2, 256, 130)], dp=2, seed=8, transposed=True)
    hp = fp8z.hparams(step=6)
    c.step(hp)
    assert_bitexact(c.results(), c.oracle(oracle, hp), c.processed)
