"""GPU 1x128 row-wise quantizer and scaling-aware transpose ("FP8-Flow-MoE"
§3.1) against the oracle, bit for bit: codes and scales, power-of-two and
amax/448 scales, zero tiles, outliers, rows whose scale forces underflow."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from blockwise_fp8_zero_gb300 import fp8z  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from blockwise_fp8_zero_gb300 import build
    build.build()
    fp8z.lib()


def _act(R, C, seed):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(R, C, generator=g)
    hit = torch.rand(R, C, generator=g) < 1e-3
    x = torch.where(hit, x * 60, x)
    x[:, :128] *= 1e-3
    if R > 7:
        x[7] *= 1e4                       # a row whose scale dwarfs the others: underflow
    if R > 3 and C > 256:
        x[3, 128:256] = 0.0               # a tile of zeros
    return x


def _gpu_quantize(x, pow2):
    R, C = x.shape
    q = torch.empty(R, C, dtype=torch.uint8, device="cuda")
    s = torch.empty(R, C // 128, device="cuda")
    fp8z.fp8z_quantize_rowwise(x.cuda(), pow2, q, s)
    return q, s


@pytest.mark.parametrize("shape", [(1, 128), (7, 384), (256, 512), (1000, 1280), (4096, 7168)])
@pytest.mark.parametrize("pow2", [True, False])
def test_quantize_rowwise(oracle, shape, pow2):
    x = _act(*shape, seed=shape[0])
    q, s = _gpu_quantize(x, pow2)
    torch.cuda.synchronize()
    qo, so = oracle.quantize_rowwise(x.numpy(), pow2=pow2)
    assert np.array_equal(s.cpu().numpy().view(np.uint32), so.view(np.uint32))
    assert np.array_equal(q.cpu().numpy(), qo)


@pytest.mark.parametrize("shape", [(128, 128), (256, 384), (1024, 1280), (4096, 7168)])
@pytest.mark.parametrize("pow2", [True, False])
def test_transpose_rowwise(oracle, shape, pow2):
    x = _act(*shape, seed=shape[1])
    # the oracle's row-wise codes and scales go to both sides
    qo, so = oracle.quantize_rowwise(x.numpy(), pow2=pow2)
    R, C = shape
    qt = torch.empty(C, R, dtype=torch.uint8, device="cuda")
    st = torch.empty(C, R // 128, device="cuda")
    fp8z.fp8z_transpose_rowwise(torch.from_numpy(qo).cuda(), torch.from_numpy(so).cuda(), qt, st)
    torch.cuda.synchronize()
    qto, sto = oracle.transpose_rowwise(qo, so)
    assert np.array_equal(st.cpu().numpy().view(np.uint32), sto.view(np.uint32))
    assert np.array_equal(qt.cpu().numpy(), qto)


def test_rowwise_argument_errors():
    x = torch.zeros(4, 100, device="cuda")
    with pytest.raises(fp8z.Fp8zError):
        fp8z.fp8z_quantize_rowwise(x, True, torch.empty(400, dtype=torch.uint8, device="cuda"),
                                   torch.empty(4, device="cuda"))
    q = torch.zeros(100, 128, dtype=torch.uint8, device="cuda")
    with pytest.raises(fp8z.Fp8zError):
        fp8z.fp8z_transpose_rowwise(q, torch.ones(100, 1, device="cuda"),
                                    torch.empty(128, 100, dtype=torch.uint8, device="cuda"),
                                    torch.empty(128, 1, device="cuda"))


@pytest.mark.parametrize("pow2", [True, False])
def test_rowwise_extreme_magnitudes(oracle, pow2):
    """Activations log-uniform over [1e-42, 1e38] with random signs and whole
    zero tiles: tiles whose amax is subnormal or near FLT_MAX, scales at both
    clamps; quantizer and scaling-aware transpose bit for bit."""
    rng = np.random.default_rng(int(pow2))
    R, C = 512, 640
    x = (10.0 ** rng.uniform(-42, 38, (R, C)) * rng.choice([-1.0, 1.0], (R, C))).astype(np.float32)
    x[rng.random((R, C)) < 0.02] = 0.0
    x[5, 128:256] = 0.0
    x[9] *= 1e-30                                  # a row of subnormal-range values
    if pow2:
        x[11, 200] = np.inf                        # an infinite tile amax takes the clamp
        x[12, 3] = -np.inf
    q, s = _gpu_quantize(torch.from_numpy(x), pow2)
    qt = torch.empty(C, R, dtype=torch.uint8, device="cuda")
    st = torch.empty(C, R // 128, device="cuda")
    fp8z.fp8z_transpose_rowwise(q, s, qt, st)
    torch.cuda.synchronize()
    qo, so = oracle.quantize_rowwise(x, pow2=pow2)
    assert np.array_equal(s.cpu().numpy().view(np.uint32), so.view(np.uint32))
    assert np.array_equal(q.cpu().numpy(), qo)
    qto, sto = oracle.transpose_rowwise(qo, so)
    assert np.array_equal(st.cpu().numpy().view(np.uint32), sto.view(np.uint32))
    assert np.array_equal(qt.cpu().numpy(), qto)
