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


def _same_floats(a, b):
    """Bitwise equal, NaN equal to NaN (the E4M3 NaN codes decode to NaN)."""
    same = (a.view(np.uint32) == b.view(np.uint32)) | (np.isnan(a) & np.isnan(b))
    assert np.all(same), f"{int((~same).sum())} differ"


@pytest.mark.parametrize("shape", [(128, 128), (256, 384), (1000, 1280), (4096, 7168)])
def test_dequant_rowwise(oracle, shape):
    """Every code (NaN codes included) under power-of-two, amax/448-like,
    subnormal-producing and near-FLT_MAX scales, row-major and transposed,
    against the oracle's dequantize."""
    R, C = shape
    rng = np.random.default_rng(R + C)
    q = rng.integers(0, 256, (R, C), dtype=np.uint8)
    q[0, :256 if C >= 256 else C] = np.arange(min(C, 256), dtype=np.uint8)
    s = (10.0 ** rng.uniform(-30, 30, (R, C // 128))).astype(np.float32)
    s[::3] = np.exp2(rng.integers(-126, 120, s[::3].shape)).astype(np.float32)
    s[1, 0] = 1e-40                                  # subnormal products
    s[2, 0] = 3e38                                   # products overflow to infinity
    want = oracle.dequant_rowwise(q, s)
    qd, sd = torch.from_numpy(q).cuda(), torch.from_numpy(s).cuda()
    out = torch.empty(R, C, device="cuda")
    fp8z.fp8z_dequant_rowwise(qd, sd, out)
    torch.cuda.synchronize()
    _same_floats(out.cpu().numpy(), want)
    if R % 128 == 0:
        out_t = torch.empty(C, R, device="cuda")
        fp8z.fp8z_dequant_rowwise(qd, sd, out_t, transpose=True)
        torch.cuda.synchronize()
        _same_floats(out_t.cpu().numpy(), np.ascontiguousarray(want.T))


def test_naive_path_from_library_kernels(oracle):
    """The naive way to the column-wise layout, dequantize-transpose then
    quantize again, run from the library's kernels, equals the oracle's
    quantize of the oracle's dequantized transpose."""
    x = _act(512, 768, seed=4)
    for pow2 in (True, False):
        qo, so = oracle.quantize_rowwise(x.numpy(), pow2=pow2)
        xt = torch.empty(768, 512, device="cuda")
        fp8z.fp8z_dequant_rowwise(torch.from_numpy(qo).cuda(), torch.from_numpy(so).cuda(), xt, transpose=True)
        qn = torch.empty(768, 512, dtype=torch.uint8, device="cuda")
        sn = torch.empty(768, 4, device="cuda")
        fp8z.fp8z_quantize_rowwise(xt, pow2, qn, sn)
        torch.cuda.synchronize()
        qw, sw = oracle.quantize_rowwise(np.ascontiguousarray(oracle.dequant_rowwise(qo, so).T), pow2=pow2)
        assert np.array_equal(qn.cpu().numpy(), qw)
        assert np.array_equal(sn.cpu().numpy().view(np.uint32), sw.view(np.uint32))
