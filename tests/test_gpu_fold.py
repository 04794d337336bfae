"""GPU fold / unfold ("Layout transform (fold/unfold)" of "A ZeRO Optimizer
Design for Blockwise FP8 Quantization") against the oracle's fold/unfold,
bit for bit, on the TMA path (row pitch a multiple of 16 bytes) and the plain
path, for FP32 and E4M3 bytes, alone and inside a multi-param folded buffer."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from blockwise_fp8_zero_gb300 import fp8z  # noqa: E402

pytestmark = pytest.mark.gpu
BLK = fp8z.BLOCK_ELEMS


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from blockwise_fp8_zero_gb300 import build
    build.build()
    fp8z.lib()


SHAPES = [(1, 256, 384), (2, 300, 260), (1, 129, 1), (3, 7, 1000), (1, 130, 257), (1, 7168, 576),
          (2, 1, 4096)]
# extreme aspect ratios: a 2 MB row pitch (4096 blocks per block row), 4097
# block rows, and 4096 one-block experts (the tensor maps' outer dimension)
EXTREME = [(1, 130, 1 << 19), (1, (1 << 19) + 5, 136), (4096, 16, 16)]


def _entry(shape):
    params, _, _, _ = fp8z.fp8z_plan_shards([shape], 1, 0, with_blocks=False)
    return params[0]


@pytest.mark.parametrize("shape", SHAPES + EXTREME)
def test_fold_unfold_fp32(oracle, shape):
    E, H, W = shape
    x = torch.randn(shape, generator=torch.Generator().manual_seed(E * H + W))
    ent = _entry(shape)
    nb = E * int(ent["hb"]) * int(ent["wb"])
    blocks = torch.full((nb * BLK,), 7.0, device="cuda")        # padding must be overwritten
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    fp8z.fp8z_fold(x.cuda(), ent, blocks, dev_status=st)
    back = torch.full(shape, -1.0, device="cuda")
    fp8z.fp8z_unfold(blocks, ent, back, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    want = oracle.fold(x.numpy()).ravel()
    assert np.array_equal(blocks.cpu().numpy().view(np.uint32), want.view(np.uint32))
    assert np.array_equal(back.cpu().numpy(), oracle.unfold(want.reshape(-1, 128, 128), E, H, W))


@pytest.mark.parametrize("shape", SHAPES + EXTREME)
def test_fold_unfold_bytes(oracle, shape):
    E, H, W = shape
    g = torch.Generator().manual_seed(W)
    x = torch.randint(0, 256, shape, dtype=torch.uint8, generator=g)
    ent = _entry(shape)
    nb = E * int(ent["hb"]) * int(ent["wb"])
    blocks = torch.full((nb * BLK,), 0x55, dtype=torch.uint8, device="cuda")
    fp8z.fp8z_fold(x.cuda(), ent, blocks)
    back = torch.zeros(shape, dtype=torch.uint8, device="cuda")
    fp8z.fp8z_unfold(blocks, ent, back)
    torch.cuda.synchronize()
    want = oracle.fold(x.numpy().astype(np.float32)).ravel().astype(np.uint8)
    assert np.array_equal(blocks.cpu().numpy(), want)
    assert np.array_equal(back.cpu().numpy(), x.numpy())


def test_fold_into_multi_param_buffer_leaves_neighbours(oracle):
    shapes = [(1, 300, 200), (2, 128, 640), (1, 64, 64)]
    params, shards, blocks, summ = fp8z.fp8z_plan_shards(shapes, 2, 1)
    cap = int(summ["capacity_blocks"])
    buf = torch.full((cap * BLK,), 3.0, device="cuda")
    x = torch.randn(shapes[1])
    fp8z.fp8z_fold(x.cuda(), params[1], buf)
    torch.cuda.synchronize()
    got = buf.cpu().numpy()
    o = int(params[1]["blk_offset"])
    nb = 2 * 1 * 5
    assert np.array_equal(got[o * BLK:(o + nb) * BLK], oracle.fold(x.numpy()).ravel())
    assert np.all(got[:o * BLK] == 3.0) and np.all(got[(o + nb) * BLK:] == 3.0)


def test_unfold_step_output_large(oracle):
    """A 7168x18432 FP32 weight through fold, and its E4M3 codes back out."""
    shape = (1, 7168, 18432)
    ent = _entry(shape)
    nb = int(ent["hb"]) * int(ent["wb"])
    x = torch.randn(shape, device="cuda")
    blocks = torch.empty(nb * BLK, device="cuda")
    fp8z.fp8z_fold(x, ent, blocks)
    y = torch.empty_like(x)
    fp8z.fp8z_unfold(blocks, ent, y)
    torch.cuda.synchronize()
    assert torch.equal(x, y)
    # spot-check the folded order against the page's view/permute on the GPU
    ref = x.view(1, 56, 128, 144, 128).permute(0, 1, 3, 2, 4).contiguous().view(-1)
    assert torch.equal(blocks, ref)
