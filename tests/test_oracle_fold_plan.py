"""Pins for the oracle's fold/unfold and shard planner (CPU only).

fold/unfold are checked against the torch view/permute that "A ZeRO Optimizer
Design for Blockwise FP8 Quantization" prints in "Layout transform
(fold/unfold)" (run with torch, a library); the planner against tables worked
out by hand from "Param-wise split" / "Block-wise split" and invariants.
"""
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _torch_fold(w):
    """[E,H,W] with H, W multiples of 128 -> [E*Hb*Wb, 128, 128] (the page's fold)."""
    E, H, W = w.shape
    return w.view(E, H // 128, 128, W // 128, 128).permute(0, 1, 3, 2, 4).contiguous().view(-1, 128, 128)


def _torch_unfold(b, E, H, W):
    return b.view(E, H // 128, W // 128, 128, 128).permute(0, 1, 3, 2, 4).contiguous().view(E, H, W)


@pytest.mark.parametrize("shape", [(1, 128, 128), (1, 256, 384), (3, 384, 256), (2, 128, 512)])
def test_fold_matches_page_permute(oracle, shape):
    x = torch.randn(shape, generator=torch.Generator().manual_seed(1))
    got = oracle.fold(x.numpy())
    assert np.array_equal(got, _torch_fold(x).numpy())
    back = oracle.unfold(got, *shape)
    assert np.array_equal(back, x.numpy())
    assert np.array_equal(_torch_unfold(torch.from_numpy(got), *shape).numpy(), x.numpy())


@pytest.mark.parametrize("shape", [(1, 1, 1), (1, 1, 129), (1, 129, 1), (2, 300, 100), (1, 7168, 576)])
def test_fold_ragged_zero_pads(oracle, shape):
    E, H, W = shape
    x = torch.randn(shape, generator=torch.Generator().manual_seed(2))
    Hp, Wp = -(-H // 128) * 128, -(-W // 128) * 128
    padded = F.pad(x, (0, Wp - W, 0, Hp - H))
    got = oracle.fold(x.numpy())
    assert np.array_equal(got, _torch_fold(padded).numpy())
    assert np.array_equal(oracle.unfold(got, E, H, W), x.numpy())


def _plan(oracle, shapes, dp, split):
    return oracle.plan_shards(shapes, dp, split)


def test_golden_sixteen_blocks_four_ranks(oracle):
    """The ZeRO-1 walk-through of "Summary": 16 units over 4 DP ranks, 4 each;
    here one 512x512 weight = 16 blocks, block-wise split at dp = 4."""
    rows = [l.split() for l in open(os.path.join(GOLDEN, "plan_16_blocks_dp4.txt"))
            if l.strip() and not l.startswith("#")]
    params, shards, blocks, summ = _plan(oracle, [(1, 512, 512)], 4, 0)
    assert [(int(s["blk_begin"]), int(s["blk_count_real"]), int(s["blk_capacity"])) for s in shards] \
        == [tuple(int(v) for v in r) for r in rows]
    assert summ["total_blocks"] == 16 and summ["shard_pad_elems"] == 0


def test_blockwise_hand_table(oracle):
    shapes = [(1, 256, 384), (1, 128, 129), (2, 300, 100)]
    params, shards, blocks, summ = _plan(oracle, shapes, 3, 0)
    # blocks: 2*3 = 6, 1*2 = 2, 2*3*1 = 6 -> B = 14, C = ceil(14/3) = 5
    assert list(params["blk_offset"]) == [0, 6, 8]
    assert list(params["hb"]) == [2, 1, 3] and list(params["wb"]) == [3, 2, 1]
    assert list(params["t_offset"]) == [0, 256 * 384, 256 * 384 + 128 * 129]
    assert list(params["t_scale_offset"]) == [0, 6, 8]
    assert [tuple(int(x) for x in s) for s in shards] == [(0, 5, 5), (5, 5, 5), (10, 4, 5)]
    assert summ["total_blocks"] == 14 and summ["capacity_blocks"] == 15
    assert summ["real_elems"] == 256 * 384 + 128 * 129 + 2 * 300 * 100
    assert summ["fold_pad_elems"] == (128 * 256 - 128 * 129) + (2 * 384 * 128 - 2 * 300 * 100)
    assert summ["shard_pad_elems"] == 1 * 16384
    # descriptors of the ragged blocks
    b = blocks
    assert tuple(b[7].tolist()) == (1, 0, 0, 1, 128, 1)          # (1,128,129): 1 valid col
    assert tuple(b[8 + 2].tolist()) == (2, 0, 2, 0, 44, 100)      # e=0, block row 2: 44 rows
    assert tuple(b[8 + 3].tolist()) == (2, 1, 0, 0, 128, 100)
    assert tuple(b[14].tolist()) == (-1, 0, 0, 0, 0, 0)           # shard padding
    assert list(params["bucket"]) == [0, 1, 1]


def test_paramwise_hand_table(oracle):
    shapes = [(1, 256, 384), (1, 128, 129), (2, 300, 100)]
    params, shards, blocks, summ = _plan(oracle, shapes, 3, 1)
    # sizes 6, 2, 6 -> order p0, p2, p1 -> buckets 0, 1, 2; cap = 6
    assert list(params["bucket"]) == [0, 2, 1]
    assert list(params["blk_offset"]) == [0, 12, 6]
    assert [tuple(int(x) for x in s) for s in shards] == [(0, 6, 6), (6, 6, 6), (12, 2, 6)]
    assert summ["capacity_blocks"] == 18 and summ["shard_pad_elems"] == 4 * 16384
    # LPT tie-break: equal loads go to the lowest bucket
    params, shards, _, _ = _plan(oracle, [(1, 128, 128)] * 5, 2, 1)
    assert list(params["bucket"]) == [0, 1, 0, 1, 0]
    assert list(params["blk_offset"]) == [0, 3, 1, 4, 2]


def test_paramwise_more_ranks_than_params(oracle):
    """Too few params for the DP size leaves empty buckets ("Param-wise split")."""
    params, shards, blocks, summ = _plan(oracle, [(1, 256, 256), (1, 128, 128)], 4, 1)
    assert [int(s["blk_count_real"]) for s in shards] == [4, 1, 0, 0]
    assert summ["capacity_blocks"] == 16
    assert np.sum(blocks["param"] >= 0) == 5


def test_naive_flat_split_straddles(oracle):
    """An even split of the unfolded flat buffer cuts blocks ("Challenges")."""
    # one 256x256 weight: dp=2 cuts at element 32768 = start of row 128 -> no cut
    assert _plan(oracle, [(1, 256, 256)], 2, 0)[3]["naive_straddled_blocks"] == 0
    # dp=3: S = 21846 -> rows 85 and 170 -> both block rows cut -> 4 blocks
    assert _plan(oracle, [(1, 256, 256)], 3, 0)[3]["naive_straddled_blocks"] == 4
    # dp=4: S = 16384 = 64 rows -> cuts inside both block rows
    assert _plan(oracle, [(1, 256, 256)], 4, 0)[3]["naive_straddled_blocks"] == 4
    # the block-wise split never cuts: every shard is whole blocks by construction


@pytest.mark.parametrize("split", [0, 1])
@pytest.mark.parametrize("dp", [1, 2, 3, 8, 16])
def test_planner_invariants(oracle, split, dp):
    rng = np.random.default_rng(dp * 7 + split)
    shapes = [(int(rng.integers(1, 3)), int(rng.integers(1, 700)), int(rng.integers(1, 700)))
              for _ in range(23)]
    params, shards, blocks, summ = _plan(oracle, shapes, dp, split)
    B = int(summ["total_blocks"])
    cap = int(shards["blk_capacity"][0])
    assert summ["capacity_blocks"] == dp * cap >= B
    assert np.all(shards["blk_begin"] == np.arange(dp) * cap)
    assert shards["blk_count_real"].sum() == B
    # every data block is in exactly one shard, inside its real range
    owner = np.full(dp * cap, -1)
    for r, s in enumerate(shards):
        owner[s["blk_begin"]:s["blk_begin"] + s["blk_count_real"]] = r
    data = blocks["param"] >= 0
    assert np.array_equal(data, owner >= 0)
    # each param's blocks are contiguous and in one shard
    for i, pe in enumerate(params):
        nb = pe["e"] * pe["hb"] * pe["wb"]
        idx = np.nonzero(blocks["param"] == i)[0]
        assert len(idx) == nb and idx[0] == pe["blk_offset"] and idx[-1] == pe["blk_offset"] + nb - 1
        if split == 1:
            assert len(set(owner[idx])) == 1
    vr = blocks["valid_rows"][data].astype(np.int64)
    vc = blocks["valid_cols"][data].astype(np.int64)
    assert int((vr * vc).sum()) == summ["real_elems"]
    assert summ["fold_pad_elems"] == B * 16384 - summ["real_elems"]
