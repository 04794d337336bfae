"""Multi-rank host logic on CPU (gloo, world size 2): each rank plans the same
block-wise layout, takes its own shard, runs the step on it (the oracle stands
in for the device here), and the all-gather of E4M3 bytes and inverse scales
that follows the update in the ZeRO design ("Summary" of "A ZeRO Optimizer
Design for Blockwise FP8 Quantization") rebuilds exactly the unsharded result.
Also checks the benchmark's max-over-ranks timing reduction."""
import os
import socket
import traceback
import zlib

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from blockwise_fp8_zero_gb300 import fp8z

BLK = fp8z.BLOCK_ELEMS
SHAPES = [(1, 256, 384), (2, 130, 257), (1, 129, 1)]


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _inputs(cap, blocks):
    from blockwise_fp8_zero_gb300 import workloads
    out = {}
    for k, d in zip("pgmv", (workloads.Dist("normal", 0.02), workloads.Dist("normal", 1e-3),
                             workloads.Dist("normal", 2e-4), workloads.Dist("uniform", 1e-7, 4e-7))):
        t = torch.empty(cap * BLK)
        workloads.fill(t, k, d, 7, blocks["valid_rows"], blocks["valid_cols"])
        out[k] = t.numpy().copy()
    return out


def _worker(rank, world, port, q):
    try:
        os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
        dist.init_process_group("gloo", rank=rank, world_size=world)
        import oracle
        import bench
        params, shards, blocks, summ = fp8z.fp8z_plan_shards(SHAPES, world, fp8z.FP8Z_SPLIT_BLOCKWISE)
        # every rank must hold the identical plan
        h = torch.tensor([zlib.crc32(blocks.tobytes()), int(summ["capacity_blocks"])])
        hs = [torch.zeros_like(h) for _ in range(world)]
        dist.all_gather(hs, h)
        assert all(torch.equal(x, h) for x in hs)
        cap = int(summ["capacity_blocks"])
        C = int(shards["blk_capacity"][0])
        st = _inputs(cap, blocks)
        b0, nb = int(shards[rank]["blk_begin"]), int(shards[rank]["blk_count_real"])
        sl = slice(b0 * BLK, (b0 + C) * BLK)
        p, g, m, v = (st[k][sl].copy() for k in "pgmv")
        q_loc = np.zeros(C * BLK, np.uint8)
        inv_loc = np.zeros(C, np.float32)
        o_blocks = oracle.plan_shards(SHAPES, world, 0)[2]          # the oracle's own plan
        desc = np.ascontiguousarray(o_blocks[b0:b0 + C])
        oracle.adamw_requant_step(p, g, m, v, q_loc, inv_loc, 0, nb, oracle.Hparams.make(step=4),
                                  desc=desc)
        # the exchange after the update: all-gather the shard's bytes and scales
        qs = [torch.zeros(C * BLK, dtype=torch.uint8) for _ in range(world)]
        ss = [torch.zeros(C) for _ in range(world)]
        dist.all_gather(qs, torch.from_numpy(q_loc))
        dist.all_gather(ss, torch.from_numpy(inv_loc))
        whole_q = torch.cat(qs).numpy()
        whole_s = torch.cat(ss).numpy()
        # reference: one process, unsharded
        p2, g2, m2, v2 = (st[k].copy() for k in "pgmv")
        q_ref = np.zeros(cap * BLK, np.uint8)
        s_ref = np.zeros(cap, np.float32)
        oracle.adamw_requant_step(p2, g2, m2, v2, q_ref, s_ref, 0, int(summ["total_blocks"]),
                                  oracle.Hparams.make(step=4),
                                  desc=o_blocks)
        data = blocks["param"] >= 0
        assert np.array_equal(whole_q, q_ref)
        assert np.array_equal(whole_s[data], s_ref[data])
        assert np.array_equal(p, p2[sl])
        # the benchmark's timing reduction takes the slowest rank
        assert bench.max_over_ranks(10.0 + rank) == 10.0 + world - 1
        dist.destroy_process_group()
        q.put((rank, "ok"))
    except Exception:  # report to the parent instead of hanging it
        q.put((rank, traceback.format_exc()))


def test_two_rank_shards_gather_to_unsharded():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=240) for _ in procs)
    for p in procs:
        p.join(timeout=60)
    assert res == {0: "ok", 1: "ok"}, res
