// plan.cpp -- host shard planner for the block-aware ZeRO-1 layout.
//
// "A ZeRO Optimizer Design for Blockwise FP8 Quantization":
//   "Block-wise split": pad every quantized dim to a multiple of 128, fold the
//     params into a flat buffer of 128x128 blocks and cut it on block
//     boundaries; a lookup table keeps the real sizes and the padding.
//   "Param-wise split": sort the FP8 params by size, spread them greedily over
//     the DP buckets, and pad every bucket to the largest one.
//   "Challenges": an even split of the plain flattened buffer can cut a
//     128x128 block across two ranks; the summary counts such blocks.
#include <algorithm>
#include <cstring>
#include <functional>
#include <numeric>
#include <queue>
#include <utility>
#include <vector>

#include "fp8z.h"
#include "fp8z_host.h"

namespace {

constexpr int64_t kB = FP8Z_BLOCK;

inline int64_t div_up(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Blocks cut by an even split (shard size S = ceil(N/dp)) of the unfolded flat
// buffer.  Shards are intervals, so a block whose lowest and highest flat
// indices fall in the same shard lies wholly inside it, and one whose ends fall
// in different shards is cut.
int64_t count_naive_straddled(const fp8z_param_shape* shapes, int32_t n, int32_t dp) {
    int64_t total = 0;
    for (int32_t i = 0; i < n; ++i) total += shapes[i].e * shapes[i].rows * shapes[i].cols;
    if (total == 0) return 0;
    const int64_t S = div_up(total, dp);
    int64_t base = 0, cut = 0;
    for (int32_t i = 0; i < n; ++i) {
        const int64_t E = shapes[i].e, H = shapes[i].rows, W = shapes[i].cols;
        for (int64_t e = 0; e < E; ++e) {
            for (int64_t r0 = 0; r0 < H; r0 += kB) {
                const int64_t r1 = std::min(H, r0 + kB) - 1;
                for (int64_t c0 = 0; c0 < W; c0 += kB) {
                    const int64_t c1 = std::min(W, c0 + kB) - 1;
                    const int64_t first = base + (e * H + r0) * W + c0;
                    const int64_t last = base + (e * H + r1) * W + c1;
                    cut += (first / S) != (last / S);
                }
            }
        }
        base += E * H * W;
    }
    return cut;
}

}  // namespace

extern "C" int fp8z_plan_shards(const fp8z_param_shape* shapes, int32_t nparams, int32_t dp,
                                int32_t split, fp8z_param_entry* params_out,
                                fp8z_shard* shards_out, fp8z_block_desc* blocks_out,
                                int64_t blocks_cap, fp8z_plan_summary* summary_out) {
    const fp8z::host::NvtxRange nvtx_range("fp8z_plan_shards");
    if (nparams < 0 || dp < 1 || !params_out || !shards_out || !summary_out) return FP8Z_EINVAL;
    if (split != FP8Z_SPLIT_BLOCKWISE && split != FP8Z_SPLIT_PARAMWISE) return FP8Z_EINVAL;
    if (nparams > 0 && !shapes) return FP8Z_EINVAL;
    for (int32_t i = 0; i < nparams; ++i) {
        const fp8z_param_shape& s = shapes[i];
        // block indices are int32 in the descriptor, valid counts uint16
        if (s.e < 1 || s.rows < 1 || s.cols < 1) return FP8Z_EINVAL;
        if (s.e > (1LL << 31) - 1 || s.rows > (1LL << 37) || s.cols > (1LL << 37))
            return FP8Z_EINVAL;
    }
    {   // the folded buffer (blocks x 16384 x 4 bytes) must stay addressable
        int64_t blocks = 0;
        for (int32_t i = 0; i < nparams; ++i) {
            const int64_t hb = div_up(shapes[i].rows, kB), wb = div_up(shapes[i].cols, kB);
            if (hb * wb > (1LL << 44) / shapes[i].e) return FP8Z_EINVAL;
            blocks += shapes[i].e * hb * wb;
            if (blocks > (1LL << 44)) return FP8Z_EINVAL;
        }
    }

    // per-param geometry and offsets of the concatenated column-major copies
    std::vector<int64_t> nblocks(static_cast<size_t>(nparams));
    int64_t real = 0, total_blocks = 0, t_off = 0, ts_off = 0;
    for (int32_t i = 0; i < nparams; ++i) {
        const fp8z_param_shape& s = shapes[i];
        fp8z_param_entry pe;
        std::memset(&pe, 0, sizeof(pe));
        pe.e = s.e;
        pe.rows = s.rows;
        pe.cols = s.cols;
        pe.hb = static_cast<int32_t>(div_up(s.rows, kB));
        pe.wb = static_cast<int32_t>(div_up(s.cols, kB));
        pe.t_offset = t_off;
        pe.t_scale_offset = ts_off;
        nblocks[i] = s.e * pe.hb * pe.wb;
        real += s.e * s.rows * s.cols;
        total_blocks += nblocks[i];
        t_off += s.e * s.rows * s.cols;
        ts_off += nblocks[i];
        params_out[i] = pe;
    }

    int64_t cap = 0;
    std::vector<int64_t> load(static_cast<size_t>(dp), 0);
    if (split == FP8Z_SPLIT_BLOCKWISE) {
        cap = div_up(total_blocks, dp);
        int64_t off = 0;
        for (int32_t i = 0; i < nparams; ++i) {
            params_out[i].blk_offset = off;
            params_out[i].bucket = cap ? static_cast<int32_t>(off / cap) : 0;
            off += nblocks[i];
        }
        for (int32_t r = 0; r < dp; ++r)
            load[r] = std::max<int64_t>(0, std::min<int64_t>(cap, total_blocks - r * cap));
    } else {
        // longest-processing-time greedy: biggest param first onto the least
        // loaded bucket; ties keep model order and go to the lowest bucket
        std::vector<int32_t> order(static_cast<size_t>(nparams));
        std::iota(order.begin(), order.end(), 0);
        std::stable_sort(order.begin(), order.end(),
                         [&](int32_t a, int32_t b) { return nblocks[a] > nblocks[b]; });
        using Slot = std::pair<int64_t, int32_t>;   // (load, bucket): min-heap order
        std::priority_queue<Slot, std::vector<Slot>, std::greater<Slot>> heap;
        for (int32_t r = 0; r < dp; ++r) heap.push({0, r});
        std::vector<int64_t> local(static_cast<size_t>(nparams));
        for (int32_t i : order) {
            Slot s = heap.top();
            heap.pop();
            params_out[i].bucket = s.second;
            local[i] = s.first;
            s.first += nblocks[i];
            load[s.second] = s.first;
            heap.push(s);
        }
        cap = *std::max_element(load.begin(), load.end());
        for (int32_t i = 0; i < nparams; ++i)
            params_out[i].blk_offset = params_out[i].bucket * cap + local[i];
    }
    for (int32_t r = 0; r < dp; ++r) {
        shards_out[r].blk_begin = r * cap;
        shards_out[r].blk_count_real = load[r];
        shards_out[r].blk_capacity = cap;
    }

    const int64_t capacity = cap * dp;
    summary_out->real_elems = real;
    summary_out->total_blocks = total_blocks;
    summary_out->fold_pad_elems = total_blocks * FP8Z_BLOCK_ELEMS - real;
    summary_out->shard_pad_elems = (capacity - total_blocks) * FP8Z_BLOCK_ELEMS;
    summary_out->capacity_blocks = capacity;
    summary_out->naive_straddled_blocks = count_naive_straddled(shapes, nparams, dp);

    if (!blocks_out) return FP8Z_OK;
    if (blocks_cap < capacity) return FP8Z_ENOSPACE;
    const fp8z_block_desc pad = {-1, 0, 0, 0, 0, 0};
    std::fill(blocks_out, blocks_out + capacity, pad);
    for (int32_t i = 0; i < nparams; ++i) {
        const fp8z_param_entry& pe = params_out[i];
        int64_t b = pe.blk_offset;
        for (int64_t e = 0; e < pe.e; ++e)
            for (int32_t hb = 0; hb < pe.hb; ++hb)
                for (int32_t wb = 0; wb < pe.wb; ++wb, ++b) {
                    fp8z_block_desc& d = blocks_out[b];
                    d.param = i;
                    d.e = static_cast<int32_t>(e);
                    d.brow = hb;
                    d.bcol = wb;
                    d.valid_rows = static_cast<uint16_t>(std::min<int64_t>(kB, pe.rows - hb * kB));
                    d.valid_cols = static_cast<uint16_t>(std::min<int64_t>(kB, pe.cols - wb * kB));
                }
    }
    return FP8Z_OK;
}
