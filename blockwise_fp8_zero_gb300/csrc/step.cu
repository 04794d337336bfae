// step.cu -- fused AdamW + blockwise-E4M3 requantization of one DP shard
// (sm_103a).
//
// Method: "A ZeRO Optimizer Design for Blockwise FP8 Quantization", "Summary":
// each DP rank updates its folded FP32 main-param shard element-wise, then
// quantizes the new FP8 weights and per-block scales from those FP32 values.
// Update as printed in the lpnh.cn "Model-Optimizer" article §4.3; scale
// 448/amax with the 1e-6 floor of mhpn.cn "Core scaling strategies in FP8
// training" §3.2/§4.2; nearest-value E4M3 rounding of "FP8-Flow-MoE" §3.1.
//
// Design (GB300): a persistent kernel, one CTA per SM.  One producer thread
// streams each 128x128 block's g, p, m, v through a ring of shared-memory
// stages with the TMA bulk-copy engine (16 rows x 128 = 2048 floats per
// tensor per stage), so ~200 KB per SM are in flight independent of register
// pressure; it also fetches the next block's descriptor and param entry and
// hands them over through shared memory.  Sixteen consumer warps apply AdamW
// in registers, stream p', m', v' straight back to HBM and keep p' (32 values
// per thread) until the block's amax is known; the amax comes from warp
// shuffles plus one shared-memory exchange, then the same registers are cast
// to E4M3.  HBM traffic is the algorithmic 16 B read + 13 B written per
// element (+1 B for the optional column-major copy).  The producer keeps
// loading the next block while the consumers reduce and quantize, so the
// memory pipe never drains.  Every wait is bounded (fp8z_device.cuh); no
// tensor cores: the op is element-wise.
//
// Three instantiations share the pipeline: the block-scaled step on folded
// buffers; the row-major variant (grad read through TMA tensor maps from each
// param's [E,H,W] tensor, E4M3 written row-major: the fold/unfold fused in);
// and the MXFP8 variant (an E8M0 scale per 32 elements, cast stage by stage
// with no block-wide amax).
#include <atomic>
#include <cfloat>
#include <cmath>
#include <cstdint>
#include <cstring>

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "fp8z.h"
#include "fp8z_device.cuh"
#include "fp8z_host.h"

namespace fp8z {
namespace {

// Build-time shape of the pipeline.  The defaults won a sweep on GB300 at
// 6e9 elements (28.0 ms per step): a deeper ring is faster (4 and 5 stages
// lose 2-6 %), plain bulk loads beat the L2 evict-first hint (+1.5 %),
// streaming stores of the FP32 outputs help once the loads are plain, and
// reading a block's column-major copy out of the shared tile during the next
// block's first stage (instead of waiting for all warps right away) gains
// 0.3 %.  Dropped from the code after losing: L2 prefetch ahead of the ring
// (-35 %), one contiguous block range per CTA (-2.5 %), streaming stores of
// the E4M3 bytes (-2.5 %), two rows per warp per stage with 3 stages (-10 %),
// dealing block rows fastest so the column-major writes of concurrent CTAs
// continue each other (-0.6 %: the reads lose more page locality than the
// column-major writes gain), one, two or four extra warps that do only the
// column-major copy while the consumers move on (-3.8 %, -0.2 %, +0.1 %),
// the same 192 KB ring as twelve 8-row stages with warps 0-7 and 8-15 on
// alternate stages (-0.9 %), and each warp loading its next stage into
// registers before computing the current one (-0.3 %).
//   FP8Z_RING             shared-memory stages in the ring
//   FP8Z_ROWS_PER_WARP    block rows each consumer warp takes per stage
//   FP8Z_STORE_STREAMING  1: p', m', v' stored with the streaming (.cs) hint
//   FP8Z_LOAD_EVICT_FIRST 1: bulk loads carry an L2 evict-first policy
#ifndef FP8Z_RING
#define FP8Z_RING 6
#endif
#ifndef FP8Z_ROWS_PER_WARP
#define FP8Z_ROWS_PER_WARP 1
#endif
#ifndef FP8Z_STORE_STREAMING
#define FP8Z_STORE_STREAMING 1
#endif
#ifndef FP8Z_LOAD_EVICT_FIRST
#define FP8Z_LOAD_EVICT_FIRST 0
#endif

constexpr int kBlk = FP8Z_BLOCK;
constexpr int kBlkElems = FP8Z_BLOCK_ELEMS;
constexpr int kConsumerWarps = 16;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kThreads = kConsumers + 32;               // + one producer warp
constexpr int kRowsPerWarp = FP8Z_ROWS_PER_WARP;
constexpr int kStageRows = kConsumerWarps * kRowsPerWarp;
constexpr int kStageElems = kStageRows * kBlk;
constexpr int kStagesPerBlock = kBlk / kStageRows;
constexpr int kKeep = kBlkElems / (kConsumers * 4);     // float4 of p' kept per thread: 8
constexpr uint32_t kTensorStageBytes = kStageElems * 4;
constexpr uint32_t kStageBytes = 4 * kTensorStageBytes; // g, p, m, v
constexpr int kRing = FP8Z_RING;
static_assert(kBlk % kStageRows == 0, "stage rows must divide the block");
static_assert(kKeep * kConsumers * 4 == kBlkElems, "consumer layout");

constexpr size_t kRingBytes = size_t(kRing) * kStageBytes;
constexpr size_t kTileBytes = kBlkElems;                 // 16 KB byte tile
constexpr size_t kAmaxBytes = 2 * kConsumerWarps * sizeof(float);
constexpr size_t kCtxOffset = kRingBytes + kTileBytes + kAmaxBytes;
constexpr size_t kCtxBytes = 2 * 96;                     // two BlockCtx slots
constexpr size_t kBarOffset = kCtxOffset + kCtxBytes;
constexpr int kNumBars = 2 * kRing + 2;
constexpr size_t kToutOffset = (kBarOffset + kNumBars * 8 + 16 + 127) / 128 * 128;
constexpr size_t kSmemBytes = kToutOffset + kTileBytes;   // + the transposed output tile

struct StepArgs {
    float* p;
    const float* g;
    float* m;
    float* v;
    uint8_t* w_fp8;
    float* inv_scale;
    int64_t blk_begin, nblk;
    const fp8z_block_desc* desc;
    const fp8z_param_entry* params;
    int32_t nparams;
    uint8_t* w_fp8_t;
    int64_t w_fp8_t_bytes;
    float* inv_scale_t;
    int64_t inv_scale_t_count;
    int32_t* dev_status;
    int64_t timeout_ns;
    // MXFP8 variant: one E8M0 scale byte per 32 elements of a block row
    uint8_t* mx_scale;
    // row-major variant: per-param grad tensor maps, whole-param E4M3 buffer
    const CUtensorMap* g_maps;
    uint8_t* w_row;
    int64_t w_row_bytes;
    float beta1, beta2, omb1, omb2, eps, step_size, rs_bc2, decay, lr_wd;
    float fp8_max, min_scale, min_scale_pow2;
    int32_t scale_mode, decay_mode;
};

// AdamW on one element, float32, one rounding per operation, never fused.
__device__ __forceinline__ void adamw1(const StepArgs& A, float p, float g, float m, float v,
                                       float& p1, float& m1, float& v1) {
    m1 = __fadd_rn(__fmul_rn(A.beta1, m), __fmul_rn(A.omb1, g));
    v1 = __fadd_rn(__fmul_rn(A.beta2, v), __fmul_rn(A.omb2, __fmul_rn(g, g)));
    const float d = __fadd_rn(__fmul_rn(__fsqrt_rn(v1), A.rs_bc2), A.eps);
    const float su = __fmul_rn(A.step_size, __fdiv_rn(m1, d));
    if (A.decay_mode == FP8Z_DECAY_PRE) {
        p1 = __fsub_rn(__fmul_rn(p, A.decay), su);
    } else {
        const float pu = __fsub_rn(p, su);
        p1 = __fsub_rn(pu, __fmul_rn(A.lr_wd, pu));
    }
}

// Largest power of two s with s * amax <= fp8_max (amax > 0, finite), from
// the exponent and significand bits.
__device__ __forceinline__ float pow2_scale(float amax, float fp8_max) {
    auto split = [](float x, int& e, uint32_t& sig) {
        uint32_t b = __float_as_uint(x);
        uint32_t ex = b >> 23, man = b & 0x7FFFFFu;
        if (ex == 0) {                       // subnormal: normalise
            int msb = 31 - __clz(man);       // 0..22
            e = msb - 149;
            sig = (man << (23 - msb)) & 0x7FFFFFu;
        } else {
            e = int(ex) - 127;
            sig = man;
        }
    };
    int ea, em;
    uint32_t sa, sm;
    split(amax, ea, sa);
    split(fp8_max, em, sm);
    int k = em - ea - (sa > sm ? 1 : 0);
    if (k > 127) k = 127;
    if (k < -126) return 0.0f;               // amax >= 2^127 * 448: cannot happen for finite amax
    return __uint_as_float(uint32_t(k + 127) << 23);
}

__device__ __forceinline__ float block_scale(const StepArgs& A, float amax) {
    if (amax == 0.0f) return 1.0f;
    float s;
    if (A.scale_mode == FP8Z_SCALE_EXACT) {
        s = __fdiv_rn(A.fp8_max, amax);
        if (s > FLT_MAX) s = FLT_MAX;
        s = fmaxf(s, A.min_scale);
    } else {
        s = (amax > FLT_MAX) ? 0.0f : pow2_scale(amax, A.fp8_max);
        s = fmaxf(s, A.min_scale_pow2);
    }
    return s;
}

__device__ __forceinline__ int64_t imin64(int64_t a, int64_t b) { return a < b ? a : b; }

// MXFP8 shared exponent of a group with largest magnitude a: floor(log2 a) - 8
// (8 = the largest E4M3 exponent, so the largest element lands in [256, 512)),
// clamped to [-127, 127]; 0 for an all-zero group, 127 for an infinite amax.
__device__ __forceinline__ int mx_exponent(float a) {
    if (a == 0.0f) return 0;
    const uint32_t b = __float_as_uint(a);
    if ((b >> 23) == 255) return 127;     // +Inf (a NaN never becomes the amax)
    const int e = (b >> 23) == 0 ? (31 - __clz(b)) - 149 : int(b >> 23) - 127;
    const int x = e - 8;
    return x < -127 ? -127 : (x > 127 ? 127 : x);
}

// 2^k as a float for k in [-127, 127] (2^-127 is subnormal, still exact).
__device__ __forceinline__ float exp2i(int k) {
    return k >= -126 ? __uint_as_float(uint32_t(k + 127) << 23) : __uint_as_float(1u << (k + 149));
}

__device__ __forceinline__ float4 lds4(const float* p) {
    return *reinterpret_cast<const float4*>(p);
}

__device__ __forceinline__ float absmax4(float acc, float4 x) {
    return fmaxf(fmaxf(fmaxf(acc, fabsf(x.x)), fmaxf(fabsf(x.y), fabsf(x.z))), fabsf(x.w));
}

struct BlockInfo {
    int vr, vc;          // valid rows / cols
    int param, e, brow, bcol;
};

// Where a block's row-major / column-major bytes go.
struct ParamInfo {
    int64_t e, H, W, hb, wb, t_off, ts_off;
};

// Row-major variant: how a block's grad reaches the consumers.
enum GradMode : int32_t {
    kGradZero = 0,       // no valid grad (bad descriptor or map slot): grad 0
    kGradTma = 1,        // a tensor-map load into the ring's grad section
    kGradPlain = 2,      // plain loads from the param's row-major grad
};

// A row-major grad whose row pitch is not a multiple of 16 bytes cannot be
// described by a tensor map (a TMA rule); its 128-byte slot in the map table
// holds this record instead, and the consumers read that grad with plain
// 4-byte loads.  The kernel tells the two apart by the param's column count
// (cols % 4 != 0: a record) and checks the record's tag and shape.
struct PlainGrad {
    uint64_t magic;          // kPlainGradMagic
    const float* ptr;        // the grad [e, rows, cols], 4-byte aligned
    int64_t e, rows, cols;   // its shape, equal to the param entry's
    uint64_t pad[11];
};
static_assert(sizeof(PlainGrad) == 128, "one map slot");
constexpr uint64_t kPlainGradMagic = 0x31647267506e6c70ull;

// A block's descriptor and param entry, fetched from global memory by the
// producer one block ahead and handed to the consumers through shared memory
// (written before the block's first stage is armed; the mbarrier's
// release/acquire orders it).  Two slots, by block parity: the producer can
// refill a slot only after every consumer warp has released a stage of the
// following block, i.e. has finished with the block that used it.
struct BlockCtx {
    BlockInfo bi;        // 24 bytes
    ParamInfo pi;        // 56 bytes
    const float* g_rows; // row-major, kGradPlain: base of the param's grad
    int32_t g_mode;      // row-major: GradMode of the block
    int32_t pad;
};
static_assert(sizeof(BlockCtx) == 96, "context slot size");
static_assert(kRing <= kStagesPerBlock, "context slots need the producer within one block");
// the deferred column-major copy reads the previous block's context slot
// before releasing stage 1; the producer refills that slot once stage
// kStagesPerBlock - 1 - kRing of the current block is released
static_assert(kRing <= kStagesPerBlock - 2, "deferred copy needs its context slot");

__device__ __forceinline__ BlockInfo load_desc(const StepArgs& A, int64_t blk) {
    BlockInfo bi{kBlk, kBlk, -1, 0, 0, 0};
    if (A.desc) {
        const int* d = reinterpret_cast<const int*>(A.desc + blk);
        bi.param = __ldg(d + 0);
        bi.e = __ldg(d + 1);
        bi.brow = __ldg(d + 2);
        bi.bcol = __ldg(d + 3);
        const uint32_t valid = static_cast<uint32_t>(__ldg(d + 4));
        bi.vr = int(valid & 0xFFFFu);
        bi.vc = int(valid >> 16);
    }
    return bi;
}

__device__ __forceinline__ ParamInfo load_param(const StepArgs& A, const BlockInfo& bi) {
    ParamInfo pi{0, 0, 0, 0, 0, 0, 0};
    if ((A.w_fp8_t != nullptr || A.w_row != nullptr) && bi.param >= 0 && bi.param < A.nparams) {
        const fp8z_param_entry* pe = A.params + bi.param;
        pi.e = __ldg(&pe->e);
        pi.H = __ldg(&pe->rows);
        pi.W = __ldg(&pe->cols);
        pi.hb = __ldg(&pe->hb);
        pi.wb = __ldg(&pe->wb);
        pi.t_off = __ldg(&pe->t_offset);
        pi.ts_off = __ldg(&pe->t_scale_offset);
    }
    return pi;
}

__device__ __forceinline__ void store4(float* dst, float4 x) {
#if FP8Z_STORE_STREAMING
    __stcs(reinterpret_cast<float4*>(dst), x);
#else
    *reinterpret_cast<float4*>(dst) = x;
#endif
}

__device__ __forceinline__ void store_word(uint8_t* dst, uint32_t x) {
    *reinterpret_cast<uint32_t*>(dst) = x;
}

// 16-byte global store carrying an L2 eviction policy.
__device__ __forceinline__ void store_v4_hint(void* dst, uint4 x, uint64_t pol) {
    asm volatile("st.global.L2::cache_hint.v4.b32 [%0], {%1, %2, %3, %4}, %5;" ::"l"(dst), "r"(x.x), "r"(x.y),
                 "r"(x.z), "r"(x.w), "l"(pol)
                 : "memory");
}

// Which blocks a CTA owns: blocks are dealt round-robin, so at any moment the
// CTAs stream neighbouring 64 KB blocks (DRAM page locality).  The grid never
// exceeds nblk, so every CTA owns at least one block.
struct BlockSched {
    int64_t first, stride, count;
    __device__ __forceinline__ int64_t blk(int64_t i) const { return first + i * stride; }
};

__device__ __forceinline__ BlockSched block_sched(int64_t blk_begin, int64_t nblk) {
    return BlockSched{blk_begin + blockIdx.x, gridDim.x,
                      (nblk - blockIdx.x + gridDim.x - 1) / gridDim.x};
}

// Does descriptor bi name a block of param pi: index, expert, block position
// and ragged edge all agreeing with the param table?
__device__ __forceinline__ bool block_in_param(const StepArgs& A, const BlockInfo& bi, const ParamInfo& pi) {
    return bi.param >= 0 && bi.param < A.nparams && bi.e >= 0 && bi.e < pi.e && bi.brow >= 0 &&
           bi.brow < pi.hb && bi.bcol >= 0 && bi.bcol < pi.wb &&
           bi.vr == imin64(kBlk, pi.H - bi.brow * int64_t(kBlk)) &&
           bi.vc == imin64(kBlk, pi.W - bi.bcol * int64_t(kBlk));
}

// Does block bi of param pi have a destination inside a buffer of `bytes`
// bytes (and, for the transposed grid, `scales` entries)?  A descriptor that
// disagrees with the param table is rejected, so no write can leave the buffer.
__device__ __forceinline__ bool dest_ok(const StepArgs& A, const BlockInfo& bi, const ParamInfo& pi,
                                        int64_t bytes, int64_t scales) {
    const int64_t H = pi.H, W = pi.W;
    return block_in_param(A, bi, pi) && pi.t_off >= 0 && pi.t_off + (bi.e + 1) * H * W <= bytes &&
           (scales < 0 || (pi.ts_off >= 0 && pi.ts_off + (bi.e + 1) * pi.hb * pi.wb <= scales));
}

// Row-major variant: how block bi's grad is read, from its param's slot in the
// map table.  A slot that does not match the param entry (a record where a
// tensor map belongs, or a record with another shape) gives kGradZero and
// FP8Z_EINVAL; plain loads also need the descriptor to agree with the param
// table, since they are not clipped at the tensor's edge like a TMA load.
__device__ __forceinline__ int32_t grad_mode(const StepArgs& A, const BlockInfo& bi, const ParamInfo& pi,
                                             const float*& g_rows) {
    g_rows = nullptr;
    if (bi.param < 0 || bi.param >= A.nparams) return kGradZero;
    const PlainGrad* r = reinterpret_cast<const PlainGrad*>(A.g_maps + bi.param);
    const bool record = r->magic == kPlainGradMagic;
    if ((pi.W & 3) == 0) {
        if (!record) return kGradTma;
    } else if (record && block_in_param(A, bi, pi) && r->e == pi.e && r->rows == pi.H && r->cols == pi.W) {
        g_rows = r->ptr;
        return kGradPlain;
    }
    report_status(A.dev_status, FP8Z_EINVAL);
    return kGradZero;
}

// Row-major variant, kGradPlain: the four grad values of (block row `row`,
// columns col..col+3) of block bi, zero past the ragged edge.
__device__ __forceinline__ float4 load_grad_plain(const float* g_rows, const BlockInfo& bi, int64_t H, int64_t W,
                                                  int row, int col) {
    float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
    if (row >= bi.vr) return x;
    const float* src =
        g_rows + (int64_t(bi.e) * H + int64_t(bi.brow) * kBlk + row) * W + int64_t(bi.bcol) * kBlk + col;
    if (col + 0 < bi.vc) x.x = __ldg(src + 0);
    if (col + 1 < bi.vc) x.y = __ldg(src + 1);
    if (col + 2 < bi.vc) x.z = __ldg(src + 2);
    if (col + 3 < bi.vc) x.w = __ldg(src + 3);
    return x;
}

// Row-major E4M3 write of one block into the whole-param buffer ("Summary"
// of the ZeRO design page: the FP8 params are unfolded back to their 2-D/3-D
// shape; here the unfold happens on the way out).  Row r of the block is 128
// contiguous bytes of row brow*128 + r of the param; like the column-major
// copy's, these scattered rows are stored with the L2 evict-last policy.  A
// whole block whose rows start on 16 bytes is staged in the warp's own eight
// rows of the linear output tile (the column-major copy has read them out at
// the start of this block and refills them only at the next one), so that
// each lane writes 16 bytes and a warp store covers four rows.
__device__ __forceinline__ void store_rowmajor(const StepArgs& A, const BlockInfo& bi, const ParamInfo& pi,
                                               const uint32_t (&words)[kKeep], uint8_t* tout, int warp,
                                               int lane, int col) {
    const int64_t H = pi.H, W = pi.W;
    const int64_t pbase = pi.t_off + bi.e * H * W;
    const int64_t base = pbase + int64_t(bi.brow) * kBlk * W + int64_t(bi.bcol) * kBlk;
    const uint64_t keep_in_l2 = l2_evict_last_policy();
    if (bi.vr == kBlk && bi.vc == kBlk && ((pbase | W) & 15) == 0) {
        // block row k * 16 + warp goes to tout row 4 * warp + k (k < 4) or
        // 64 + 4 * warp + k - 4: the rows column_major_out gives this warp
#pragma unroll
        for (int k = 0; k < kKeep; ++k)
            *reinterpret_cast<uint32_t*>(tout + ((k >> 2) * 64 + 4 * warp + (k & 3)) * 128 + col) = words[k];
        __syncwarp();
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int k = 4 * h + (lane >> 3), ch = lane & 7;
            const uint4 x = *reinterpret_cast<const uint4*>(tout + (h * 64 + 4 * warp + (lane >> 3)) * 128 + ch * 16);
            store_v4_hint(A.w_row + base + int64_t(k * kConsumerWarps + warp) * W + ch * 16, x, keep_in_l2);
        }
        __syncwarp();
        return;
    }
    const bool aligned = ((pi.t_off + bi.e * H * W) | W) % 4 == 0;
#pragma unroll
    for (int k = 0; k < kKeep; ++k) {
        const int row = k * kConsumerWarps + warp;
        if (row >= bi.vr || col >= bi.vc) continue;
        uint8_t* dst = A.w_row + base + int64_t(row) * W + col;
        if (aligned && col + 3 < bi.vc) {
            store_u32_hint(dst, words[k], keep_in_l2);
        } else {
            for (int b = 0; b < 4 && col + b < bi.vc; ++b) dst[b] = uint8_t(words[k] >> (8 * b));
        }
    }
}

// Column-major copy of one block: the quantized words go through a swizzled
// shared tile; each warp then takes four output rows (input columns) per pass
// from 4x4 byte transposes.  The stores carry an L2 evict-last policy: a block
// adds 128 bytes to each of 128 output rows, and lines kept longer in L2 meet
// their row neighbours from other blocks before they are written back
// (28.24 -> 27.93 ms per step on GB300 at 117 x 7168^2; 1.0 of the lines beat
// 0.5 and 0.25).  A whole block whose output rows start on 16 bytes goes
// through a second, linear shared tile (the warp's own output rows, 128 bytes
// each) so that every lane writes 16 bytes and a warp store covers four output
// rows: 28.21 -> 28.06 ms against 4-byte stores straight from the transposes
// (a 128-byte bulk copy per output row, or one tensor-map store of the tile,
// measured no faster, or 10 % slower).  column_major_in stages the block
// (false when the descriptor does not match the param table: nothing is
// staged); column_major_out waits until every warp has staged its rows and
// writes the block out (false when that wait gave up).
__device__ __forceinline__ bool column_major_in(const StepArgs& A, const BlockInfo& bi, const ParamInfo& pi,
                                                const uint32_t (&words)[kKeep], float inv, uint32_t* tile,
                                                uint32_t tile_bar, int tid, int warp, int lane) {
    if (!dest_ok(A, bi, pi, A.w_fp8_t_bytes, A.inv_scale_t_count)) {
        if (tid == 0) report_status(A.dev_status, FP8Z_EINVAL);
        return false;
    }
#pragma unroll
    for (int k = 0; k < kKeep; ++k) {
        const int row = k * kConsumerWarps + warp;
        tile[row * 32 + (lane ^ tile_swz(row))] = words[k];
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(tile_bar);
    if (tid == 0) A.inv_scale_t[pi.ts_off + bi.e * pi.wb * pi.hb + bi.bcol * pi.hb + bi.brow] = inv;
    return true;
}

__device__ __forceinline__ bool column_major_out(const StepArgs& A, const BlockInfo& bi, const ParamInfo& pi,
                                                 const uint32_t* tile, uint8_t* tout, uint32_t tile_bar,
                                                 uint32_t& tile_phase, const Watchdog& wd, int warp,
                                                 int lane) {
    if (!mbar_wait_bounded(tile_bar, tile_phase, wd)) return false;
    tile_phase ^= 1;
    const uint64_t keep_in_l2 = l2_evict_last_policy();
    const int64_t H = pi.H;
    const int64_t t_base = pi.t_off + bi.e * H * pi.W;
    const int r0 = lane * 4;                           // input rows r0..r0+3
    uint8_t* out_blk = A.w_fp8_t + t_base + bi.brow * int64_t(kBlk);
    if (bi.vr == kBlk && bi.vc == kBlk && ((t_base | H) & 15) == 0) {
        // a warp writes and reads back only its own eight rows of tout, so
        // the warp barrier orders both and no other warp touches them
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int cg = warp + h * kConsumerWarps;  // input cols 4cg..4cg+3
            uint32_t w4[4];
#pragma unroll
            for (int ii = 0; ii < 4; ++ii) w4[ii] = tile[(r0 + ii) * 32 + (cg ^ tile_swz(r0 + ii))];
            uint32_t o[4];
            transpose4x4(w4[0], w4[1], w4[2], w4[3], o[0], o[1], o[2], o[3]);
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) *reinterpret_cast<uint32_t*>(tout + (4 * cg + cc) * 128 + r0) = o[cc];
        }
        __syncwarp();
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int c = 4 * (warp + h * kConsumerWarps) + (lane >> 3), ch = lane & 7;
            const uint4 x = *reinterpret_cast<const uint4*>(tout + c * 128 + ch * 16);
            store_v4_hint(out_blk + (bi.bcol * int64_t(kBlk) + c) * H + ch * 16, x, keep_in_l2);
        }
        __syncwarp();
        return true;
    }
    const bool aligned = ((t_base | H) & 3) == 0;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int cg = warp + h * kConsumerWarps;      // input cols 4cg..4cg+3
        uint32_t w4[4];
#pragma unroll
        for (int ii = 0; ii < 4; ++ii) w4[ii] = tile[(r0 + ii) * 32 + (cg ^ tile_swz(r0 + ii))];
        uint32_t o[4];
        transpose4x4(w4[0], w4[1], w4[2], w4[3], o[0], o[1], o[2], o[3]);
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
            const int c = 4 * cg + cc;
            if (c >= bi.vc || r0 >= bi.vr) continue;
            uint8_t* dst = out_blk + (bi.bcol * int64_t(kBlk) + c) * H + r0;
            if (aligned && r0 + 3 < bi.vr) {
                store_u32_hint(dst, o[cc], keep_in_l2);
            } else {
                for (int b = 0; b < 4 && r0 + b < bi.vr; ++b) dst[b] = uint8_t(o[cc] >> (8 * b));
            }
        }
    }
    return true;
}

template <bool kRowMajor, bool kMx>
__global__ void __launch_bounds__(kThreads, 1) fp8z_step_kernel(const StepArgs A) {
    extern __shared__ __align__(1024) unsigned char smem[];
    float* ring = reinterpret_cast<float*>(smem);
    uint32_t* tile = reinterpret_cast<uint32_t*>(smem + kRingBytes);
    uint8_t* tout = smem + kToutOffset;
    float* amax_x = reinterpret_cast<float*>(smem + kRingBytes + kTileBytes);
    BlockCtx* ctx = reinterpret_cast<BlockCtx*>(smem + kCtxOffset);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kBarOffset);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + kNumBars);

    const uint32_t full0 = smem_addr(bars);
    const uint32_t empty0 = smem_addr(bars + kRing);
    const uint32_t amax_bar = smem_addr(bars + 2 * kRing);
    const uint32_t tile_bar = smem_addr(bars + 2 * kRing + 1);

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;

    if (tid == 0) {
        for (int s = 0; s < kRing; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, kConsumerWarps);
        }
        mbar_init(amax_bar, kConsumerWarps);
        mbar_init(tile_bar, kConsumerWarps);
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();

    const Watchdog wd{abort_flag, A.dev_status, A.timeout_ns};
    const BlockSched sched = block_sched(A.blk_begin, A.nblk);
    const int64_t nmine = sched.count;

    if (warp == kConsumerWarps) {
        // ------------------------------------------------------ producer
        if (lane != 0) return;
#if FP8Z_LOAD_EVICT_FIRST
        const uint64_t pol = l2_evict_first_policy();
#endif
        const uint32_t ring0 = smem_addr(ring);
        int slot = 0;
        uint32_t phase = 0;
        int64_t issued = 0;
        int32_t acquired_map = -1;        // row-major: the grad map this thread last acquired
        BlockInfo pbi = load_desc(A, sched.blk(0));
        int32_t pmode = kGradZero;
        {
            const ParamInfo pi0 = load_param(A, pbi);
            const float* g_rows = nullptr;
            if (kRowMajor) pmode = grad_mode(A, pbi, pi0, g_rows);
            ctx[0].bi = pbi;
            ctx[0].pi = pi0;
            ctx[0].g_rows = g_rows;
            ctx[0].g_mode = pmode;
        }
        for (int64_t i = 0; i < nmine; ++i) {
            const size_t base = size_t(sched.blk(i)) * kBlkElems;
            const bool has_next = i + 1 < nmine;
            // the next block's descriptor now, its param entry mid-block: both
            // have landed by the time the next block's context is written
            BlockInfo pnext = pbi;
            ParamInfo pinext{0, 0, 0, 0, 0, 0, 0};
            if (has_next) pnext = load_desc(A, sched.blk(i + 1));
            // row-major grad, kGradTma: the stage is rows [k*16, k*16+16) of
            // the block's 128x128 tile of the param's [E,H,W] grad, zero past
            // its edge; the other modes leave the ring's grad section unloaded
            const bool g_tma = kRowMajor && pmode == kGradTma;
            if (g_tma && pbi.param != acquired_map) {
                tensormap_acquire(A.g_maps + pbi.param);
                acquired_map = pbi.param;
            }
            for (int k = 0; k < kStagesPerBlock; ++k) {
                if (has_next && k == kStagesPerBlock / 2) pinext = load_param(A, pnext);
                if (!mbar_wait_bounded(empty0 + 8 * slot, phase ^ 1, wd)) goto drain;
                // The consumers read this slot with plain loads and released it
                // (release arrive, acquired by the wait above); the TMA refill is
                // an async-proxy write, which that release/acquire alone does not
                // order after those reads.  A proxy fence on the path between
                // them does.  Without one, a variant that kept its loaded values
                // unused for a stage read refilled data in every run; with this
                // fence, or with one in every consumer before its arrive, none
                // did, and this one costs no measurable time.
                fence_proxy_async();
                const uint32_t full = full0 + 8 * slot;
                mbar_arrive_expect_tx(full, (kRowMajor && !g_tma) ? 3 * kTensorStageBytes : kStageBytes);
                const uint32_t dst = ring0 + slot * kStageBytes;
                const size_t off = base + size_t(k) * kStageElems;
                if (kRowMajor) {
                    if (g_tma)
                        tma_load_3d(dst, A.g_maps + pbi.param, pbi.bcol * kBlk,
                                    pbi.brow * kBlk + k * kStageRows, pbi.e, full);
                } else {
#if FP8Z_LOAD_EVICT_FIRST
                    bulk_g2s(dst + 0 * kTensorStageBytes, A.g + off, kTensorStageBytes, full, pol);
#else
                    bulk_g2s_nohint(dst + 0 * kTensorStageBytes, A.g + off, kTensorStageBytes, full);
#endif
                }
#if FP8Z_LOAD_EVICT_FIRST
                bulk_g2s(dst + 1 * kTensorStageBytes, A.p + off, kTensorStageBytes, full, pol);
                bulk_g2s(dst + 2 * kTensorStageBytes, A.m + off, kTensorStageBytes, full, pol);
                bulk_g2s(dst + 3 * kTensorStageBytes, A.v + off, kTensorStageBytes, full, pol);
#else
                bulk_g2s_nohint(dst + 1 * kTensorStageBytes, A.p + off, kTensorStageBytes, full);
                bulk_g2s_nohint(dst + 2 * kTensorStageBytes, A.m + off, kTensorStageBytes, full);
                bulk_g2s_nohint(dst + 3 * kTensorStageBytes, A.v + off, kTensorStageBytes, full);
#endif
                ++issued;
                if (++slot == kRing) { slot = 0; phase ^= 1; }
            }
            if (has_next) {
                const float* g_rows = nullptr;
                if (kRowMajor) pmode = grad_mode(A, pnext, pinext, g_rows);
                ctx[(i + 1) & 1].bi = pnext;
                ctx[(i + 1) & 1].pi = pinext;
                ctx[(i + 1) & 1].g_rows = g_rows;
                ctx[(i + 1) & 1].g_mode = pmode;
            }
            pbi = pnext;
        }
    drain:
        // After the last stage, or after giving up: every copy this thread
        // issued lands before it leaves, so the CTA never exits (consumers
        // that gave up may already have left) while the copy engine still
        // writes its ring.  Only the last kRing stages can be in flight: each
        // earlier stage shared its slot with a later one, issued only after
        // the consumers had read it.  The drain wait ignores the abort flag and
        // has its own, far longer limit.
        for (int64_t j = (issued > kRing ? issued - kRing : 0); j < issued; ++j)
            mbar_wait_drain(full0 + 8 * int(j % kRing), uint32_t((j / kRing) & 1), A.dev_status);
        return;
    }

    // ---------------------------------------------------------- consumers
    // Stage k holds block rows [k*kStageRows, (k+1)*kStageRows); within it,
    // warp w takes rows r*kConsumerWarps + w (r < kRowsPerWarp), each lane four
    // consecutive columns, so every warp access is 512 contiguous bytes.
    const int col = lane * 4;
    const bool transposed = (A.w_fp8_t != nullptr);
    int slot = 0;
    uint32_t phase = 0;
    uint32_t tile_phase = 0;
    bool staged = false;          // the previous block waits in the tile for its column-major copy

    for (int64_t i = 0; i < nmine; ++i) {
        const int64_t blk = sched.blk(i);
        const size_t base = size_t(blk) * kBlkElems;
        const BlockCtx* c = ctx + (i & 1);
        int vr = kBlk, vc = kBlk;
        int32_t g_mode = kGradTma;
        const float* g_rows = nullptr;
        BlockInfo gbi{};
        int64_t gH = 0, gW = 0;

        float4 keep[kKeep];
        float lmax = 0.0f;
#pragma unroll
        for (int k = 0; k < kStagesPerBlock; ++k) {
            if (!mbar_wait_bounded(full0 + 8 * slot, phase, wd)) return;
            if (k == 0) {        // the block's context is visible once its first stage is
                vr = c->bi.vr;
                vc = c->bi.vc;
                if (kRowMajor) {
                    g_mode = c->g_mode;
                    if (g_mode == kGradPlain) {
                        g_rows = c->g_rows;
                        gbi = c->bi;
                        gH = c->pi.H;
                        gW = c->pi.W;
                    }
                }
            }
            const float* st = ring + size_t(slot) * (kStageBytes / 4);
            float4 g4[kRowsPerWarp], p4[kRowsPerWarp], m4[kRowsPerWarp], v4[kRowsPerWarp];
#pragma unroll
            for (int r = 0; r < kRowsPerWarp; ++r) {
                const int e0 = r * kConsumers * 4 + tid * 4;
                g4[r] = lds4(st + 0 * kStageElems + e0);
                p4[r] = lds4(st + 1 * kStageElems + e0);
                m4[r] = lds4(st + 2 * kStageElems + e0);
                v4[r] = lds4(st + 3 * kStageElems + e0);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(empty0 + 8 * slot);
            if (++slot == kRing) { slot = 0; phase ^= 1; }
            if (kRowMajor && g_mode != kGradTma) {
#pragma unroll
                for (int r = 0; r < kRowsPerWarp; ++r)
                    g4[r] = g_mode == kGradPlain
                                ? load_grad_plain(g_rows, gbi, gH, gW,
                                                  (k * kRowsPerWarp + r) * kConsumerWarps + warp, col)
                                : make_float4(0.f, 0.f, 0.f, 0.f);
            }

#pragma unroll
            for (int r = 0; r < kRowsPerWarp; ++r) {
                float4 p1, m1, v1;
                adamw1(A, p4[r].x, g4[r].x, m4[r].x, v4[r].x, p1.x, m1.x, v1.x);
                adamw1(A, p4[r].y, g4[r].y, m4[r].y, v4[r].y, p1.y, m1.y, v1.y);
                adamw1(A, p4[r].z, g4[r].z, m4[r].z, v4[r].z, p1.z, m1.z, v1.z);
                adamw1(A, p4[r].w, g4[r].w, m4[r].w, v4[r].w, p1.w, m1.w, v1.w);

                const int kk = k * kRowsPerWarp + r;
                const int row = kk * kConsumerWarps + warp;
                if (row >= vr || col + 3 >= vc) {           // padding of a ragged edge block
                    const bool rv = row < vr;
                    if (!(rv && col + 0 < vc)) { p1.x = 0.f; m1.x = 0.f; v1.x = 0.f; }
                    if (!(rv && col + 1 < vc)) { p1.y = 0.f; m1.y = 0.f; v1.y = 0.f; }
                    if (!(rv && col + 2 < vc)) { p1.z = 0.f; m1.z = 0.f; v1.z = 0.f; }
                    if (!(rv && col + 3 < vc)) { p1.w = 0.f; m1.w = 0.f; v1.w = 0.f; }
                }
                const size_t off = base + size_t(row) * kBlk + col;
                store4(A.p + off, p1);
                store4(A.m + off, m1);
                store4(A.v + off, v1);
                if constexpr (kMx) {
                    // MXFP8: the 8 lanes of a 32-element group agree on its
                    // exponent, then cast right away -- no block-wide amax
                    float a = absmax4(0.0f, p1);
                    a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, 1));
                    a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, 2));
                    a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, 4));
                    const int ex = mx_exponent(a);
                    const float mult = exp2i(-ex);
                    store_word(A.w_fp8 + off, pack_e4m3x4(__fmul_rn(p1.x, mult), __fmul_rn(p1.y, mult),
                                                          __fmul_rn(p1.z, mult), __fmul_rn(p1.w, mult)));
                    if ((lane & 7) == 0)
                        A.mx_scale[size_t(blk) * (kBlkElems / 32) + size_t(row) * (kBlk / 32) + (lane >> 3)] =
                            uint8_t(ex + 127);
                } else {
                    keep[kk] = p1;
                    lmax = absmax4(lmax, p1);
                }
            }
            // The previous block's column-major copy, out of the tile now that
            // every warp has long staged its rows.  Its context slot stays valid
            // until this warp releases stage 1, and the tile is refilled only
            // after this block's amax exchange, which every warp reaches after
            // this point.
            if (k == 0 && staged) {
                const BlockCtx* pc = ctx + ((i - 1) & 1);
                if (!column_major_out(A, pc->bi, pc->pi, tile, tout, tile_bar, tile_phase, wd, warp, lane))
                    return;
                staged = false;
            }
        }
        if constexpr (!kMx) {       // MXFP8 blocks are complete after their stages
            // ---- block amax: warp shuffle, then one exchange through shared memory
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) lmax = fmaxf(lmax, __shfl_xor_sync(0xFFFFFFFFu, lmax, o));
            float* ax = amax_x + (i & 1) * kConsumerWarps;
            if (lane == 0) {
                ax[warp] = lmax;
                mbar_arrive(amax_bar);
            }
            if (!mbar_wait_bounded(amax_bar, uint32_t(i & 1), wd)) return;
            float amax = ax[0];
#pragma unroll
            for (int w = 1; w < kConsumerWarps; ++w) amax = fmaxf(amax, ax[w]);

            const float s = block_scale(A, amax);
            const float inv = __fdiv_rn(1.0f, s);
            if (tid == 0) A.inv_scale[blk] = inv;

            // ---- quantize the kept p' and store the E4M3 block
            uint32_t words[kKeep];
#pragma unroll
            for (int k = 0; k < kKeep; ++k) {
                const float4 x = keep[k];
                words[k] = pack_e4m3x4(__fmul_rn(x.x, s), __fmul_rn(x.y, s), __fmul_rn(x.z, s),
                                       __fmul_rn(x.w, s));
                if (!kRowMajor) {
                    const int row = k * kConsumerWarps + warp;
                    store_word(A.w_fp8 + base + size_t(row) * kBlk + col, words[k]);
                }
            }
            const BlockInfo bi = c->bi;
            const ParamInfo pi = c->pi;
            if (kRowMajor && bi.param >= 0) {
                if (dest_ok(A, bi, pi, A.w_row_bytes, -1))
                    store_rowmajor(A, bi, pi, words, tout, warp, lane, col);
                else if (tid == 0)
                    report_status(A.dev_status, FP8Z_EINVAL);
            }

            // ---- optional column-major copy of the param + transposed scale grid
            if (transposed && bi.param >= 0) {
                staged = column_major_in(A, bi, pi, words, inv, tile, tile_bar, tid, warp, lane);
            }
        }
    }
    if (staged) {
        const BlockCtx* pc = ctx + ((nmine - 1) & 1);
        column_major_out(A, pc->bi, pc->pi, tile, tout, tile_bar, tile_phase, wd, warp, lane);
    }
}

}  // namespace
}  // namespace fp8z

using namespace fp8z;

namespace {

// Checks shared by the three step entry points; fills the common fields of A.
// The per-block output scales (inv_scale or the E8M0 grid) are each entry's own.
int prepare(StepArgs& A, float* p, float* m, float* v, int64_t capacity_blocks,
            int64_t blk_begin, int64_t nblk, const fp8z_block_desc* desc,
            const fp8z_param_entry* params, int32_t nparams, uint8_t* w_fp8_t,
            int64_t w_fp8_t_bytes, float* inv_scale_t, int64_t inv_scale_t_count,
            const fp8z_adamw_hparams* hp, int32_t* dev_status) {
    if (!p || !m || !v || !hp) return FP8Z_EINVAL;
    if (capacity_blocks < 0 || blk_begin < 0 || nblk < 0) return FP8Z_EINVAL;
    if (capacity_blocks > (INT64_MAX / kBlkElems) / 4) return FP8Z_EINVAL;
    if (blk_begin > capacity_blocks || nblk > capacity_blocks - blk_begin) return FP8Z_ENOSPACE;
    const bool want_t = (w_fp8_t != nullptr) || (inv_scale_t != nullptr);
    if (want_t && (!w_fp8_t || !inv_scale_t || !desc || !params || nparams <= 0 ||
                   w_fp8_t_bytes < 0 || inv_scale_t_count < 0))
        return FP8Z_EINVAL;
    if (!host::aligned(p, 16) || !host::aligned(m, 16) || !host::aligned(v, 16) ||
        !host::aligned(desc, 4) || !host::aligned(params, 8) ||
        !host::aligned(w_fp8_t, 16) || !host::aligned(inv_scale_t, 4) || !host::aligned(dev_status, 4))
        return FP8Z_EALIGN;
    if (!host::hparams_valid(*hp)) return FP8Z_EINVAL;
    std::memset(&A, 0, sizeof(A));
    A.p = p; A.m = m; A.v = v;
    A.blk_begin = blk_begin; A.nblk = nblk;
    A.desc = desc;
    A.params = params;
    A.nparams = params ? nparams : 0;
    A.w_fp8_t = want_t ? w_fp8_t : nullptr;
    A.w_fp8_t_bytes = w_fp8_t_bytes;
    A.inv_scale_t = want_t ? inv_scale_t : nullptr;
    A.inv_scale_t_count = inv_scale_t_count;
    A.dev_status = dev_status;
    A.timeout_ns = host::wait_limit_ns();
    const host::AdamwScalars sc = host::adamw_scalars(*hp);
    A.beta1 = sc.beta1; A.beta2 = sc.beta2; A.omb1 = sc.omb1; A.omb2 = sc.omb2;
    A.eps = sc.eps; A.step_size = sc.step_size; A.rs_bc2 = sc.rs_bc2;
    A.decay = sc.decay; A.lr_wd = sc.lr_wd;
    A.fp8_max = hp->fp8_max; A.min_scale = hp->min_scale;
    A.min_scale_pow2 = host::pow2_at_least(hp->min_scale);
    A.scale_mode = hp->scale_mode; A.decay_mode = hp->decay_mode;
    return FP8Z_OK;
}

template <bool kRowMajor, bool kMx = false>
int launch(const StepArgs& A, void* stream) {
    if (A.nblk == 0) return FP8Z_OK;
    int sms = 0;
    int rc = host::device_sms(&sms);
    if (rc != FP8Z_OK) return rc;
    static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
    rc = host::set_smem_once(reinterpret_cast<const void*>(&fp8z_step_kernel<kRowMajor, kMx>),
                             kMx ? 4 : (kRowMajor ? 1 : 0), int(kSmemBytes));
    if (rc != FP8Z_OK) return rc;
    const int64_t grid = A.nblk < sms ? A.nblk : sms;
    fp8z_step_kernel<kRowMajor, kMx><<<dim3(unsigned(grid)), dim3(kThreads), kSmemBytes,
                                       static_cast<cudaStream_t>(stream)>>>(A);
    return cudaGetLastError() == cudaSuccess ? FP8Z_OK : FP8Z_ECUDA;
}

}  // namespace

extern "C" int fp8z_adamw_requant_step(float* p, const float* g, float* m, float* v,
                                       uint8_t* w_fp8, float* inv_scale, int64_t capacity_blocks,
                                       int64_t blk_begin, int64_t nblk,
                                       const fp8z_block_desc* desc,
                                       const fp8z_param_entry* params, int32_t nparams,
                                       uint8_t* w_fp8_t, int64_t w_fp8_t_bytes,
                                       float* inv_scale_t, int64_t inv_scale_t_count,
                                       const fp8z_adamw_hparams* hp, int32_t* dev_status,
                                       void* stream) {
    const fp8z::host::NvtxRange nvtx_range("fp8z_adamw_requant_step");
    if (!g || !w_fp8 || !inv_scale) return FP8Z_EINVAL;
    if (!host::aligned(g, 16) || !host::aligned(w_fp8, 16) || !host::aligned(inv_scale, 4))
        return FP8Z_EALIGN;
    const bool want_t = (w_fp8_t != nullptr) || (inv_scale_t != nullptr);
    StepArgs A;
    const int rc = prepare(A, p, m, v, capacity_blocks, blk_begin, nblk, desc,
                           want_t ? params : nullptr, nparams, w_fp8_t, w_fp8_t_bytes, inv_scale_t,
                           inv_scale_t_count, hp, dev_status);
    if (rc != FP8Z_OK) return rc;
    A.g = g;
    A.w_fp8 = w_fp8;
    A.inv_scale = inv_scale;
    return launch<false, false>(A, stream);
}

extern "C" int fp8z_adamw_requant_step_rowmajor(float* p, float* m, float* v, const void* g_maps,
                                                uint8_t* w_row, int64_t w_row_bytes, float* inv_scale,
                                                int64_t capacity_blocks, int64_t blk_begin, int64_t nblk,
                                                const fp8z_block_desc* desc,
                                                const fp8z_param_entry* params, int32_t nparams,
                                                uint8_t* w_fp8_t, int64_t w_fp8_t_bytes,
                                                float* inv_scale_t, int64_t inv_scale_t_count,
                                                const fp8z_adamw_hparams* hp, int32_t* dev_status,
                                                void* stream) {
    const fp8z::host::NvtxRange nvtx_range("fp8z_adamw_requant_step_rowmajor");
    if (!g_maps || !w_row || !inv_scale || !desc || !params || nparams <= 0 || w_row_bytes < 0)
        return FP8Z_EINVAL;
    if (!host::aligned(g_maps, 64) || !host::aligned(w_row, 16) || !host::aligned(inv_scale, 4))
        return FP8Z_EALIGN;
    StepArgs A;
    const int rc = prepare(A, p, m, v, capacity_blocks, blk_begin, nblk, desc, params,
                           nparams, w_fp8_t, w_fp8_t_bytes, inv_scale_t, inv_scale_t_count, hp,
                           dev_status);
    if (rc != FP8Z_OK) return rc;
    A.g_maps = static_cast<const CUtensorMap*>(g_maps);
    A.inv_scale = inv_scale;
    A.w_row = w_row;
    A.w_row_bytes = w_row_bytes;
    return launch<true, false>(A, stream);
}

extern "C" int fp8z_adamw_requant_step_mx(float* p, const float* g, float* m, float* v,
                                          uint8_t* w_fp8, uint8_t* mx_scale, int64_t capacity_blocks,
                                          int64_t blk_begin, int64_t nblk, const fp8z_block_desc* desc,
                                          const fp8z_adamw_hparams* hp, int32_t* dev_status,
                                          void* stream) {
    const fp8z::host::NvtxRange nvtx_range("fp8z_adamw_requant_step_mx");
    if (!g || !w_fp8 || !mx_scale) return FP8Z_EINVAL;
    if (!host::aligned(g, 16) || !host::aligned(w_fp8, 16)) return FP8Z_EALIGN;
    StepArgs A;
    const int rc = prepare(A, p, m, v, capacity_blocks, blk_begin, nblk, desc, nullptr, 0, nullptr, 0,
                           nullptr, 0, hp, dev_status);
    if (rc != FP8Z_OK) return rc;
    A.g = g;
    A.w_fp8 = w_fp8;
    A.mx_scale = mx_scale;
    return launch<false, true>(A, stream);
}

extern "C" int fp8z_encode_grad_maps(const void* const* g_ptrs, const fp8z_param_entry* params,
                                     int32_t nparams, void* maps_out) {
    const fp8z::host::NvtxRange nvtx_range("fp8z_encode_grad_maps");
    if (!g_ptrs || !params || !maps_out || nparams <= 0) return FP8Z_EINVAL;
    if (!host::aligned(maps_out, 64)) return FP8Z_EALIGN;
    auto enc = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(host::tensor_map_encoder());
    if (!enc) return FP8Z_ECUDA;
    CUtensorMap* maps = static_cast<CUtensorMap*>(maps_out);
    for (int32_t i = 0; i < nparams; ++i) {
        const fp8z_param_entry& pe = params[i];
        if (!g_ptrs[i] || pe.e < 1 || pe.rows < 1 || pe.cols < 1 || pe.e > 0x7FFFFFFFLL ||
            pe.rows > 0xFFFFFFFFLL || pe.cols > 0xFFFFFFFFLL)
            return FP8Z_EINVAL;
        if ((pe.cols * 4) % 16 != 0) {
            // no tensor map can step over these rows: the slot holds a record
            // for plain loads instead
            if (!host::aligned(g_ptrs[i], 4)) return FP8Z_EALIGN;
            PlainGrad rec;
            std::memset(&rec, 0, sizeof(rec));
            rec.magic = kPlainGradMagic;
            rec.ptr = static_cast<const float*>(g_ptrs[i]);
            rec.e = pe.e;
            rec.rows = pe.rows;
            rec.cols = pe.cols;
            std::memcpy(&maps[i], &rec, sizeof(rec));
            continue;
        }
        if (!host::aligned(g_ptrs[i], 16)) return FP8Z_EALIGN;
        const cuuint64_t dims[3] = {cuuint64_t(pe.cols), cuuint64_t(pe.rows), cuuint64_t(pe.e)};
        const cuuint64_t strides[2] = {cuuint64_t(pe.cols * 4), cuuint64_t(pe.rows * pe.cols * 4)};
        const cuuint32_t boxd[3] = {kBlk, kStageRows, 1};
        const cuuint32_t estr[3] = {1, 1, 1};
        std::memset(&maps[i], 0, sizeof(CUtensorMap));
        if (enc(&maps[i], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(g_ptrs[i]), dims, strides,
                boxd, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return FP8Z_EINVAL;
    }
    return FP8Z_OK;
}

// ------------------------------------------- row-major step, no allocation
// The grad tensor maps of fp8z_adamw_requant_step_rowmajor_static live in this
// array, not in a buffer the caller allocates.  Every device that loads the
// library holds it (128 KB) until the process exits; host code reaches it
// only through the address cudaGetSymbolAddress gives for the current device.
static __device__ __align__(256) CUtensorMap g_static_grad_maps[FP8Z_STATIC_GRAD_MAPS];

namespace {

constexpr int kMaxStaticDevices = 64;
std::atomic<void*> g_static_maps_addr[kMaxStaticDevices];

// Device address of g_static_grad_maps on the current device, looked up once
// per device (with that device current) and kept.
int static_maps_address(void** addr) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return FP8Z_ECUDA;
    if (dev < 0 || dev >= kMaxStaticDevices) return FP8Z_EUNSUPPORTED;
    void* a = g_static_maps_addr[dev].load(std::memory_order_acquire);
    if (!a) {
        if (cudaGetSymbolAddress(&a, g_static_grad_maps) != cudaSuccess || !a) return FP8Z_ECUDA;
        g_static_maps_addr[dev].store(a, std::memory_order_release);
    }
    *addr = a;
    return FP8Z_OK;
}

}  // namespace

extern "C" int fp8z_adamw_requant_step_rowmajor_static(
    float* p, float* m, float* v, const void* const* g_ptrs, const fp8z_param_entry* params_host,
    uint8_t* w_row, int64_t w_row_bytes, float* inv_scale, int64_t capacity_blocks, int64_t blk_begin,
    int64_t nblk, const fp8z_block_desc* desc, const fp8z_param_entry* params, int32_t nparams,
    uint8_t* w_fp8_t, int64_t w_fp8_t_bytes, float* inv_scale_t, int64_t inv_scale_t_count,
    const fp8z_adamw_hparams* hp, int32_t* dev_status, void* stream) {
    const fp8z::host::NvtxRange nvtx_range("fp8z_adamw_requant_step_rowmajor_static");
    if (!g_ptrs || !params_host || !w_row || !inv_scale || !desc || !params || nparams <= 0 ||
        w_row_bytes < 0)
        return FP8Z_EINVAL;
    if (nparams > FP8Z_STATIC_GRAD_MAPS) return FP8Z_ENOSPACE;
    if (!host::aligned(w_row, 16) || !host::aligned(inv_scale, 4)) return FP8Z_EALIGN;
    StepArgs A;
    int rc = prepare(A, p, m, v, capacity_blocks, blk_begin, nblk, desc, params, nparams, w_fp8_t,
                     w_fp8_t_bytes, inv_scale_t, inv_scale_t_count, hp, dev_status);
    if (rc != FP8Z_OK) return rc;
    if (nblk == 0) return FP8Z_OK;
    void* maps = nullptr;
    rc = static_maps_address(&maps);
    if (rc != FP8Z_OK) return rc;
    // Encode the maps on the host a few at a time and copy them into the
    // array on the stream, ahead of the launch.  A copy from pageable host
    // memory has read its source by the time cudaMemcpyAsync returns, so the
    // staging buffer can be reused at once.
    constexpr int kChunk = 32;
    alignas(64) CUtensorMap chunk[kChunk];
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    for (int32_t i = 0; i < nparams; i += kChunk) {
        const int32_t n = nparams - i < kChunk ? nparams - i : kChunk;
        rc = fp8z_encode_grad_maps(g_ptrs + i, params_host + i, n, chunk);
        if (rc != FP8Z_OK) return rc;
        if (cudaMemcpyAsync(static_cast<CUtensorMap*>(maps) + i, chunk, size_t(n) * sizeof(CUtensorMap),
                            cudaMemcpyHostToDevice, st) != cudaSuccess)
            return FP8Z_ECUDA;
    }
    A.g_maps = static_cast<const CUtensorMap*>(maps);
    A.inv_scale = inv_scale;
    A.w_row = w_row;
    A.w_row_bytes = w_row_bytes;
    return launch<true, false>(A, stream);
}
