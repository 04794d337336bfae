// aux.cu -- dequantize, standalone column-major transpose, the E4M3 cast on
// its own, and the watchdog self-test (sm_103a).
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

constexpr int kBlk = FP8Z_BLOCK;
constexpr int kBlkElems = FP8Z_BLOCK_ELEMS;

// ------------------------------------------------------------- dequantize
// "FP8-Flow-MoE" §3.1: D(Q(x)) = Q(x) * s, here value(code) * inv_scale.
// HBM-bound (1 B read + 4 B written per element).  Persistent, one CTA per SM:
// one thread streams each block's 16 KB of codes into a ring of kDqStages
// shared buffers with bulk copies; the 1024 threads decode one 32-bit word of
// codes each per pass (exact, cvt.rn.f16x2.e4m3x2, times the block's inverse
// scale) into one of kDqOut 64 KB FP32 tiles; the thread writes the tile back
// with one 64 KB bulk store.  Measured on GB300 (65,536 blocks): 0.966 of the
// copy bandwidth, against 0.889 for a grid-stride kernel with 16-byte stores
// (plain stores cap a 1:4 read:write stream near 0.92; bulk stores write at
// 1.02 of the copy bandwidth).
constexpr int kDqStages = 3, kDqOut = 2, kDqThreads = 1024;
constexpr int kDqSmemBytes = kDqStages * kBlkElems + kDqOut * kBlkElems * 4 + kDqStages * 8 + 16;

__global__ void __launch_bounds__(kDqThreads) dequant_kernel(const uint8_t* __restrict__ q,
                                                             const float* __restrict__ inv, int64_t nblk,
                                                             float* __restrict__ out, int32_t* dev_status,
                                                             int64_t timeout_ns) {
    extern __shared__ __align__(128) unsigned char smem[];
    unsigned char* codes = smem;                                              // kDqStages x 16 KB
    float* tiles = reinterpret_cast<float*>(smem + kDqStages * kBlkElems);   // kDqOut x 64 KB
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kDqStages * kBlkElems + kDqOut * kBlkElems * 4);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + kDqStages);
    const int tid = threadIdx.x;
    const uint32_t bar0 = smem_addr(bars);
    if (tid == 0) {
        for (int s = 0; s < kDqStages; ++s) mbar_init(bar0 + 8 * s, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    const Watchdog wd{abort_flag, dev_status, timeout_ns};
    const int64_t count = (nblk - blockIdx.x + gridDim.x - 1) / gridDim.x;   // grid <= nblk
    auto issue = [&](int64_t k) {
        const int64_t b = blockIdx.x + k * gridDim.x;
        const int s = int(k % kDqStages);
        mbar_arrive_expect_tx(bar0 + 8 * s, kBlkElems);
        bulk_g2s_nohint(smem_addr(codes + s * kBlkElems), q + b * kBlkElems, kBlkElems, bar0 + 8 * s);
    };
    if (tid == 0)
        for (int64_t k = 0; k < count && k < kDqStages; ++k) issue(k);
    int64_t k = 0;
    for (; k < count; ++k) {
        const int64_t b = blockIdx.x + k * gridDim.x;
        const int s = int(k % kDqStages), ot = int(k % kDqOut);
        if (tid == 0) bulk_wait_read<kDqOut - 1>();        // tile ot has been written out
        mbar_wait_bounded(bar0 + 8 * s, uint32_t((k / kDqStages) & 1), wd);
        __syncthreads();
        if (*abort_flag) break;
        const float sc = __ldg(inv + b);
        const uint32_t* cw = reinterpret_cast<const uint32_t*>(codes + s * kBlkElems);
        float4* t4 = reinterpret_cast<float4*>(tiles + ot * kBlkElems);
#pragma unroll
        for (int it = 0; it < kBlkElems / 4 / kDqThreads; ++it) {
            const int w = it * kDqThreads + tid;
            const uint32_t word = cw[w];
            const float2 lo = e4m3x2_to_float2(word);
            const float2 hi = e4m3x2_to_float2(word >> 16);
            t4[w] = make_float4(__fmul_rn(lo.x, sc), __fmul_rn(lo.y, sc), __fmul_rn(hi.x, sc),
                                __fmul_rn(hi.y, sc));
        }
        fence_proxy_async();
        __syncthreads();
        if (tid == 0) {
            bulk_s2g(out + b * kBlkElems, smem_addr(tiles + ot * kBlkElems), kBlkElems * 4);
            bulk_commit();
            if (k + kDqStages < count) issue(k + kDqStages);
        }
    }
    if (tid == 0) {
        // gave up at block k: blocks k .. k + kDqStages - 1 may have loads in
        // flight (every earlier load was waited for); let them land
        if (k < count)
            for (int64_t kk = k; kk < count && kk < k + kDqStages; ++kk)
                mbar_wait_drain(bar0 + 8 * int(kk % kDqStages), uint32_t((kk / kDqStages) & 1), dev_status);
        bulk_wait_all();
    }
}

// -------------------------------------------------------------- transpose
// One CTA per folded block of one param: the 16 KB block is staged in a
// swizzled shared tile, each warp then emits four output rows (input columns)
// per pass with 4x4 byte transposes, a warp writing 128 contiguous bytes of
// one output row.  With one scale per 128x128 block the transposed block
// keeps its scale, so the copy is exact ("FP8-Flow-MoE" §3.1).
struct TransposeArgs {
    const uint8_t* q;          // first block of the param
    const float* inv;          // its first scale
    uint8_t* out;              // [E, W, H], ld = H
    float* inv_t;              // [E, Wb, Hb]
    int64_t H, W;
    int32_t hb, wb;
};

__global__ void __launch_bounds__(256) transpose_kernel(const TransposeArgs T) {
    __shared__ uint32_t tile[kBlkElems / 4];
    const int64_t b = blockIdx.x;                       // block within the param
    const int64_t e = b / (int64_t(T.hb) * T.wb);
    const int brow = int((b / T.wb) % T.hb);
    const int bcol = int(b % T.wb);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    const uint4* src = reinterpret_cast<const uint4*>(T.q + b * kBlkElems);
#pragma unroll
    for (int it = 0; it < 4; ++it) {
        const int idx = it * 256 + tid;                  // 16-byte chunk in the block
        const uint4 w = __ldcs(src + idx);
        const int r = idx >> 3, w0 = (idx & 7) * 4;
        const int sw = tile_swz(r);
        tile[r * 32 + ((w0 + 0) ^ sw)] = w.x;
        tile[r * 32 + ((w0 + 1) ^ sw)] = w.y;
        tile[r * 32 + ((w0 + 2) ^ sw)] = w.z;
        tile[r * 32 + ((w0 + 3) ^ sw)] = w.w;
    }
    __syncthreads();
    if (tid == 0) T.inv_t[e * T.wb * T.hb + int64_t(bcol) * T.hb + brow] = T.inv[b];

    const int vr = int(T.H - int64_t(brow) * kBlk < kBlk ? T.H - int64_t(brow) * kBlk : kBlk);
    const int vc = int(T.W - int64_t(bcol) * kBlk < kBlk ? T.W - int64_t(bcol) * kBlk : kBlk);
    const int r0 = lane * 4;
    const bool aligned = ((reinterpret_cast<uintptr_t>(T.out) | uintptr_t(T.H)) & 3) == 0;
    uint8_t* out_blk = T.out + e * T.W * T.H + int64_t(brow) * kBlk;
    if (r0 >= vr) return;
#pragma unroll
    for (int h = 0; h < 4; ++h) {
        const int cg = warp + 8 * h;
        uint32_t w4[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) w4[i] = tile[(r0 + i) * 32 + (cg ^ tile_swz(r0 + i))];
        uint32_t o[4];
        transpose4x4(w4[0], w4[1], w4[2], w4[3], o[0], o[1], o[2], o[3]);
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
            const int c = 4 * cg + cc;
            if (c >= vc) continue;
            uint8_t* dst = out_blk + (int64_t(bcol) * kBlk + c) * T.H + r0;
            if (aligned && r0 + 3 < vr) {
                *reinterpret_cast<uint32_t*>(dst) = o[cc];
            } else {
                for (int k = 0; k < 4 && r0 + k < vr; ++k) dst[k] = uint8_t(o[cc] >> (8 * k));
            }
        }
    }
}

// The same copy moved by the TMA engine (row length a multiple of 16 bytes).
// Persistent CTAs, two per SM: one thread loads each folded block with a
// 128B-swizzled tensor-map load into a ring of kTStages tiles, the eight warps
// transpose it into one of kTOut swizzled output tiles, and the thread writes
// that tile with a 3-D tensor-map store that clips at the param's edges (rows
// and cols of each expert).  Lane l takes the 4x4-byte pieces of input rows
// 4g..4g+3 with g = ((l & 15) << 1) | (l >> 4) and input column words
// (l & 15) ^ u for the warp's four units u: with the 128B swizzle on both tiles
// every shared load and store of a warp touches 32 distinct banks.  Measured on
// GB300 (32 tiles of 7168^2): 0.97-0.99 of the copy bandwidth against 0.90 for
// the one-CTA-per-block kernel above, whose global loads, shared round trip and
// stores run back to back in each CTA.
constexpr int kTStages = 4, kTOut = 2;
constexpr int kTileBytesT = kBlkElems;
constexpr int kTSmemBytes = (kTStages + kTOut) * kTileBytesT + 1024;

struct TransposeTmaArgs {
    const float* inv;          // the param's first scale
    float* inv_t;              // [E, Wb, Hb]
    int64_t nb, hb, wb;
    int32_t* dev_status;
    int64_t timeout_ns;
};

__global__ void __launch_bounds__(256) transpose_tma_kernel(const __grid_constant__ CUtensorMap in_map,
                                                            const __grid_constant__ CUtensorMap out_map,
                                                            const TransposeTmaArgs T) {
    extern __shared__ __align__(1024) unsigned char smem[];
    unsigned char* in0 = smem;
    unsigned char* out0 = smem + kTStages * kTileBytesT;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + (kTStages + kTOut) * kTileBytesT);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + kTStages);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t bar0 = smem_addr(bars);
    if (smem_addr(smem) & 1023) {          // the swizzle pattern assumes 1024-byte aligned tiles
        if (tid == 0) report_status(T.dev_status, FP8Z_EALIGN);
        return;
    }
    if (tid == 0) {
        for (int q = 0; q < kTStages; ++q) mbar_init(bar0 + 8 * q, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    const Watchdog wd{abort_flag, T.dev_status, T.timeout_ns};
    const int64_t count = (T.nb - blockIdx.x + gridDim.x - 1) / gridDim.x;   // grid <= nb
    auto issue = [&](int64_t k) {
        const int64_t b = blockIdx.x + k * gridDim.x;
        const int q = int(k % kTStages);
        mbar_arrive_expect_tx(bar0 + 8 * q, kTileBytesT);
        tma_load_2d(smem_addr(in0 + q * kTileBytesT), &in_map, 0, int(b * kBlk), bar0 + 8 * q);
    };
    if (tid == 0)
        for (int64_t k = 0; k < count && k < kTStages; ++k) issue(k);
    const int g = ((lane & 15) << 1) | (lane >> 4);       // this lane's input rows 4g..4g+3
    const int64_t per = T.hb * T.wb;
    int64_t k = 0;
    for (; k < count; ++k) {
        const int64_t b = blockIdx.x + k * gridDim.x;
        const int64_t e = b / per, brow = (b % per) / T.wb, bcol = b % T.wb;
        const int q = int(k % kTStages), ob = int(k % kTOut);
        if (tid == 0) {
            bulk_wait_read<kTOut - 1>();                   // output tile ob is free again
            T.inv_t[e * per + bcol * T.hb + brow] = T.inv[b];
        }
        mbar_wait_bounded(bar0 + 8 * q, uint32_t((k / kTStages) & 1), wd);
        __syncthreads();
        if (*abort_flag) break;
        const unsigned char* tin = in0 + q * kTileBytesT;
        unsigned char* tout = out0 + ob * kTileBytesT;
#pragma unroll
        for (int h = 0; h < 4; ++h) {
            const int cg = (lane & 15) ^ (warp * 4 + h);  // input columns 4cg..4cg+3
            uint32_t w4[4];
#pragma unroll
            for (int i = 0; i < 4; ++i)
                w4[i] = *reinterpret_cast<const uint32_t*>(tin + swz128(4 * g + i, 4 * cg));
            uint32_t o[4];
            transpose4x4(w4[0], w4[1], w4[2], w4[3], o[0], o[1], o[2], o[3]);
#pragma unroll
            for (int cc = 0; cc < 4; ++cc)                // output row 4cg+cc, bytes 4g..4g+3
                *reinterpret_cast<uint32_t*>(tout + swz128(4 * cg + cc, 4 * g)) = o[cc];
        }
        fence_proxy_async();
        __syncthreads();
        if (tid == 0) {
            tma_store_3d(&out_map, int(brow * kBlk), int(bcol * kBlk), int(e), smem_addr(tout));
            bulk_commit();
            if (k + kTStages < count) issue(k + kTStages);
        }
    }
    if (tid == 0) {
        // gave up at block k: blocks k .. k + kTStages - 1 may have loads in
        // flight (every earlier load was waited for); let them land
        if (k < count)
            for (int64_t kk = k; kk < count && kk < k + kTStages; ++kk)
                mbar_wait_drain(bar0 + 8 * int(kk % kTStages), uint32_t((kk / kTStages) & 1), T.dev_status);
        bulk_wait_all();
    }
}

// The same copy by pairs of vertically adjacent blocks (block rows brow and
// brow + 1 of one block column): the two blocks are loaded like the kernel
// above (128B-swizzled tiles), warps 0-7 transpose the first and warps 8-15
// the second, each into its half of one linear [128 output rows][256 bytes]
// tile (a 256-byte row pitch keeps the lanes' stores on 32 distinct banks), and
// one 256-byte-wide tensor-map store writes both, so every output row piece
// is 256 contiguous bytes instead of 128.  A last odd block row loads only its
// first block; the store clips the other half at the param's edge.  Two CTAs
// per SM, each with two pairs in flight and one output tile.  Measured on
// GB300 at 117 x 7168^2: 1.795 ms against 1.889 ms for the one-block kernel
// (1.005 against 0.955 of the copy bandwidth; one CTA per SM with four pairs
// and two output tiles: 2.85 ms).
constexpr int kPairStages = 2, kPairOut = 1, kPairCtasPerSm = 2;
constexpr int kPairTileBytes = 2 * kBlkElems;
constexpr int kPairSmemBytes = (kPairStages + kPairOut) * kPairTileBytes + 1024;

struct TransposePairArgs {
    const float* inv;          // the param's first scale
    float* inv_t;              // [E, Wb, Hb]
    int64_t hb, wb, hp, npairs;   // hp = ceil(hb / 2) pair rows per expert
    int32_t* dev_status;
    int64_t timeout_ns;
};

__global__ void __launch_bounds__(512, kPairCtasPerSm) transpose_pair_kernel(
    const __grid_constant__ CUtensorMap in_map, const __grid_constant__ CUtensorMap out_map,
    const TransposePairArgs P) {
    extern __shared__ __align__(1024) unsigned char smem[];
    unsigned char* in0 = smem;
    unsigned char* out0 = smem + kPairStages * kPairTileBytes;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + (kPairStages + kPairOut) * kPairTileBytes);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + kPairStages);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t bar0 = smem_addr(bars);
    if (smem_addr(smem) & 1023) {          // the swizzle pattern assumes 1024-byte aligned tiles
        if (tid == 0) report_status(P.dev_status, FP8Z_EALIGN);
        return;
    }
    if (tid == 0) {
        for (int q = 0; q < kPairStages; ++q) mbar_init(bar0 + 8 * q, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    const Watchdog wd{abort_flag, P.dev_status, P.timeout_ns};
    const int64_t count = (P.npairs - blockIdx.x + gridDim.x - 1) / gridDim.x;   // grid <= npairs
    const int64_t per = P.hp * P.wb;
    // pair k of this CTA -> expert, pair row, block column, its first block
    auto coords = [&](int64_t k, int64_t& e, int64_t& pr, int64_t& bcol, int64_t& b0) {
        const int64_t it = int64_t(blockIdx.x) + k * gridDim.x;
        e = it / per;
        pr = (it % per) / P.wb;
        bcol = it % P.wb;
        b0 = (e * P.hb + 2 * pr) * P.wb + bcol;
    };
    auto issue = [&](int64_t k) {
        int64_t e, pr, bcol, b0;
        coords(k, e, pr, bcol, b0);
        const bool second = 2 * pr + 1 < P.hb;
        const int q = int(k % kPairStages);
        mbar_arrive_expect_tx(bar0 + 8 * q, second ? kPairTileBytes : kBlkElems);
        tma_load_2d(smem_addr(in0 + q * kPairTileBytes), &in_map, 0, int(b0 * kBlk), bar0 + 8 * q);
        if (second)
            tma_load_2d(smem_addr(in0 + q * kPairTileBytes + kBlkElems), &in_map, 0, int((b0 + P.wb) * kBlk),
                        bar0 + 8 * q);
    };
    if (tid == 0)
        for (int64_t k = 0; k < count && k < kPairStages; ++k) issue(k);
    const int g = ((lane & 15) << 1) | (lane >> 4);       // this lane's input rows 4g..4g+3
    const int half = warp >> 3, w8 = warp & 7;
    int64_t k = 0;
    for (; k < count; ++k) {
        int64_t e, pr, bcol, b0;
        coords(k, e, pr, bcol, b0);
        const int q = int(k % kPairStages), ob = int(k % kPairOut);
        if (tid == 0) {
            bulk_wait_read<kPairOut - 1>();                // output tile ob is free again
            P.inv_t[e * P.wb * P.hb + bcol * P.hb + 2 * pr] = P.inv[b0];
            if (2 * pr + 1 < P.hb) P.inv_t[e * P.wb * P.hb + bcol * P.hb + 2 * pr + 1] = P.inv[b0 + P.wb];
        }
        mbar_wait_bounded(bar0 + 8 * q, uint32_t((k / kPairStages) & 1), wd);
        __syncthreads();
        if (*abort_flag) break;
        const unsigned char* tin = in0 + q * kPairTileBytes + half * kBlkElems;
        unsigned char* tout = out0 + ob * kPairTileBytes;
#pragma unroll
        for (int h = 0; h < 4; ++h) {
            const int cg = (lane & 15) ^ (w8 * 4 + h);   // input columns 4cg..4cg+3
            uint32_t w4[4];
#pragma unroll
            for (int i = 0; i < 4; ++i)
                w4[i] = *reinterpret_cast<const uint32_t*>(tin + swz128(4 * g + i, 4 * cg));
            uint32_t o[4];
            transpose4x4(w4[0], w4[1], w4[2], w4[3], o[0], o[1], o[2], o[3]);
#pragma unroll
            for (int cc = 0; cc < 4; ++cc)                // output row 4cg+cc, bytes 4g..4g+3 of this half
                *reinterpret_cast<uint32_t*>(tout + (4 * cg + cc) * 256 + half * 128 + 4 * g) = o[cc];
        }
        fence_proxy_async();
        __syncthreads();
        if (tid == 0) {
            tma_store_3d(&out_map, int(2 * pr * kBlk), int(bcol * kBlk), int(e), smem_addr(tout));
            bulk_commit();
            if (k + kPairStages < count) issue(k + kPairStages);
        }
    }
    if (tid == 0) {
        // gave up at pair k: pairs k .. k + kPairStages - 1 may have loads in
        // flight (every earlier load was waited for); let them land
        if (k < count)
            for (int64_t kk = k; kk < count && kk < k + kPairStages; ++kk)
                mbar_wait_drain(bar0 + 8 * int(kk % kPairStages), uint32_t((kk / kPairStages) & 1), P.dev_status);
        bulk_wait_all();
    }
}

// ---------------------------------------------------- E4M3 cast on its own
__global__ void encode_bits_kernel(uint32_t first, int64_t nwords, uint32_t* out) {
    const int64_t stride = int64_t(gridDim.x) * blockDim.x;
    for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < nwords; i += stride) {
        const uint32_t b = first + uint32_t(i) * 4u;
        out[i] = pack_e4m3x4(__uint_as_float(b), __uint_as_float(b + 1u), __uint_as_float(b + 2u),
                             __uint_as_float(b + 3u));
    }
}

// ------------------------------------------------------ watchdog self-test
// Waits on a barrier that nothing will complete; the bounded wait gives up
// after timeout_ns and reports FP8Z_ETIMEOUT.
__global__ void watchdog_kernel(int32_t* dev_status, int64_t timeout_ns) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x != 0) return;
    abort_flag = 0;
    const uint32_t b = smem_addr(&bar);
    mbar_init(b, 1);
    fence_mbar_init();
    const Watchdog wd{&abort_flag, dev_status, timeout_ns};
    mbar_wait_bounded(b, 0, wd);
}

int grid_for(int64_t work, int per_sm) {
    int sms = 0;
    if (host::device_sms(&sms) != FP8Z_OK) return -1;
    const int64_t full = int64_t(sms) * per_sm;
    return int(work < full ? (work > 0 ? work : 1) : full);
}

}  // namespace
}  // namespace fp8z

using namespace fp8z;

extern "C" int fp8z_dequant(const uint8_t* w_fp8, const float* inv_scale, int64_t nblk, float* out,
                            int32_t* dev_status, void* stream) {
    const fp8z::host::NvtxRange nvtx_range("fp8z_dequant");
    if (!w_fp8 || !inv_scale || !out || nblk < 0) return FP8Z_EINVAL;
    if (nblk > (INT64_MAX / kBlkElems) / 4) return FP8Z_EINVAL;
    if (!host::aligned(w_fp8, 16) || !host::aligned(out, 16) || !host::aligned(inv_scale, 4) ||
        !host::aligned(dev_status, 4))
        return FP8Z_EALIGN;
    if (nblk == 0) return FP8Z_OK;
    int sms = 0;
    int rc = host::device_sms(&sms);
    if (rc != FP8Z_OK) return rc;
    rc = host::set_smem_once(reinterpret_cast<const void*>(&dequant_kernel), 6, kDqSmemBytes);
    if (rc != FP8Z_OK) return rc;
    const unsigned grid = unsigned(nblk < sms ? nblk : sms);
    dequant_kernel<<<grid, kDqThreads, kDqSmemBytes, static_cast<cudaStream_t>(stream)>>>(
        w_fp8, inv_scale, nblk, out, dev_status, host::wait_limit_ns());
    return cudaGetLastError() == cudaSuccess ? FP8Z_OK : FP8Z_ECUDA;
}

namespace {

// The tensor maps of the TMA transpose: the param's folded blocks as a 2-D
// byte matrix of 128-byte rows, and the column-major output as [E, W, H]
// bytes.  False when a dimension is out of the engine's range.
bool transpose_maps(const fp8z_param_entry& pe, const uint8_t* blocks, uint8_t* out, CUtensorMap* in_map,
                    CUtensorMap* out_map) {
    auto enc = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(host::tensor_map_encoder());
    const int64_t nb = pe.e * pe.hb * pe.wb;
    if (!enc || nb * kBlk > 0x7FFFFFFFLL || pe.rows > 0x7FFFFFFFLL || pe.cols > 0x7FFFFFFFLL ||
        pe.e > 0x7FFFFFFFLL)
        return false;
    const cuuint32_t box2[2] = {kBlk, kBlk}, box3[3] = {kBlk, kBlk, 1}, one[3] = {1, 1, 1};
    const cuuint64_t in_dims[2] = {cuuint64_t(kBlk), cuuint64_t(nb * kBlk)};
    const cuuint64_t in_strides[1] = {cuuint64_t(kBlk)};
    const cuuint64_t out_dims[3] = {cuuint64_t(pe.rows), cuuint64_t(pe.cols), cuuint64_t(pe.e)};
    const cuuint64_t out_strides[2] = {cuuint64_t(pe.rows), cuuint64_t(pe.rows * pe.cols)};
    std::memset(in_map, 0, sizeof(CUtensorMap));
    std::memset(out_map, 0, sizeof(CUtensorMap));
    return enc(in_map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(blocks), in_dims, in_strides, box2,
               one, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS &&
           enc(out_map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, out, out_dims, out_strides, box3, one,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The pair kernel's output map: the same [E, W, H] bytes, a 256-byte-wide box,
// no swizzle (a 128B swizzle spans at most 128 bytes of a box row).
bool pair_out_map(const fp8z_param_entry& pe, uint8_t* out, CUtensorMap* map) {
    auto enc = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(host::tensor_map_encoder());
    if (!enc) return false;
    const cuuint64_t dims[3] = {cuuint64_t(pe.rows), cuuint64_t(pe.cols), cuuint64_t(pe.e)};
    const cuuint64_t strides[2] = {cuuint64_t(pe.rows), cuuint64_t(pe.rows * pe.cols)};
    const cuuint32_t box[3] = {2 * kBlk, kBlk, 1}, one[3] = {1, 1, 1};
    std::memset(map, 0, sizeof(CUtensorMap));
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, out, dims, strides, box, one, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

extern "C" int fp8z_transpose_fp8(const uint8_t* w_fp8, const float* inv_scale,
                                  const fp8z_param_entry* entry, uint8_t* out, float* inv_scale_t,
                                  int32_t* dev_status, void* stream) {
    const fp8z::host::NvtxRange nvtx_range("fp8z_transpose_fp8");
    if (!w_fp8 || !inv_scale || !entry || !out || !inv_scale_t) return FP8Z_EINVAL;
    const fp8z_param_entry& pe = *entry;
    if (pe.e < 1 || pe.rows < 1 || pe.cols < 1 || pe.blk_offset < 0) return FP8Z_EINVAL;
    if (pe.hb != (pe.rows + kBlk - 1) / kBlk || pe.wb != (pe.cols + kBlk - 1) / kBlk)
        return FP8Z_EINVAL;
    const int64_t nb = pe.e * pe.hb * pe.wb;
    if (nb > 0x7FFFFFFFLL) return FP8Z_EINVAL;
    if (!host::aligned(w_fp8, 16) || !host::aligned(out, 16) || !host::aligned(inv_scale, 4) ||
        !host::aligned(inv_scale_t, 4) || !host::aligned(dev_status, 4))
        return FP8Z_EALIGN;
    int sms = 0;
    int rc = host::device_sms(&sms);
    if (rc != FP8Z_OK) return rc;
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    const uint8_t* blocks = w_fp8 + pe.blk_offset * kBlkElems;
    CUtensorMap in_map, out_map;
    CUtensorMap out_pair;
    if (pe.rows % 16 == 0 && transpose_maps(pe, blocks, out, &in_map, &out_map) &&
        pair_out_map(pe, out, &out_pair)) {
        rc = host::set_smem_once(reinterpret_cast<const void*>(&transpose_pair_kernel), 10, kPairSmemBytes);
        if (rc != FP8Z_OK) return rc;
        TransposePairArgs P;
        P.inv = inv_scale + pe.blk_offset;
        P.inv_t = inv_scale_t;
        P.hb = pe.hb;
        P.wb = pe.wb;
        P.hp = (pe.hb + 1) / 2;
        P.npairs = pe.e * P.hp * pe.wb;
        P.dev_status = dev_status;
        P.timeout_ns = host::wait_limit_ns();
        const int64_t cap = int64_t(sms) * kPairCtasPerSm;
        transpose_pair_kernel<<<unsigned(P.npairs < cap ? P.npairs : cap), 512, kPairSmemBytes, st>>>(
            in_map, out_pair, P);
        return cudaGetLastError() == cudaSuccess ? FP8Z_OK : FP8Z_ECUDA;
    }
    if (pe.rows % 16 == 0 && transpose_maps(pe, blocks, out, &in_map, &out_map)) {
        rc = host::set_smem_once(reinterpret_cast<const void*>(&transpose_tma_kernel), 5, kTSmemBytes);
        int per_sm = 0;
        if (rc == FP8Z_OK)
            rc = host::resident_ctas(reinterpret_cast<const void*>(&transpose_tma_kernel),
                                     host::kResidentTransposeTma, 256, kTSmemBytes, &per_sm);
        if (rc != FP8Z_OK) return rc;
        const int64_t cap = int64_t(sms) * per_sm;
        TransposeTmaArgs T;
        T.inv = inv_scale + pe.blk_offset;
        T.inv_t = inv_scale_t;
        T.nb = nb;
        T.hb = pe.hb;
        T.wb = pe.wb;
        T.dev_status = dev_status;
        T.timeout_ns = host::wait_limit_ns();
        transpose_tma_kernel<<<unsigned(nb < cap ? nb : cap), 256, kTSmemBytes, st>>>(in_map, out_map, T);
        return cudaGetLastError() == cudaSuccess ? FP8Z_OK : FP8Z_ECUDA;
    }
    TransposeArgs T;
    T.q = blocks;
    T.inv = inv_scale + pe.blk_offset;
    T.out = out;
    T.inv_t = inv_scale_t;
    T.H = pe.rows;
    T.W = pe.cols;
    T.hb = pe.hb;
    T.wb = pe.wb;
    transpose_kernel<<<unsigned(nb), 256, 0, st>>>(T);
    return cudaGetLastError() == cudaSuccess ? FP8Z_OK : FP8Z_ECUDA;
}

extern "C" int fp8z_e4m3_encode_bits(uint32_t first_bits, int64_t n, uint8_t* out, void* stream) {
    const fp8z::host::NvtxRange nvtx_range("fp8z_e4m3_encode_bits");
    if (!out || n < 0 || (n & 3) != 0 || n > (int64_t(1) << 32)) return FP8Z_EINVAL;
    if (!host::aligned(out, 16)) return FP8Z_EALIGN;
    if (n == 0) return FP8Z_OK;
    const int grid = grid_for((n / 4 + 255) / 256, 8);
    if (grid < 0) return FP8Z_EUNSUPPORTED;
    encode_bits_kernel<<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(
        first_bits, n / 4, reinterpret_cast<uint32_t*>(out));
    return cudaGetLastError() == cudaSuccess ? FP8Z_OK : FP8Z_ECUDA;
}

extern "C" int fp8z_watchdog_selftest(int32_t* dev_status, int64_t timeout_ns, void* stream) {
    const fp8z::host::NvtxRange nvtx_range("fp8z_watchdog_selftest");
    if (!dev_status || timeout_ns < 0 || timeout_ns > 10000000000LL) return FP8Z_EINVAL;
    if (!host::aligned(dev_status, 4)) return FP8Z_EALIGN;
    int sms = 0;
    const int rc = host::device_sms(&sms);
    if (rc != FP8Z_OK) return rc;
    watchdog_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(dev_status, timeout_ns);
    return cudaGetLastError() == cudaSuccess ? FP8Z_OK : FP8Z_ECUDA;
}
