// rowwise.cu -- 1x128-tile row-wise E4M3 quantization and the scaling-aware
// transpose to the column-wise layout (sm_103a).
//
// "FP8-Flow-MoE: A Casting-Free FP8 Recipe without Double Quantization Error",
// §3.1: a row-wise quantized tensor keeps one scale per 128 consecutive
// elements of a row (s = amax/448, Q(x) = round(x/s)); the column-wise layout
// a weight-gradient GEMM needs is reached without going back to high
// precision by aligning the 128 row scales of each 128x128 tile to the
// largest and re-expressing every code under it.  With power-of-two scales
// that is a pure exponent shift (E' = E - D, M' = M), exact unless the value
// underflows; dequantize -> transpose -> requantize would instead round most
// values a second time when the scales are not powers of two.
//
// Both kernels are HBM-bound: quantize 4 B in + 1 B out per element, the
// transpose 1 B in + 1 B out per element (+ 1/32 B of scales each way).
#include <cfloat>
#include <cstdint>

#include <cuda_runtime.h>

#include "fp8z.h"
#include "fp8z_device.cuh"
#include "fp8z_host.h"

namespace fp8z {
namespace {

constexpr int kTile = FP8Z_BLOCK;         // 128 elements per scale
constexpr int kTilesPerWarp = 4;          // tiles a warp has in flight

// Smallest power of two >= amax/448 (exact, from the bits of amax), kept in
// the normal float range [2^-126, 2^127].  448 = 1.75 * 2^8, so with
// amax = m * 2^e (m in [1, 2)) the answer is 2^(e-8), or 2^(e-7) when m > 1.75.
__device__ __forceinline__ float pow2_tile_scale(float amax) {
    const uint32_t b = __float_as_uint(amax);
    int e;
    uint32_t man;
    if ((b >> 23) == 0) {                 // subnormal: normalise
        const int msb = 31 - __clz(b);
        e = msb - 149;
        man = (b << (23 - msb)) & 0x7FFFFFu;
    } else {
        e = int(b >> 23) - 127;
        man = b & 0x7FFFFFu;
    }
    int k = e - 8 + (man > 0x600000u ? 1 : 0);     // 0x600000 = 0.75 * 2^23
    k = k < -126 ? -126 : (k > 127 ? 127 : k);
    return __uint_as_float(uint32_t(k + 127) << 23);
}

__global__ void __launch_bounds__(256) quantize_rowwise_kernel(const float* __restrict__ x,
                                                               int64_t ntiles, int pow2,
                                                               uint8_t* __restrict__ q,
                                                               float* __restrict__ s) {
    const int lane = threadIdx.x & 31;
    const int64_t warps = int64_t(gridDim.x) * (blockDim.x >> 5);
    const int64_t w0 = int64_t(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
    for (int64_t t0 = w0; t0 < ntiles; t0 += warps * kTilesPerWarp) {
        float4 v[kTilesPerWarp];
#pragma unroll
        for (int u = 0; u < kTilesPerWarp; ++u) {
            const int64_t t = t0 + u * warps;
            v[u] = t < ntiles ? __ldcs(reinterpret_cast<const float4*>(x + t * kTile) + lane)
                              : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int u = 0; u < kTilesPerWarp; ++u) {
            const int64_t t = t0 + u * warps;
            if (t >= ntiles) break;
            float a = fmaxf(fmaxf(fabsf(v[u].x), fabsf(v[u].y)), fmaxf(fabsf(v[u].z), fabsf(v[u].w)));
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, o));
            float sc;
            uint32_t w;
            if (a == 0.0f || pow2) {
                // a power of two: x/s is exactly x * (1/s), one multiply instead of a divide
                sc = a == 0.0f ? 1.0f : pow2_tile_scale(a);
                const float r = __fdiv_rn(1.0f, sc);
                w = pack_e4m3x4(__fmul_rn(v[u].x, r), __fmul_rn(v[u].y, r), __fmul_rn(v[u].z, r),
                                __fmul_rn(v[u].w, r));
            } else {
                sc = fmaxf(__fdiv_rn(a, 448.0f), FLT_MIN);
                w = pack_e4m3x4(__fdiv_rn(v[u].x, sc), __fdiv_rn(v[u].y, sc), __fdiv_rn(v[u].z, sc),
                                __fdiv_rn(v[u].w, sc));
            }
            reinterpret_cast<uint32_t*>(q + t * kTile)[lane] = w;
            if (lane == 0) s[t] = sc;
        }
    }
}

__device__ __forceinline__ uint32_t f16x2_pack(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// Two E4M3 codes (low byte first) times two FP16 factors, rounded once back
// to E4M3 (nearest even, saturating).
__device__ __forceinline__ uint32_t e4m3x2_scale_f16(uint32_t two_codes, uint32_t f16x2) {
    uint32_t h;
    uint16_t in = static_cast<uint16_t>(two_codes), out;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"(in));
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(h) : "r"(h), "r"(f16x2));
    asm("cvt.rn.satfinite.e4m3x2.f16x2 %0, %1;" : "=h"(out) : "r"(h));
    return out;
}

// One CTA per 128x128 tile (row tile i, column tile j).  The tile's 128 row
// scales are staged once in shared memory.  Lane l of every warp owns input
// rows 4l..4l+3 of the tile: it reads their four row scales, the warp
// reduces the tile's largest scale s', and the lane keeps the four
// ratios s_r / s'.  The codes pass through the swizzled shared tile; each
// warp then writes four output rows (input columns) per pass, re-expressing
// the four bytes of each output word with their rows' ratios (decode, multiply,
// one rounding to E4M3; in f16x2 when the whole warp's ratios allow it).  Consecutive CTAs take consecutive row tiles of one column
// tile, so their output rows continue each other in memory (measured on GB300
// at 65536x7168: 0.189 ms, against 0.201 ms with column tiles fastest).

__global__ void __launch_bounds__(256) transpose_rowwise_kernel(const uint8_t* __restrict__ q,
                                                                const float* __restrict__ s,
                                                                int64_t R, int64_t C,
                                                                uint8_t* __restrict__ qt,
                                                                float* __restrict__ st) {
    __shared__ uint32_t tile[kTile * kTile / 4];
    __shared__ float scales[kTile];
    const int64_t ntc = C / kTile, ntr = R / kTile;
    const int64_t i = blockIdx.x % ntr, j = blockIdx.x / ntr;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid < kTile) scales[tid] = __ldg(s + (i * kTile + tid) * ntc + j);

    const uint4* src = reinterpret_cast<const uint4*>(q + (i * kTile) * C + j * kTile);
#pragma unroll
    for (int it = 0; it < 4; ++it) {
        const int idx = it * 256 + tid;                  // 16-byte chunk: row idx>>3, chunk idx&7
        const int r = idx >> 3, w0 = (idx & 7) * 4;
        const uint4 w = __ldcs(src + r * (C / 16) + (idx & 7));
        const int sw = tile_swz(r);
        tile[r * 32 + ((w0 + 0) ^ sw)] = w.x;
        tile[r * 32 + ((w0 + 1) ^ sw)] = w.y;
        tile[r * 32 + ((w0 + 2) ^ sw)] = w.z;
        tile[r * 32 + ((w0 + 3) ^ sw)] = w.w;
    }
    __syncthreads();
    const int r0 = lane * 4;
    float sr[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) sr[k] = scales[r0 + k];
    float smax = fmaxf(fmaxf(sr[0], sr[1]), fmaxf(sr[2], sr[3]));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) smax = fmaxf(smax, __shfl_xor_sync(0xFFFFFFFFu, smax, o));
    float ratio[4];
    // Power-of-two ratios 2^-D with D <= 15: an E4M3 value times 2^-D has its
    // lowest bit at or above 2^-24, so the product is exact in FP16 and the
    // whole re-expression can run as f16x2 (decode, multiply, one rounding).
    bool pow2_small = true;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        ratio[k] = __fdiv_rn(sr[k], smax);
        const uint32_t rb = __float_as_uint(ratio[k]);
        const int d = 127 - int(rb >> 23);
        pow2_small = pow2_small && (rb & 0x7FFFFFu) == 0 && (rb >> 23) != 0 && d >= 0 && d <= 15;
    }
    const bool warp_f16 = __all_sync(0xFFFFFFFFu, pow2_small);
    const uint32_t rr01 = f16x2_pack(ratio[0], ratio[1]);
    const uint32_t rr23 = f16x2_pack(ratio[2], ratio[3]);
    if (tid < kTile) st[(j * kTile + tid) * ntr + i] = smax;

#pragma unroll
    for (int h = 0; h < 4; ++h) {
        const int cg = warp + 8 * h;                     // input columns 4cg..4cg+3
        uint32_t w4[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) w4[k] = tile[(r0 + k) * 32 + (cg ^ tile_swz(r0 + k))];
        uint32_t o[4];
        transpose4x4(w4[0], w4[1], w4[2], w4[3], o[0], o[1], o[2], o[3]);
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
            uint32_t word = o[cc];                       // bytes: rows r0..r0+3 of column 4cg+cc
            if (warp_f16) {
                word = e4m3x2_scale_f16(word, rr01) | (e4m3x2_scale_f16(word >> 16, rr23) << 16);
            } else {
                const float2 a = e4m3x2_to_float2(word);
                const float2 b = e4m3x2_to_float2(word >> 16);
                word = pack_e4m3x4(__fmul_rn(a.x, ratio[0]), __fmul_rn(a.y, ratio[1]),
                                   __fmul_rn(b.x, ratio[2]), __fmul_rn(b.y, ratio[3]));
            }
            const int64_t c = j * kTile + 4 * cg + cc;
            *reinterpret_cast<uint32_t*>(qt + c * R + i * kTile + r0) = word;
        }
    }
}

}  // namespace
}  // namespace fp8z

using namespace fp8z;

extern "C" int fp8z_quantize_rowwise(const float* x, int64_t rows, int64_t cols, int32_t pow2,
                                     uint8_t* q, float* s, void* stream) {
    if (!x || !q || !s || rows < 0 || cols < 0 || (cols % kTile) != 0 || (pow2 != 0 && pow2 != 1))
        return FP8Z_EINVAL;
    if (rows > (INT64_MAX / 4) / (cols > 0 ? cols : 1)) return FP8Z_EINVAL;
    if (!host::aligned(x, 16) || !host::aligned(q, 16) || !host::aligned(s, 4)) return FP8Z_EALIGN;
    const int64_t ntiles = rows * (cols / kTile);
    if (ntiles == 0) return FP8Z_OK;
    int sms = 0;
    const int rc = host::device_sms(&sms);
    if (rc != FP8Z_OK) return rc;
    const int64_t want = (ntiles + 8 * kTilesPerWarp - 1) / (8 * kTilesPerWarp);
    const int64_t cap = int64_t(sms) * 8;
    const unsigned grid = unsigned(want < cap ? want : cap);
    quantize_rowwise_kernel<<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(x, ntiles, pow2, q, s);
    return cudaGetLastError() == cudaSuccess ? FP8Z_OK : FP8Z_ECUDA;
}

extern "C" int fp8z_transpose_rowwise(const uint8_t* q, const float* s, int64_t rows, int64_t cols,
                                      uint8_t* q_t, float* s_t, void* stream) {
    if (!q || !s || !q_t || !s_t || rows < 0 || cols < 0 || rows % kTile || cols % kTile)
        return FP8Z_EINVAL;
    const int64_t ntiles = (rows / kTile) * (cols / kTile);
    if (ntiles > 0x7FFFFFFFLL || rows > (INT64_MAX / 2) / (cols > 0 ? cols : 1)) return FP8Z_EINVAL;
    if (!host::aligned(q, 16) || !host::aligned(q_t, 16) || !host::aligned(s, 4) || !host::aligned(s_t, 4))
        return FP8Z_EALIGN;
    if (ntiles == 0) return FP8Z_OK;
    int sms = 0;
    const int rc = host::device_sms(&sms);
    if (rc != FP8Z_OK) return rc;
    transpose_rowwise_kernel<<<unsigned(ntiles), 256, 0, static_cast<cudaStream_t>(stream)>>>(
        q, s, rows, cols, q_t, s_t);
    return cudaGetLastError() == cudaSuccess ? FP8Z_OK : FP8Z_ECUDA;
}
