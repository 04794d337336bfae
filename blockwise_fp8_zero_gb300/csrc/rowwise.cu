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
// Traffic: quantize 4 B in + 1 B out per element, the transpose 1 B in + 1 B
// out per element (+ 1/32 B of scales each way).  The quantizer runs at the
// HBM bound; the transpose at the pace of its re-expression arithmetic and
// the latency of its staging loads (about 24 instructions per 4-byte output
// word, the ALU pipe near 44 %, DRAM near 76 %).
#include <cfloat>
#include <cstdint>

#include <cuda_runtime.h>

#include "fp8z.h"
#include "fp8z_device.cuh"
#include "fp8z_host.h"

namespace fp8z {
namespace {

constexpr int kTile = FP8Z_BLOCK;         // 128 elements per scale
// Exponent k of the smallest power of two >= amax/448 (exact, from the bits
// of amax > 0), kept in the normal float range [-126, 127]; an infinite amax
// takes the clamp, 127.  448 = 1.75 * 2^8, so with amax = m * 2^e (m in [1, 2))
// the answer is e-8, or e-7 when m > 1.75.
__device__ __forceinline__ int pow2_tile_exponent(float amax) {
    const uint32_t b = __float_as_uint(amax);
    if ((b >> 23) == 255) return 127;     // +Inf (a NaN never becomes the amax)
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
    const int k = e - 8 + (man > 0x600000u ? 1 : 0);     // 0x600000 = 0.75 * 2^23
    return k < -126 ? -126 : (k > 127 ? 127 : k);
}

// 2^k as a float for k in [-127, 127] (2^-127 is subnormal, still exact).
__device__ __forceinline__ float exp2i(int k) {
    return k >= -126 ? __uint_as_float(uint32_t(k + 127) << 23) : __uint_as_float(1u << (k + 149));
}

// Streaming 16-byte load through the non-coherent path with a 256-byte L2
// fetch: the first load of a tile's 128-byte line also brings the next line
// into L2.  On GB300 at 65536x7168 the quantizer ran 0.334 ms with it against
// 0.358 ms with `.cs` loads (.cs or L1::no_allocate with the same 256-byte
// fetch: 0.360 ms).  The input is read-only for the kernel's lifetime.
__device__ __forceinline__ float4 ld_stream_l2_256(const float4* p) {
    float4 r;
    asm volatile("ld.global.nc.L2::256B.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(r.x), "=f"(r.y), "=f"(r.z), "=f"(r.w)
                 : "l"(p));
    return r;
}

// The same load for 16 bytes of codes.
__device__ __forceinline__ uint4 ld_stream_l2_256(const uint4* p) {
    uint4 r;
    asm volatile("ld.global.nc.L2::256B.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

__device__ __forceinline__ float absmax4(float acc, float4 x) {
    return fmaxf(fmaxf(fmaxf(acc, fabsf(x.x)), fmaxf(fabsf(x.y), fabsf(x.z))), fabsf(x.w));
}

// Eight lanes per 128-element tile, so a warp takes four consecutive tiles
// (2 KB of input) at a time: lane j of a tile holds float4s j, j+8, j+16, j+24
// (every load instruction reads whole 128-byte lines), the tile's amax needs
// three shuffles, and the lane writes four 4-byte code words.  Measured on
// GB300 at 65536x7168: 98 % of the copy bandwidth, against 82 % with one warp
// per tile (five shuffles per four elements made that version issue-bound);
// 106 % with the loads' 256-byte L2 fetch (ld_stream_l2_256), the ceiling a
// plain kernel with this 4:1 read:write mix reaches.
__global__ void __launch_bounds__(256) quantize_rowwise_kernel(const float* __restrict__ x,
                                                               int64_t ntiles, int pow2,
                                                               uint8_t* __restrict__ q,
                                                               float* __restrict__ s) {
    const int lane = threadIdx.x & 31, sub = lane >> 3, j = lane & 7;
    const int64_t nwarps = int64_t(gridDim.x) * (blockDim.x >> 5);
    const int64_t nquads = (ntiles + 3) >> 2;
    for (int64_t qd = int64_t(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); qd < nquads;
         qd += nwarps) {
        const int64_t t = qd * 4 + sub;                  // this lane's tile
        const bool valid = t < ntiles;
        float4 v[4];
#pragma unroll
        for (int k = 0; k < 4; ++k)
            v[k] = valid ? ld_stream_l2_256(reinterpret_cast<const float4*>(x + t * kTile) + j + 8 * k)
                         : make_float4(0.f, 0.f, 0.f, 0.f);
        float a = 0.0f;
#pragma unroll
        for (int k = 0; k < 4; ++k) a = absmax4(a, v[k]);
        a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, 1));
        a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, 2));
        a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, 4));
        if (!valid) continue;
        float sc;
        uint32_t w[4];
        if (a == 0.0f || pow2) {
            // a power of two: x/s is exactly x * 2^-k, one multiply instead of a divide
            const int k2 = a == 0.0f ? 0 : pow2_tile_exponent(a);
            sc = exp2i(k2);
            const float r = exp2i(-k2);
#pragma unroll
            for (int k = 0; k < 4; ++k)
                w[k] = pack_e4m3x4(__fmul_rn(v[k].x, r), __fmul_rn(v[k].y, r), __fmul_rn(v[k].z, r),
                                   __fmul_rn(v[k].w, r));
        } else {
            sc = fmaxf(__fdiv_rn(a, 448.0f), FLT_MIN);
#pragma unroll
            for (int k = 0; k < 4; ++k)
                w[k] = pack_e4m3x4(__fdiv_rn(v[k].x, sc), __fdiv_rn(v[k].y, sc), __fdiv_rn(v[k].z, sc),
                                   __fdiv_rn(v[k].w, sc));
        }
        uint32_t* dst = reinterpret_cast<uint32_t*>(q + t * kTile) + j;
#pragma unroll
        for (int k = 0; k < 4; ++k) dst[8 * k] = w[k];
        if (j == 0) s[t] = sc;
    }
}

__device__ __forceinline__ uint32_t f16x2_pack(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// Re-express the bytes of two output words.  pair01 holds the codes of input
// rows 0, 1 of column c (low half) and of column c+1 (high half), pair23 the
// same for rows 2, 3; out_c / out_c1 get the four re-expressed codes of
// columns c and c+1, row 0 in the low byte.  f16x2 path: decode two codes to
// f16x2, multiply by the rows' two ratios, round once to E4M3 (nearest even,
// saturating).
__device__ __forceinline__ void rescale_words_f16(uint32_t pair01, uint32_t pair23, uint32_t rr01,
                                                  uint32_t rr23, uint32_t& out_c, uint32_t& out_c1) {
    asm("{\n\t.reg .b16 a0, a1, b0, b1, o0, o1, o2, o3;\n\t.reg .b32 h;\n\t"
        "mov.b32 {a0, a1}, %2;\n\t"
        "mov.b32 {b0, b1}, %3;\n\t"
        "cvt.rn.f16x2.e4m3x2 h, a0;\n\tmul.rn.f16x2 h, h, %4;\n\tcvt.rn.satfinite.e4m3x2.f16x2 o0, h;\n\t"
        "cvt.rn.f16x2.e4m3x2 h, b0;\n\tmul.rn.f16x2 h, h, %5;\n\tcvt.rn.satfinite.e4m3x2.f16x2 o1, h;\n\t"
        "cvt.rn.f16x2.e4m3x2 h, a1;\n\tmul.rn.f16x2 h, h, %4;\n\tcvt.rn.satfinite.e4m3x2.f16x2 o2, h;\n\t"
        "cvt.rn.f16x2.e4m3x2 h, b1;\n\tmul.rn.f16x2 h, h, %5;\n\tcvt.rn.satfinite.e4m3x2.f16x2 o3, h;\n\t"
        "mov.b32 %0, {o0, o1};\n\t"
        "mov.b32 %1, {o2, o3};\n\t}"
        : "=r"(out_c), "=r"(out_c1)
        : "r"(pair01), "r"(pair23), "r"(rr01), "r"(rr23));
}

// The same in FP32: decode, multiply by the row's ratio, round once to E4M3.
__device__ __forceinline__ void rescale_words_f32(uint32_t pair01, uint32_t pair23, const float (&ratio)[4],
                                                  uint32_t& out_c, uint32_t& out_c1) {
    const float2 a0 = e4m3x2_to_float2(pair01), b0 = e4m3x2_to_float2(pair23);
    const float2 a1 = e4m3x2_to_float2(pair01 >> 16), b1 = e4m3x2_to_float2(pair23 >> 16);
    out_c = pack_e4m3x4(__fmul_rn(a0.x, ratio[0]), __fmul_rn(a0.y, ratio[1]), __fmul_rn(b0.x, ratio[2]),
                        __fmul_rn(b0.y, ratio[3]));
    out_c1 = pack_e4m3x4(__fmul_rn(a1.x, ratio[0]), __fmul_rn(a1.y, ratio[1]), __fmul_rn(b1.x, ratio[2]),
                         __fmul_rn(b1.y, ratio[3]));
}

// The 128 output words of one warp pass set: input columns 4cg..4cg+3
// (cg = warp + 8h) of rows r0..r0+3, read from the swizzled tile, 4x4
// byte-transposed, re-expressed and written to output rows 4cg..4cg+3.  The
// transpose stops after its first byte-permutation stage: each 16-bit half of
// its words is already the pair of codes (rows r0, r0+1 or r0+2, r0+3 of one
// column) that one conversion takes, so the re-expression reads them there and
// its packing of the results is the second stage (0.1589 against 0.1617 ms
// with the full transpose first, at 65536x7168).  The f16x2 / FP32 choice is
// made once per tile, outside these loops.
template <bool kF16>
__device__ __forceinline__ void transpose_tile_words(const uint32_t* tile, int warp, int r0, uint8_t* out,
                                                     int64_t R, uint32_t rr01, uint32_t rr23,
                                                     const float (&ratio)[4]) {
    // The 128-byte pieces land in 128 output rows R bytes apart; keeping them
    // in L2 until the rest of each row's sector arrives saves partial writes.
    const uint64_t keep_in_l2 = l2_evict_last_policy();
#pragma unroll
    for (int h = 0; h < 4; ++h) {
        const int cg = warp + 8 * h;                     // input columns 4cg..4cg+3
        uint32_t w4[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) w4[k] = tile[(r0 + k) * 32 + (cg ^ tile_swz(r0 + k))];
        // rows r0, r0+1 (r0+2, r0+3) of columns 0|1 and of columns 2|3
        const uint32_t p01_c01 = __byte_perm(w4[0], w4[1], 0x5140);
        const uint32_t p01_c23 = __byte_perm(w4[0], w4[1], 0x7362);
        const uint32_t p23_c01 = __byte_perm(w4[2], w4[3], 0x5140);
        const uint32_t p23_c23 = __byte_perm(w4[2], w4[3], 0x7362);
        uint32_t o[4];                                   // o[cc]: rows r0..r0+3 of column 4cg+cc
        if (kF16) {
            rescale_words_f16(p01_c01, p23_c01, rr01, rr23, o[0], o[1]);
            rescale_words_f16(p01_c23, p23_c23, rr01, rr23, o[2], o[3]);
        } else {
            rescale_words_f32(p01_c01, p23_c01, ratio, o[0], o[1]);
            rescale_words_f32(p01_c23, p23_c23, ratio, o[2], o[3]);
        }
        uint8_t* dst = out + int64_t(4 * cg) * R;
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
            store_u32_hint(dst, o[cc], keep_in_l2);
            dst += R;
        }
    }
}

// The ratios of one 128x128 tile (row tile i, column tile j), computed by one
// warp: lane l reads the row scales of input rows 4l..4l+3, the warp reduces
// the tile's largest scale s' (the column-wise scale of all 128 output rows,
// which the warp writes), and the lane keeps the four ratios s_r / s' (IEEE
// divide) in FP32 and as f16x2 pairs.  The f16x2 re-expression is chosen for
// the tile when every ratio is a power of two 2^-D with D <= 15: an E4M3 value
// times such a ratio has its lowest bit at or above 2^-24, so the product is
// exact in FP16 and decode, multiply and one rounding run as f16x2.
struct TileRatios {
    float4 ratio[32];                     // lane l: rows 4l..4l+3
    uint2 f16[32];                        // the same, as two f16x2 pairs
    int use_f16;
};

__device__ __forceinline__ void tile_ratios(const float* s, int64_t i, int64_t j, int64_t ntc, int64_t ntr,
                                            float* st, int lane, TileRatios& out) {
    const int r0 = lane * 4;
    float sr[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) sr[k] = __ldg(s + (i * kTile + r0 + k) * ntc + j);
    float smax = fmaxf(fmaxf(sr[0], sr[1]), fmaxf(sr[2], sr[3]));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) smax = fmaxf(smax, __shfl_xor_sync(0xFFFFFFFFu, smax, o));
    float ratio[4];
    bool pow2_small = true;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        ratio[k] = __fdiv_rn(sr[k], smax);
        const uint32_t rb = __float_as_uint(ratio[k]);
        const int d = 127 - int(rb >> 23);
        pow2_small = pow2_small && (rb & 0x7FFFFFu) == 0 && (rb >> 23) != 0 && d >= 0 && d <= 15;
    }
    const bool use_f16 = __all_sync(0xFFFFFFFFu, pow2_small);
    out.ratio[lane] = make_float4(ratio[0], ratio[1], ratio[2], ratio[3]);
    out.f16[lane] = make_uint2(f16x2_pack(ratio[0], ratio[1]), f16x2_pack(ratio[2], ratio[3]));
    if (lane == 0) out.use_f16 = use_f16;
#pragma unroll
    for (int k = 0; k < 4; ++k) st[(j * kTile + r0 + k) * ntr + i] = smax;
}

// One CTA per strip of kW column tiles of one row tile: the strip's rows are
// read as kW*128 contiguous bytes and staged in swizzled shared tiles while
// warp u computes the ratios of tile u; then each tile is written out
// column-wise by all eight warps, lane l re-expressing the bytes of input
// rows 4l..4l+3 with their ratios, a warp writing 128 contiguous bytes of one
// output row per store.  Consecutive CTAs take consecutive row tiles of one
// strip, so their output rows continue each other in memory.  Measured on
// GB300 at 65536x7168: 0.150 ms with the staging loads' 256-byte L2 fetch
// (ld_stream_l2_256; 0.158 ms with `.cs` loads), three CTAs per SM (80
// registers; with `.cs` loads 0.162
// ms at 64 registers and four CTAs, 0.175 ms at 93 and two; before the
// one-stage transpose, 0.192 ms at 48 registers and five); before that,
// 0.170 against 0.162 ms when all eight warps computed the same ratios (four
// IEEE divides per lane per tile, a fifth of the instructions); 0.166-0.189
// ms with the ratio arithmetic after the staging
// stores (the strided scale loads then sit on the CTA's critical path); 0.189
// ms with one tile per CTA (128-byte reads per row), 0.201 ms with column
// tiles fastest; a persistent variant that moved the tiles with TMA
// (128B-swizzled loads and stores) reached 0.181 ms, and one that prefetched
// the next strip into registers while writing the current one 0.175-0.196 ms
// (two to four CTAs per SM), and one that staged the output words in plain
// shared tiles written by one 2-D TMA tensor store each 0.20-0.26 ms, and
// one that took two row tiles per CTA so that a lane re-expressed eight input
// rows and a warp wrote 256 bytes of an output row per 8-byte store (half the
// store instructions) 0.160-0.229 ms: with one column tile per CTA, four CTAs
// per SM, 0.160 ms; with two, 69 KB of shared tiles per CTA left the SM's
// carveout so little L1 for the staging loads in flight that they throttled
// the memory pipe (0.229 ms at three CTAs per SM, 0.173 ms at two): the
// re-expression arithmetic and the staging
// loads' latency, not the memory system's bandwidth, set the pace.  The tile
// loop stays
// rolled: unrolled, the two copies of both re-expression paths ran 25 %
// slower.  Tiles are kTileWords apart, not 4096, so the two tiles' row writes
// fall on different banks.
constexpr int kTileWords = kTile * kTile / 4 + 2;

template <int kW>
__global__ void __launch_bounds__(256, 3) transpose_rowwise_kernel(const uint8_t* __restrict__ q,
                                                                const float* __restrict__ s,
                                                                int64_t R, int64_t C,
                                                                uint8_t* __restrict__ qt,
                                                                float* __restrict__ st) {
    __shared__ uint32_t tile[kW][kTileWords];
    __shared__ TileRatios ratios[kW];
    const int64_t ntc = C / kTile, ntr = R / kTile;
    const int64_t i = blockIdx.x % ntr, jw = (blockIdx.x / ntr) * kW;   // first column tile of the strip
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    // 16-byte chunks: row r of the strip is 8*kW chunks, chunk ch of tile ch/8
    constexpr int kChunks = kW * 8;
    constexpr int kIters = kTile * kChunks / 256;
    const uint4* src = reinterpret_cast<const uint4*>(q + (i * kTile) * C + jw * kTile);
    uint4 buf[kIters];
#pragma unroll
    for (int it = 0; it < kIters; ++it) {
        const int idx = it * 256 + tid;
        buf[it] = ld_stream_l2_256(src + (idx / kChunks) * (C / 16) + idx % kChunks);
    }
    if (warp < kW) tile_ratios(s, i, jw + warp, ntc, ntr, st, lane, ratios[warp]);
#pragma unroll
    for (int it = 0; it < kIters; ++it) {
        const int idx = it * 256 + tid;
        const int r = idx / kChunks, ch = idx % kChunks;
        const int w0 = (ch & 7) * 4, sw = tile_swz(r);
        uint32_t* row = tile[ch >> 3] + r * 32;
        row[(w0 + 0) ^ sw] = buf[it].x;
        row[(w0 + 1) ^ sw] = buf[it].y;
        row[(w0 + 2) ^ sw] = buf[it].z;
        row[(w0 + 3) ^ sw] = buf[it].w;
    }
    __syncthreads();
    const int r0 = lane * 4;
#pragma unroll 1
    for (int u = 0; u < kW; ++u) {
        const float4 rt = ratios[u].ratio[lane];
        const uint2 rr = ratios[u].f16[lane];
        const float ratio[4] = {rt.x, rt.y, rt.z, rt.w};
        uint8_t* out = qt + ((jw + u) * kTile) * R + i * kTile + r0;
        if (ratios[u].use_f16)
            transpose_tile_words<true>(tile[u], warp, r0, out, R, rr.x, rr.y, ratio);
        else
            transpose_tile_words<false>(tile[u], warp, r0, out, R, rr.x, rr.y, ratio);
    }
}

// ------------------------------------------------------ row-wise dequantize
// "FP8-Flow-MoE" §3.1: D(Q(x)) = Q(x) * s, here decode(q[r][c]) * s[r][c/128]
// in FP32 (the decode is exact, the product rounds once).  The first step of
// the naive way to the column-wise layout (dequantize, transpose, quantize
// again), kept so that path can be run and timed from the library's own
// kernels.  HBM-bound: 1 B read + 4 B written per element.
//
// Row-major output: each thread turns 16 codes (one 16-byte load, which never
// crosses a 128-column tile) into four 16-byte streaming stores.
__global__ void __launch_bounds__(256) dequant_rowwise_kernel(const uint8_t* __restrict__ q,
                                                              const float* __restrict__ s, int64_t nchunks,
                                                              int64_t C, float* __restrict__ x) {
    const int64_t per_row = C / 16, nt = C / kTile;
    const int64_t stride = int64_t(gridDim.x) * blockDim.x;
    for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < nchunks; i += stride) {
        const uint4 w = ld_stream_l2_256(reinterpret_cast<const uint4*>(q) + i);
        const int64_t r = i / per_row, c = (i % per_row) * 16;
        const float sc = __ldg(s + r * nt + c / kTile);
        float4* dst = reinterpret_cast<float4*>(x + r * C + c);
        const uint32_t words[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float2 lo = e4m3x2_to_float2(words[k]), hi = e4m3x2_to_float2(words[k] >> 16);
            __stcs(dst + k, make_float4(__fmul_rn(lo.x, sc), __fmul_rn(lo.y, sc), __fmul_rn(hi.x, sc),
                                        __fmul_rn(hi.y, sc)));
        }
    }
}

// Transposed output, out[c][r] = decode(q[r][c]) * s[r][c/128]: dequantize and
// transpose of the naive path in one pass.  One CTA per 128x128 tile: the
// tile's codes are staged in a swizzled shared tile, then lane l of every warp
// takes input rows 4l..4l+3 (with their four row scales) and, per group of
// four input columns, byte-transposes four words and writes four output rows,
// a warp storing 512 contiguous bytes of one output row.  Consecutive CTAs
// take consecutive row tiles of one column tile, so their output rows continue
// each other in memory.
__global__ void __launch_bounds__(256) dequant_rowwise_t_kernel(const uint8_t* __restrict__ q,
                                                                const float* __restrict__ s, int64_t R,
                                                                int64_t C, float* __restrict__ xt) {
    __shared__ uint32_t tile[kTile * 32];
    const int64_t ntr = R / kTile, ntc = C / kTile;
    const int64_t i = blockIdx.x % ntr, j = blockIdx.x / ntr;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint4* src = reinterpret_cast<const uint4*>(q + (i * kTile) * C + j * kTile);
#pragma unroll
    for (int it = 0; it < 4; ++it) {
        const int idx = it * 256 + tid;                  // 16-byte chunk of the tile
        const int r = idx >> 3, w0 = (idx & 7) * 4, sw = tile_swz(r);
        const uint4 w = ld_stream_l2_256(src + r * (C / 16) + (idx & 7));
        tile[r * 32 + ((w0 + 0) ^ sw)] = w.x;
        tile[r * 32 + ((w0 + 1) ^ sw)] = w.y;
        tile[r * 32 + ((w0 + 2) ^ sw)] = w.z;
        tile[r * 32 + ((w0 + 3) ^ sw)] = w.w;
    }
    const int r0 = lane * 4;
    float sc[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) sc[k] = __ldg(s + (i * kTile + r0 + k) * ntc + j);
    __syncthreads();
#pragma unroll
    for (int h = 0; h < 4; ++h) {
        const int cg = warp + 8 * h;                     // input columns 4cg..4cg+3
        uint32_t w4[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) w4[k] = tile[(r0 + k) * 32 + (cg ^ tile_swz(r0 + k))];
        uint32_t o[4];
        transpose4x4(w4[0], w4[1], w4[2], w4[3], o[0], o[1], o[2], o[3]);
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {                 // output row j*128 + 4cg + cc
            const float2 lo = e4m3x2_to_float2(o[cc]), hi = e4m3x2_to_float2(o[cc] >> 16);
            float4* dst = reinterpret_cast<float4*>(xt + (j * kTile + 4 * cg + cc) * R + i * kTile + r0);
            __stcs(dst, make_float4(__fmul_rn(lo.x, sc[0]), __fmul_rn(lo.y, sc[1]), __fmul_rn(hi.x, sc[2]),
                                    __fmul_rn(hi.y, sc[3])));
        }
    }
}

}  // namespace
}  // namespace fp8z

using namespace fp8z;

extern "C" int fp8z_dequant_rowwise(const uint8_t* q, const float* s, int64_t rows, int64_t cols,
                                    int32_t transpose, float* out, void* stream) {
    const fp8z::host::NvtxRange nvtx_range("fp8z_dequant_rowwise");
    if (!q || !s || !out || rows < 0 || cols < 0 || cols % kTile || (transpose != 0 && transpose != 1))
        return FP8Z_EINVAL;
    if (transpose && rows % kTile) return FP8Z_EINVAL;
    if (rows > (INT64_MAX / 4) / (cols > 0 ? cols : 1)) return FP8Z_EINVAL;
    if (!host::aligned(q, 16) || !host::aligned(out, 16) || !host::aligned(s, 4)) return FP8Z_EALIGN;
    const int64_t n = rows * cols;
    if (n == 0) return FP8Z_OK;
    int sms = 0;
    const int rc = host::device_sms(&sms);
    if (rc != FP8Z_OK) return rc;
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (transpose) {
        const int64_t ntiles = (rows / kTile) * (cols / kTile);
        if (ntiles > 0x7FFFFFFFLL) return FP8Z_EINVAL;
        dequant_rowwise_t_kernel<<<unsigned(ntiles), 256, 0, st>>>(q, s, rows, cols, out);
    } else {
        const int64_t nchunks = n / 16;
        const int64_t want = (nchunks + 255) / 256, cap = int64_t(sms) * 8;
        dequant_rowwise_kernel<<<unsigned(want < cap ? want : cap), 256, 0, st>>>(q, s, nchunks, cols, out);
    }
    return cudaGetLastError() == cudaSuccess ? FP8Z_OK : FP8Z_ECUDA;
}

extern "C" int fp8z_quantize_rowwise(const float* x, int64_t rows, int64_t cols, int32_t pow2,
                                     uint8_t* q, float* s, void* stream) {
    const fp8z::host::NvtxRange nvtx_range("fp8z_quantize_rowwise");
    if (!x || !q || !s || rows < 0 || cols < 0 || (cols % kTile) != 0 || (pow2 != 0 && pow2 != 1))
        return FP8Z_EINVAL;
    if (rows > (INT64_MAX / 4) / (cols > 0 ? cols : 1)) return FP8Z_EINVAL;
    if (!host::aligned(x, 16) || !host::aligned(q, 16) || !host::aligned(s, 4)) return FP8Z_EALIGN;
    const int64_t ntiles = rows * (cols / kTile);
    if (ntiles == 0) return FP8Z_OK;
    int sms = 0, per_sm = 0;
    int rc = host::device_sms(&sms);
    if (rc != FP8Z_OK) return rc;
    rc = host::resident_ctas(reinterpret_cast<const void*>(&quantize_rowwise_kernel),
                             host::kResidentQuantizeRowwise, 256, 0, &per_sm);
    if (rc != FP8Z_OK) return rc;
    const int64_t want = (ntiles + 31) / 32;            // 8 warps x 4 tiles per CTA and pass
    const int64_t cap = int64_t(sms) * per_sm;
    const unsigned grid = unsigned(want < cap ? want : cap);
    quantize_rowwise_kernel<<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(x, ntiles, pow2, q, s);
    return cudaGetLastError() == cudaSuccess ? FP8Z_OK : FP8Z_ECUDA;
}

extern "C" int fp8z_transpose_rowwise(const uint8_t* q, const float* s, int64_t rows, int64_t cols,
                                      uint8_t* q_t, float* s_t, void* stream) {
    const fp8z::host::NvtxRange nvtx_range("fp8z_transpose_rowwise");
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
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    if ((cols / kTile) % 2 == 0)
        transpose_rowwise_kernel<2><<<unsigned(ntiles / 2), 256, 0, st>>>(q, s, rows, cols, q_t, s_t);
    else
        transpose_rowwise_kernel<1><<<unsigned(ntiles), 256, 0, st>>>(q, s, rows, cols, q_t, s_t);
    return cudaGetLastError() == cudaSuccess ? FP8Z_OK : FP8Z_ECUDA;
}
