// aux.cu -- dequantize, standalone column-major transpose, the E4M3 cast on
// its own, and the watchdog self-test (sm_103a).
#include <cstdint>

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
// HBM-bound (1 B read + 4 B written per element).  Each thread takes one
// 32-bit word of codes (4 elements) per step, so a warp reads 128 contiguous
// bytes of codes and writes 512 contiguous bytes of floats per instruction;
// eight independent words per iteration keep loads in flight (with four the
// kernel stalled on load latency: 71 % of DRAM peak).
__global__ void __launch_bounds__(256) dequant_kernel(const uint32_t* __restrict__ q,
                                                      const float* __restrict__ inv,
                                                      int64_t nwords, float4* __restrict__ out) {
    const int64_t stride = int64_t(gridDim.x) * blockDim.x;
    constexpr int kU = 8;
    for (int64_t w0 = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; w0 < nwords; w0 += kU * stride) {
        uint32_t words[kU];
        float s[kU];
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            const int64_t w = w0 + u * stride;
            words[u] = w < nwords ? __ldcs(q + w) : 0u;
            s[u] = w < nwords ? __ldg(inv + (w >> 12)) : 0.0f;   // 4096 words per block
        }
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            const int64_t w = w0 + u * stride;
            if (w >= nwords) break;
            const float2 a = e4m3x2_to_float2(words[u]);
            const float2 b = e4m3x2_to_float2(words[u] >> 16);
            __stcs(out + w, make_float4(__fmul_rn(a.x, s[u]), __fmul_rn(a.y, s[u]),
                                        __fmul_rn(b.x, s[u]), __fmul_rn(b.y, s[u])));
        }
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
                            void* stream) {
    if (!w_fp8 || !inv_scale || !out || nblk < 0) return FP8Z_EINVAL;
    if (nblk > (INT64_MAX / kBlkElems) / 4) return FP8Z_EINVAL;
    if (!host::aligned(w_fp8, 16) || !host::aligned(out, 16) || !host::aligned(inv_scale, 4))
        return FP8Z_EALIGN;
    if (nblk == 0) return FP8Z_OK;
    int sms = 0, per_sm = 0;
    int rc = host::device_sms(&sms);
    if (rc != FP8Z_OK) return rc;
    rc = host::resident_ctas(reinterpret_cast<const void*>(&dequant_kernel), host::kResidentDequant, 256, 0,
                             &per_sm);
    if (rc != FP8Z_OK) return rc;
    const int64_t nwords = nblk * (kBlkElems / 4);
    const int64_t want = (nwords + 2047) / 2048;
    const int64_t cap = int64_t(sms) * per_sm;      // one wave: 8 per SM would be 1.3 waves (+3.5 %)
    const unsigned grid = unsigned(want < cap ? want : cap);
    dequant_kernel<<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(
        reinterpret_cast<const uint32_t*>(w_fp8), inv_scale, nwords, reinterpret_cast<float4*>(out));
    return cudaGetLastError() == cudaSuccess ? FP8Z_OK : FP8Z_ECUDA;
}

extern "C" int fp8z_transpose_fp8(const uint8_t* w_fp8, const float* inv_scale,
                                  const fp8z_param_entry* entry, uint8_t* out, float* inv_scale_t,
                                  void* stream) {
    if (!w_fp8 || !inv_scale || !entry || !out || !inv_scale_t) return FP8Z_EINVAL;
    const fp8z_param_entry& pe = *entry;
    if (pe.e < 1 || pe.rows < 1 || pe.cols < 1 || pe.blk_offset < 0) return FP8Z_EINVAL;
    if (pe.hb != (pe.rows + kBlk - 1) / kBlk || pe.wb != (pe.cols + kBlk - 1) / kBlk)
        return FP8Z_EINVAL;
    const int64_t nb = pe.e * pe.hb * pe.wb;
    if (nb > 0x7FFFFFFFLL) return FP8Z_EINVAL;
    if (!host::aligned(w_fp8, 16) || !host::aligned(out, 16) || !host::aligned(inv_scale, 4) ||
        !host::aligned(inv_scale_t, 4))
        return FP8Z_EALIGN;
    int sms = 0;
    const int rc = host::device_sms(&sms);
    if (rc != FP8Z_OK) return rc;
    TransposeArgs T;
    T.q = w_fp8 + pe.blk_offset * kBlkElems;
    T.inv = inv_scale + pe.blk_offset;
    T.out = out;
    T.inv_t = inv_scale_t;
    T.H = pe.rows;
    T.W = pe.cols;
    T.hb = pe.hb;
    T.wb = pe.wb;
    transpose_kernel<<<unsigned(nb), 256, 0, static_cast<cudaStream_t>(stream)>>>(T);
    return cudaGetLastError() == cudaSuccess ? FP8Z_OK : FP8Z_ECUDA;
}

extern "C" int fp8z_e4m3_encode_bits(uint32_t first_bits, int64_t n, uint8_t* out, void* stream) {
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
    if (!dev_status || timeout_ns < 0 || timeout_ns > 10000000000LL) return FP8Z_EINVAL;
    if (!host::aligned(dev_status, 4)) return FP8Z_EALIGN;
    int sms = 0;
    const int rc = host::device_sms(&sms);
    if (rc != FP8Z_OK) return rc;
    watchdog_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(dev_status, timeout_ns);
    return cudaGetLastError() == cudaSuccess ? FP8Z_OK : FP8Z_ECUDA;
}
