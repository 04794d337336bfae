// fp8z_device.cuh -- sm_103a building blocks shared by the library's kernels:
// mbarrier and bulk-copy (TMA engine) wrappers, a bounded wait, and the
// float32 <-> E4M3 conversions.  Inline PTX only; no CUTLASS.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "fp8z.h"

namespace fp8z {

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Make barrier initialisation visible to the async (bulk-copy) proxy.
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

// True once the phase with the given parity has completed.  The instruction
// itself may suspend the thread for a short, hardware-defined time.
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred P;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 P, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, P;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    return done != 0;
}

// The same test without suspending the thread at all: true once the phase
// with the given parity has completed, false at once otherwise.
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred P;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 P, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, P;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    return done != 0;
}

// Below this limit a bounded wait polls with mbar_test_wait and measures the
// wait in SM clock cycles (two per nanosecond: about the limit at the 2.07
// GHz top clock, longer at lower clocks) instead of suspending in try_wait
// and reading the global timer: a copy that lands within the hardware's own
// suspend window, or within one tick of the global timer, would otherwise
// never let a short limit be checked.  Limits this short are set only to
// exercise the abort paths (fp8z_set_wait_limit_ns).
constexpr int64_t kPolledWaitBelowNs = 1000000;

// Shared state for the bounded waits of one CTA.
struct Watchdog {
    volatile int* abort_flag;   // shared: set once any wait of the CTA gave up
    int32_t* dev_status;        // global, nullable
    int64_t timeout_ns;
};

__device__ __forceinline__ void report_status(int32_t* dev_status, int32_t code) {
    if (dev_status) atomicCAS(dev_status, 0, code);
}

// Wait for `parity` on `bar`, for at most wd.timeout_ns nanoseconds.  Returns
// false (after raising the CTA's abort flag and reporting FP8Z_ETIMEOUT) when
// the limit is reached, or when another thread of the CTA has already
// aborted.  Never spins without a limit.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, const Watchdog& wd) {
    if (wd.timeout_ns < kPolledWaitBelowNs) {
        const long long c0 = clock64();
        while (true) {
            if (mbar_test_wait(bar, parity)) return true;
            if (*wd.abort_flag) return false;
            if (clock64() - c0 > 2 * wd.timeout_ns) {
                *wd.abort_flag = 1;
                report_status(wd.dev_status, FP8Z_ETIMEOUT);
                return false;
            }
        }
    }
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*wd.abort_flag) return false;
        if (global_timer_ns() - t0 > static_cast<uint64_t>(wd.timeout_ns)) {
            *wd.abort_flag = 1;
            report_status(wd.dev_status, FP8Z_ETIMEOUT);
            return false;
        }
    }
}

// Limit for the waits of an abort path: a CTA that gave up still lets every
// bulk copy it issued land before it exits, so the copy engine never writes
// shared memory the CTA no longer owns.  A copy from a valid address always
// completes, so this limit is far above any real wait, and it is separate from
// the normal limit: a short normal limit never shortens a drain.
constexpr int64_t kDrainLimitNs = 20000000000LL;   // 20 s

// Wait for `parity` on `bar` on an abort path: ignores the CTA's abort flag,
// gives up only after kDrainLimitNs (reporting FP8Z_ETIMEOUT).
__device__ __forceinline__ bool mbar_wait_drain(uint32_t bar, uint32_t parity, int32_t* dev_status) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (global_timer_ns() - t0 > static_cast<uint64_t>(kDrainLimitNs)) {
            report_status(dev_status, FP8Z_ETIMEOUT);
            return false;
        }
    }
}

// ------------------------------------------------------------ bulk copies
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

__device__ __forceinline__ uint64_t l2_evict_last_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// 4-byte global store carrying an L2 eviction policy.
__device__ __forceinline__ void store_u32_hint(void* dst, uint32_t x, uint64_t pol) {
    asm volatile("st.global.L2::cache_hint.b32 [%0], %1, %2;" ::"l"(dst), "r"(x), "l"(pol) : "memory");
}

// Global -> shared bulk copy on the TMA engine; completion is counted as
// transaction bytes on `bar`.  dst, src 16-byte aligned, bytes % 16 == 0.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar), "l"(policy)
        : "memory");
}

// The same copy without an L2 cache hint.
__device__ __forceinline__ void bulk_g2s_nohint(uint32_t dst, const void* src, uint32_t bytes,
                                                uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

// A tensor map kept in global memory and written there by a host copy must be
// acquired into the tensor-map proxy before the copy engine uses it (system
// scope: the writer was the host).  Once per map per thread is enough.
__device__ __forceinline__ void tensormap_acquire(const void* map) {
    asm volatile("fence.proxy.tensormap::generic.acquire.sys [%0], 128;" ::"l"(map) : "memory");
}

// Tiled 3-D tensor-map load into shared memory (x innermost; x * element size
// must be a multiple of 16 bytes; out-of-range elements read as zero).
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int x, int y, int z,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
        "l"(map), "r"(x), "r"(y), "r"(z), "r"(bar)
        : "memory");
}

// Tiled 2-D tensor-map load into shared memory (same rules as the 3-D one).
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(map), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

// ------------------------------------------------------- bulk stores out
// Shared -> global copies by the TMA engine, tracked in per-thread bulk
// groups: commit after issuing, then wait before the shared source is reused
// (the .read form returns once the engine has read the source).  Before the
// copy, generic-proxy writes of the source must be fenced into the async proxy.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, int x, int y, int z, uint32_t src) {
    asm volatile(
        "cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%1, %2, %3}], [%4];" ::"l"(map),
        "r"(x), "r"(y), "r"(z), "r"(src)
        : "memory");
}

__device__ __forceinline__ void bulk_s2g(void* dst, uint32_t src, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(src),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// Wait until at most N bulk groups of this thread still read shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ void fence_proxy_async() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Byte offset of (row r, byte b) in a tile of 128-byte rows that a tensor map
// with CU_TENSOR_MAP_SWIZZLE_128B loads or stores (tile 1024-byte aligned):
// the 16-byte chunk index is XORed with r mod 8.
__device__ __forceinline__ int swz128(int r, int b) {
    return r * 128 + ((((b >> 4) ^ (r & 7)) << 4) | (b & 15));
}

// ------------------------------------------------------------- E4M3 cast
// Two floats -> two E4M3 codes, round to nearest even, saturating to ±448
// (NaN stays NaN).  `lo` lands in the low byte.
__device__ __forceinline__ uint32_t cvt_e4m3x2(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ uint32_t pack_e4m3x4(float a, float b, float c, float d) {
    return cvt_e4m3x2(a, b) | (cvt_e4m3x2(c, d) << 16);
}

// Two E4M3 codes (low byte first) -> two exact float values.
__device__ __forceinline__ float2 e4m3x2_to_float2(uint32_t two_codes) {
    uint32_t h2;
    uint16_t in = static_cast<uint16_t>(two_codes);
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(in));
    float lo, hi;
    uint16_t hlo = static_cast<uint16_t>(h2), hhi = static_cast<uint16_t>(h2 >> 16);
    asm("cvt.f32.f16 %0, %1;" : "=f"(lo) : "h"(hlo));
    asm("cvt.f32.f16 %0, %1;" : "=f"(hi) : "h"(hhi));
    return make_float2(lo, hi);
}

// ------------------------------------------------------ transposition tile
// A 128x128 byte tile kept as 128 rows x 32 words in shared memory.  Word w of
// row r is stored at r*32 + (w ^ swz(r)): a warp writing one row, a warp
// writing four rows of eight 16-byte chunks, and a warp reading word w of rows
// 4j+i (j = lane) all hit 32 distinct banks.
__device__ __forceinline__ int tile_swz(int r) { return ((r >> 2) & 31) ^ (r & 3); }

// 4x4 byte transpose: in word i holds bytes (row i, cols 0..3); out word c
// holds bytes (rows 0..3, col c).
__device__ __forceinline__ void transpose4x4(uint32_t w0, uint32_t w1, uint32_t w2, uint32_t w3,
                                             uint32_t& o0, uint32_t& o1, uint32_t& o2,
                                             uint32_t& o3) {
    const uint32_t a_lo = __byte_perm(w0, w1, 0x5140);   // w0.b0 w1.b0 w0.b1 w1.b1
    const uint32_t a_hi = __byte_perm(w0, w1, 0x7362);   // w0.b2 w1.b2 w0.b3 w1.b3
    const uint32_t b_lo = __byte_perm(w2, w3, 0x5140);
    const uint32_t b_hi = __byte_perm(w2, w3, 0x7362);
    o0 = __byte_perm(a_lo, b_lo, 0x5410);
    o1 = __byte_perm(a_lo, b_lo, 0x7632);
    o2 = __byte_perm(a_hi, b_hi, 0x5410);
    o3 = __byte_perm(a_hi, b_hi, 0x7632);
}

}  // namespace fp8z
