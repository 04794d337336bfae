// host.cpp -- argument checks, device queries and AdamW scalars for the C ABI.
// Compiled with -ffp-contract=off: the scalars must round exactly as written.
#include <atomic>
#include <cmath>
#include <cfloat>

#include <cuda_runtime.h>

#include "fp8z.h"
#include "fp8z_host.h"

namespace fp8z {
namespace host {

// Bias-corrected AdamW scalars (lpnh.cn "Model-Optimizer" article §4.3:
// step_size = lr / (1 - beta1^t), denominator sqrt(v)/sqrt(1 - beta2^t) + eps).
AdamwScalars adamw_scalars(const fp8z_adamw_hparams& hp) {
    const double lr = hp.lr, b1 = hp.beta1, b2 = hp.beta2, wd = hp.weight_decay;
    const double t = static_cast<double>(hp.step);
    const double c1 = 1.0 - std::pow(b1, t);
    const double c2 = 1.0 - std::pow(b2, t);
    AdamwScalars s;
    s.beta1 = hp.beta1;
    s.beta2 = hp.beta2;
    s.omb1 = static_cast<float>(1.0 - b1);
    s.omb2 = static_cast<float>(1.0 - b2);
    s.eps = hp.eps;
    s.step_size = static_cast<float>(lr / c1);
    s.rs_bc2 = static_cast<float>(1.0 / std::sqrt(c2));
    const double lr_wd = lr * wd;
    s.decay = static_cast<float>(1.0 - lr_wd);
    s.lr_wd = static_cast<float>(lr_wd);
    return s;
}

bool hparams_valid(const fp8z_adamw_hparams& hp) {
    auto fin = [](float x) { return std::isfinite(x); };
    if (!fin(hp.lr) || hp.lr < 0.0f) return false;
    if (!fin(hp.beta1) || hp.beta1 < 0.0f || hp.beta1 >= 1.0f) return false;
    if (!fin(hp.beta2) || hp.beta2 < 0.0f || hp.beta2 >= 1.0f) return false;
    if (!fin(hp.eps) || hp.eps <= 0.0f) return false;
    if (!fin(hp.weight_decay) || hp.weight_decay < 0.0f) return false;
    if (hp.step < 1) return false;
    if (!(hp.fp8_max > 0.0f && hp.fp8_max <= 448.0f && hp.fp8_max >= FLT_MIN)) return false;
    if (!fin(hp.min_scale) || hp.min_scale < 0.0f) return false;
    if (hp.scale_mode != FP8Z_SCALE_EXACT && hp.scale_mode != FP8Z_SCALE_POW2) return false;
    if (hp.decay_mode != FP8Z_DECAY_PRE && hp.decay_mode != FP8Z_DECAY_POST) return false;
    return true;
}

float pow2_at_least(float x) {
    if (!(x > 0.0f)) return 0.0f;
    int e = 0;
    const double f = std::frexp(static_cast<double>(x), &e);   // x = f * 2^e, f in [0.5, 1)
    const double r = (f == 0.5) ? std::ldexp(1.0, e - 1) : std::ldexp(1.0, e);
    return static_cast<float>(r);
}

int device_sms(int* sms) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return FP8Z_ECUDA;
    int major = 0, minor = 0, n = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return FP8Z_ECUDA;
    if (major != 10 || minor != 3) return FP8Z_EUNSUPPORTED;
    *sms = n;
    return FP8Z_OK;
}

namespace {
std::atomic<int64_t> g_wait_limit_ns{kDefaultTimeoutNs};
}  // namespace

int64_t wait_limit_ns() { return g_wait_limit_ns.load(std::memory_order_relaxed); }

namespace {
constexpr int kMaxDevices = 64;
constexpr int kMaxSlots = 12;
std::atomic<int> g_smem_done[kMaxSlots][kMaxDevices];
}  // namespace

int set_smem_once(const void* kernel, int slot, int bytes) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return FP8Z_ECUDA;
    const bool cacheable = dev >= 0 && dev < kMaxDevices && slot >= 0 && slot < kMaxSlots;
    if (cacheable && g_smem_done[slot][dev].load(std::memory_order_acquire) == bytes)
        return FP8Z_OK;
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) !=
        cudaSuccess)
        return FP8Z_ECUDA;
    if (cacheable) g_smem_done[slot][dev].store(bytes, std::memory_order_release);
    return FP8Z_OK;
}

namespace {
std::atomic<int> g_resident[kMaxSlots][kMaxDevices];
}  // namespace

int resident_ctas(const void* kernel, int slot, int threads, int smem, int* per_sm) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return FP8Z_ECUDA;
    const bool cacheable = dev >= 0 && dev < kMaxDevices && slot >= 0 && slot < kMaxSlots;
    int n = cacheable ? g_resident[slot][dev].load(std::memory_order_acquire) : 0;
    if (n == 0) {
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, threads, size_t(smem)) != cudaSuccess)
            return FP8Z_ECUDA;
        if (n < 1) n = 1;
        if (cacheable) g_resident[slot][dev].store(n, std::memory_order_release);
    }
    *per_sm = n;
    return FP8Z_OK;
}

void* tensor_map_encoder() {
    static std::atomic<void*> fn{nullptr};
    void* f = fn.load(std::memory_order_acquire);
    if (!f) {
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        fn.store(f, std::memory_order_release);
    }
    return f;
}

}  // namespace host
}  // namespace fp8z

extern "C" int fp8z_set_wait_limit_ns(int64_t ns) {
    if (ns < 0 || ns > 10000000000LL) return FP8Z_EINVAL;
    fp8z::host::g_wait_limit_ns.store(ns == 0 ? fp8z::host::kDefaultTimeoutNs : ns,
                                      std::memory_order_relaxed);
    return FP8Z_OK;
}

extern "C" int64_t fp8z_get_wait_limit_ns(void) { return fp8z::host::wait_limit_ns(); }

extern "C" const char* fp8z_status_string(int status) {
    switch (status) {
        case FP8Z_OK: return "FP8Z_OK";
        case FP8Z_EINVAL: return "FP8Z_EINVAL: invalid argument";
        case FP8Z_EALIGN: return "FP8Z_EALIGN: pointer not aligned";
        case FP8Z_ENOSPACE: return "FP8Z_ENOSPACE: range exceeds capacity";
        case FP8Z_ECUDA: return "FP8Z_ECUDA: CUDA runtime or launch error";
        case FP8Z_ETIMEOUT: return "FP8Z_ETIMEOUT: bounded device wait ran out of time";
        case FP8Z_EUNSUPPORTED: return "FP8Z_EUNSUPPORTED: needs an sm_103 (GB300) device";
        default: return "FP8Z: unknown status";
    }
}
