// fp8z_host.h -- host-side helpers of the library (argument checks, device
// queries, per-step AdamW scalars).  Internal; not part of the C ABI.
#pragma once

#include <cstdint>

#include <nvtx3/nvToolsExt.h>

#include "fp8z.h"

namespace fp8z {
namespace host {

// A named NVTX range over one library call, so a profiler timeline shows each
// call with the kernels it enqueued.  Header-only NVTX: without an attached
// tool a push/pop pair costs a few nanoseconds.
struct NvtxRange {
    explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
    NvtxRange(const NvtxRange&) = delete;
    NvtxRange& operator=(const NvtxRange&) = delete;
};

// Default limit for every bounded device wait (2 s): far above any legitimate
// wait in a step, far below anything that would look like a hung GPU.
constexpr int64_t kDefaultTimeoutNs = 2000000000LL;

// The limit the next launches take: kDefaultTimeoutNs unless
// fp8z_set_wait_limit_ns changed it (process-wide).
int64_t wait_limit_ns();

inline bool aligned(const void* ptr, uintptr_t a) {
    return (reinterpret_cast<uintptr_t>(ptr) & (a - 1)) == 0;
}

// Scalars of one AdamW step, formed in double from the float hyper-parameters
// and rounded once to float.
struct AdamwScalars {
    float beta1, beta2, omb1, omb2, eps, step_size, rs_bc2, decay, lr_wd;
};

AdamwScalars adamw_scalars(const fp8z_adamw_hparams& hp);
bool hparams_valid(const fp8z_adamw_hparams& hp);

// Smallest power of two >= x (x > 0, finite); 0 for x == 0.
float pow2_at_least(float x);

// SM count of the current device; FP8Z_EUNSUPPORTED unless it is an sm_103
// part (the library is built for sm_103a only).
int device_sms(int* sms);

// cudaFuncSetAttribute(MaxDynamicSharedMemorySize) once per (kernel slot, device).
int set_smem_once(const void* kernel, int slot, int bytes);

// CTAs of `kernel` that fit on one SM at `threads` threads and `smem` bytes
// of dynamic shared memory (at least 1), queried once per (kernel slot,
// device).  Grid-stride kernels launch exactly SMs x this many CTAs: a grid
// that does not fit in one wave leaves its last CTAs running alone.
int resident_ctas(const void* kernel, int slot, int threads, int smem, int* per_sm);
enum ResidentSlot { kResidentQuantizeRowwise = 0, kResidentTransposeTma = 1 };

// The driver's cuTensorMapEncodeTiled (through the runtime's entry-point
// query, so the library needs no link against libcuda); nullptr if absent.
void* tensor_map_encoder();

}  // namespace host
}  // namespace fp8z
