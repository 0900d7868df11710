// common.h -- host-side helpers shared by the library's translation units.
#pragma once

#include <atomic>
#include <cstdint>
#include <mutex>
#include <cuda_runtime.h>

#include "../../include/moe_combine.h"

namespace nqg {

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Streaming multiprocessors of the current device (cached per device).
int sm_count();

// Routing-build override from moe_tuning_set: 0 automatic, -1 the
// three-kernel path, 1..16 the largest cluster the single-launch path may use.
void set_route_cluster(int v);

// moe_debug_stall's setting: -1, or the ring slots (combine) / token loads
// (dispatch permute) that CTA 0 issues before it stops.
int64_t debug_stall_slots();

// Per device, the dynamic shared memory a kernel has been allowed so far.
struct SmemLimit {
    std::atomic<int> bytes[64];  // static storage: starts at zero
    std::mutex mu;
};

// Lets `kern` use `need` bytes of dynamic shared memory on device `dev`.  The
// attribute is only ever raised, under a lock, so that calls from several host
// threads cannot leave it lower than a launch needs; once it is high enough
// the check is one atomic load.
template <typename Kern>
cudaError_t ensure_dynamic_smem(Kern kern, int dev, int need, SmemLimit &lim)
{
    if (dev < 0 || dev >= 64)
        return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, need);
    if (lim.bytes[dev].load(std::memory_order_acquire) >= need)
        return cudaSuccess;
    std::lock_guard<std::mutex> guard(lim.mu);
    if (lim.bytes[dev].load(std::memory_order_relaxed) >= need)
        return cudaSuccess;
    const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, need);
    if (e == cudaSuccess)
        lim.bytes[dev].store(need, std::memory_order_release);
    return e;
}

// Status of the launches just made: MOE_ERR_CUDA if any failed.
inline moe_status launch_status()
{
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

} // namespace nqg
