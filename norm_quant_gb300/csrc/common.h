// common.h -- host-side helpers shared by the library's translation units.
#pragma once

#include <cstdint>
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

// Status of the launches just made: MOE_ERR_CUDA if any failed.
inline moe_status launch_status()
{
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

} // namespace nqg
