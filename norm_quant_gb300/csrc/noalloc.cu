// noalloc.cu -- the routing build for callers that cannot allocate device
// memory: its scratch lives in a fixed array that the library itself holds.
#include <atomic>
#include <cstdint>
#include <cuda_runtime.h>

#include "common.h"

namespace {

// The routing build's scratch (its error word, then per-chunk histograms),
// held by every GPU that loads the library until the process exits.  In host
// code this name is only a stand-in for the device array: its device address
// comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_route_scratch[MOE_NOALLOC_SCRATCH_BYTES];

// Device address of g_route_scratch on the current device, looked up once per
// device (with that device current); nullptr if the lookup fails.
void *route_scratch_address()
{
    static std::atomic<void *> addr[64];  // static storage: starts null
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return nullptr;
    void *a = addr[dev].load(std::memory_order_acquire);
    if (!a) {
        if (cudaGetSymbolAddress(&a, g_route_scratch) != cudaSuccess) {
            cudaGetLastError();
            return nullptr;
        }
        addr[dev].store(a, std::memory_order_release);  // every thread finds the same address
    }
    return a;
}

} // namespace

extern "C" moe_status moe_build_row_map_noalloc(const int32_t *topk_ids, int64_t T, int32_t top_k, int32_t E,
                                                int32_t *counts, int32_t *offsets, int32_t *row_map,
                                                int32_t *src_row, int32_t *error_flag, moe_stream_t stream)
{
    size_t need = 0;
    const moe_status st = moe_build_row_map_workspace_size(T, top_k, E, &need);
    if (st != MOE_OK)
        return st;
    if (need > MOE_NOALLOC_SCRATCH_BYTES)
        return MOE_ERR_UNSUPPORTED;  // the fixed scratch is too small for this T * top_k and E
    if (reinterpret_cast<uintptr_t>(error_flag) & 3u)
        return MOE_ERR_INVALID_ARG;
    void *scratch = route_scratch_address();
    if (!scratch)
        return MOE_ERR_CUDA;
    // the build clears the error word itself and writes every histogram
    // entry before reading it, so nothing left by an earlier call leaks in
    const moe_status r = moe_build_row_map(topk_ids, T, top_k, E, counts, offsets, row_map, src_row, scratch,
                                           MOE_NOALLOC_SCRATCH_BYTES, stream);
    if (r != MOE_OK || !error_flag)
        return r;
    // the error word is the scratch's first int32 (as moe_build_row_map_check reads it)
    if (cudaMemcpyAsync(error_flag, scratch, sizeof(int32_t), cudaMemcpyDeviceToDevice,
                        reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
        return MOE_ERR_CUDA;
    return MOE_OK;
}
