// noalloc.cu -- the routing build for callers that cannot allocate device
// memory: its scratch lives in a fixed array that the library itself holds.
#include <cstdint>
#include <mutex>

#include <cuda.h>  // CUcontext and CUresult types only; no libcuda symbol is linked
#include <cuda_runtime.h>

#include "common.h"

namespace {

// The routing build's scratch (its error word, then per-chunk histograms),
// held by every GPU that loads the library until the process exits.  In host
// code this name is only a stand-in for the device array: its device address
// comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_route_scratch[MOE_NOALLOC_SCRATCH_BYTES];

// The current CUDA context's process-unique id (cuCtxGetId), or 0 when no
// context is current or the driver cannot say.  The driver functions come
// through the runtime's entry-point query, so the library links no libcuda.
unsigned long long current_context_id()
{
    using get_current_fn = CUresult (*)(CUcontext *);
    using get_id_fn = CUresult (*)(CUcontext, unsigned long long *);
    static get_current_fn get_current = nullptr;
    static get_id_fn get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<get_current_fn>(f);
        f = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<get_id_fn>(f);
        cudaGetLastError();
    });
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS)
        return 0;
    return id;
}

// Device address of g_route_scratch in the current context, looked up with
// cudaGetSymbolAddress the first time a context asks and remembered under the
// context's id: a context made after cudaDeviceReset, or a caller's own
// driver-API context, gets its own lookup instead of an address that belongs
// to another context.  nullptr if the lookup fails.
void *route_scratch_address()
{
    struct Entry {
        unsigned long long ctx;
        void *addr;
    };
    static Entry cache[64];  // static storage: starts empty
    static int used = 0;
    static std::mutex mu;
    unsigned long long id = current_context_id();
    if (id) {
        std::lock_guard<std::mutex> lock(mu);
        for (int i = 0; i < used; ++i)
            if (cache[i].ctx == id)
                return cache[i].addr;
    }
    void *a = nullptr;
    if (cudaGetSymbolAddress(&a, g_route_scratch) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    if (!id)
        id = current_context_id();  // the lookup made the device's primary context current
    if (id) {
        std::lock_guard<std::mutex> lock(mu);
        if (used < 64)
            cache[used++] = Entry{id, a};  // a full table only means later lookups repeat
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
