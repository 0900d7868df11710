// api.cu -- small C entry points: version, status names, ABI size check,
// scale-matrix sizes; and the per-device SM count used for grid sizing.
#include <atomic>
#include <cstdint>
#include <cuda_runtime.h>

#include "common.h"

namespace nqg {

int sm_count()
{
    static std::atomic<int> cache[64];  // 0 = not yet queried
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return 0;
    if (dev >= 0 && dev < 64) {
        const int c = cache[dev].load(std::memory_order_relaxed);
        if (c > 0)
            return c;
    }
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return 0;
    if (dev >= 0 && dev < 64)
        cache[dev].store(n, std::memory_order_relaxed);
    return n;
}

} // namespace nqg

extern "C" int moe_abi_version(void) { return MOE_ABI_VERSION; }

extern "C" size_t moe_combine_args_size(void) { return sizeof(moe_combine_args); }

extern "C" const char *moe_status_string(int status)
{
    switch (status) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG: invalid argument";
    case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED: outside this library's limits";
    case MOE_ERR_WORKSPACE: return "MOE_ERR_WORKSPACE: workspace missing or too small";
    case MOE_ERR_INVALID_EXPERT: return "MOE_ERR_INVALID_EXPERT: a topk id outside [-1, E)";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA: a CUDA call failed";
    case MOE_ERR_ROW_OUT_OF_RANGE: return "MOE_ERR_ROW_OUT_OF_RANGE: a row_map entry >= n_expert_rows";
    case MOE_ERR_DEVICE_TIMEOUT: return "MOE_ERR_DEVICE_TIMEOUT: a bounded device wait gave up";
    default: return "unknown moe_status";
    }
}

extern "C" moe_status moe_scales_bytes(int64_t T, int32_t H, int32_t quant, int32_t sf_layout, size_t *bytes)
{
    if (!bytes || T < 0 || H < 1)
        return MOE_ERR_INVALID_ARG;
    int64_t vec;
    if (quant == MOE_QUANT_MXFP8 || quant == MOE_QUANT_MXFP4)
        vec = 32;
    else if (quant == MOE_QUANT_NVFP4)
        vec = 16;
    else
        return MOE_ERR_INVALID_ARG;
    if (H % vec != 0)
        return MOE_ERR_INVALID_ARG;
    const int64_t C = H / vec;
    if (sf_layout == MOE_SF_LINEAR)
        *bytes = static_cast<size_t>(T * C);
    else if (sf_layout == MOE_SF_SWIZZLED_128x4)
        *bytes = static_cast<size_t>((T + 127) / 128 * 128 * ((C + 3) / 4 * 4));
    else
        return MOE_ERR_INVALID_ARG;
    return MOE_OK;
}
