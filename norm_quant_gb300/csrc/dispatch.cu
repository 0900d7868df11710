// dispatch.cu -- the dispatch-side permute: every token's row is copied to
// the expert-grouped rows its routing slots name, the step before the expert
// computation and the inverse of the combine's gather
// (flashinfer.comm.moe_a2a_combine: combine is the inverse of
// moe_a2a_dispatch; Struct_ep_combine_skip_a2a: src_info).
//
// One warp per CTA drives the TMA engine: token rows are bulk-loaded into a
// ring of shared-memory slots (mbarrier completion), and each loaded row is
// bulk-stored straight from its slot to every destination row (one bulk
// group per token).  A slot is refilled only after its stores have finished
// reading it.  Bytes: 2H read per token, 2H written per valid slot.  All
// waits are bounded, like the combine's.
#include <cstdint>
#include <cuda_runtime.h>

#include "common.h"
#include "ptx.cuh"

namespace nqg {
namespace {

constexpr uint64_t kWaitLimitNs = 2000000000ull;
constexpr size_t kDispatchCtaSmem = 50 * 1024;  // at H = 7168: 3 slots, 5 CTAs an SM (88.2 us vs 89.7 at 100 KB)
constexpr int kDispatchMaxSlots = 16;

__device__ __forceinline__ void report(int32_t *status, int32_t code)
{
    if (status)
        atomicCAS(status, 0, code);
}

__global__ void __launch_bounds__(32) dispatch_kernel(const uint8_t *__restrict__ x, int64_t T, int32_t H,
                                                      const int32_t *__restrict__ row_map, int32_t k,
                                                      uint8_t *__restrict__ xg, int64_t n_rows,
                                                      int32_t *__restrict__ status, int32_t S, int64_t stall_after)
{
    extern __shared__ __align__(128) uint8_t smem[];
    const int lane = threadIdx.x;
    const uint32_t row_bytes = static_cast<uint32_t>(H) * 2u;
    const uint32_t row_stride = (row_bytes + 127u) & ~127u;
    const uint32_t ring = smem_u32(smem);
    const uint32_t full0 = ring + static_cast<uint32_t>(S) * row_stride;
    const int64_t G = gridDim.x;
    const int64_t n = (T - blockIdx.x + G - 1) / G;  // tokens of this CTA: blockIdx.x + i * G
    if (lane == 0) {
        for (int s = 0; s < S; ++s)
            mbar_init(full0 + 8u * s, 1);
        fence_mbar_init();
    }
    __syncwarp();
    grid_dependency_wait();  // see the combine kernel: programmatic dependent launch

    // test hook (moe_debug_stall): CTA 0 issues no loads from token stall_after on
    const bool stalls = stall_after >= 0 && blockIdx.x == 0;
    auto load = [&](int64_t i) {  // lane 0 only; false if the hook held it back
        if (stalls && i >= stall_after)
            return false;
        const uint32_t s = static_cast<uint32_t>(i % S);
        mbar_arrive_expect_tx(full0 + 8u * s, row_bytes);
        bulk_g2s(ring + s * row_stride, x + (blockIdx.x + i * G) * row_bytes, row_bytes, full0 + 8u * s);
        return true;
    };
    const int64_t pro = n < S ? n : S;
    int64_t loaded = 0;  // loads issued (lane 0's count)
    if (lane == 0)
        for (int64_t q = 0; q < pro; ++q)
            loaded += load(q) ? 1 : 0;

    int32_t r_next = (n > 0 && lane < k) ? __ldg(row_map + static_cast<int64_t>(blockIdx.x) * k + lane) : -1;
    bool ok = true;
    for (int64_t i = 0; i < n; ++i) {
        const int64_t t = blockIdx.x + i * G;
        const int32_t r = r_next;
        if (i + 1 < n && lane < k)
            r_next = __ldg(row_map + (t + G) * k + lane);
        bool valid = lane < k && r >= 0;
        if (valid && r >= n_rows) {
            report(status, MOE_ERR_ROW_OUT_OF_RANGE);
            valid = false;
        }
        uint32_t m = __ballot_sync(0xffffffffu, valid);
        const uint32_t s = static_cast<uint32_t>(i % S);
        bool good = true;
        if (lane == 0) {
            good = mbar_wait_bounded(full0 + 8u * s, static_cast<uint32_t>((i / S) & 1), kWaitLimitNs);
            if (good)
                fence_proxy_async_smem();
        }
        good = __shfl_sync(0xffffffffu, good, 0);
        if (!good) {
            ok = false;
            break;
        }
        while (m) {
            const int j = __ffs(m) - 1;
            m &= m - 1;
            const int32_t rj = __shfl_sync(0xffffffffu, r, j);
            if (lane == 0)
                bulk_s2g(xg + static_cast<int64_t>(rj) * row_bytes, ring + s * row_stride, row_bytes);
        }
        if (lane == 0) {
            bulk_commit();
            // refill the previous token's slot once its stores have read it
            if (i >= 1 && loaded < n) {
                bulk_wait_read_all_but_one();
                if (load(loaded))
                    ++loaded;
            }
        }
    }
    if (lane == 0) {
        if (!ok) {
            report(status, MOE_ERR_DEVICE_TIMEOUT);
            // let the loads this warp started land before shared memory goes away
            for (int64_t q = loaded - (loaded < S ? loaded : S); q < loaded; ++q)
                mbar_wait_bounded(full0 + 8u * static_cast<uint32_t>(q % S), static_cast<uint32_t>((q / S) & 1),
                                  kWaitLimitNs);
        }
        bulk_wait_all();
    }
}

} // namespace
} // namespace nqg

using namespace nqg;

extern "C" moe_status moe_dispatch_permute(const void *x, int64_t T, int32_t H, const int32_t *row_map,
                                           int32_t top_k, void *x_grouped, int64_t n_rows, int32_t *status,
                                           moe_stream_t stream)
{
    if (T < 0 || H < 8 || H % 8 != 0 || top_k < 1 || n_rows < 0)
        return MOE_ERR_INVALID_ARG;
    if (H > MOE_MAX_HIDDEN || top_k > MOE_MAX_TOP_K)
        return MOE_ERR_UNSUPPORTED;
    if (T == 0)
        return MOE_OK;
    if (!x || !row_map || (n_rows > 0 && !x_grouped))
        return MOE_ERR_INVALID_ARG;
    if (!aligned16(x) || (x_grouped && !aligned16(x_grouped)) || (reinterpret_cast<uintptr_t>(row_map) & 3u) ||
        (reinterpret_cast<uintptr_t>(status) & 3u))
        return MOE_ERR_INVALID_ARG;
    const size_t row_stride = (static_cast<size_t>(H) * 2 + 127) / 128 * 128;
    int S = static_cast<int>(kDispatchCtaSmem / (row_stride + 8));
    S = S < 2 ? 2 : (S > kDispatchMaxSlots ? kDispatchMaxSlots : S);
    const size_t smem = static_cast<size_t>(S) * (row_stride + 8);
    static SmemLimit smem_limit;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return MOE_ERR_CUDA;
    if (ensure_dynamic_smem(dispatch_kernel, dev, static_cast<int>(smem), smem_limit) != cudaSuccess) {
        cudaGetLastError();
        return MOE_ERR_CUDA;
    }
    const int per_sm = static_cast<int>((220 * 1024) / (smem + 1024));
    const int64_t ctas = static_cast<int64_t>(sm_count()) * (per_sm < 1 ? 1 : per_sm);
    if (ctas <= 0)
        return MOE_ERR_CUDA;
    const int grid = static_cast<int>(T < ctas ? T : ctas);
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(32);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = reinterpret_cast<cudaStream_t>(stream);
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, dispatch_kernel, static_cast<const uint8_t *>(x), T, H, row_map, top_k,
                           static_cast<uint8_t *>(x_grouped), n_rows, status, S, debug_stall_slots()) != cudaSuccess) {
        cudaGetLastError();
        return MOE_ERR_CUDA;
    }
    return MOE_OK;
}
