// Exhaustive check of rsqrt_newton (the combine's RMSNorm scale 1/sqrt(m))
// against the correctly rounded __frsqrt_rn, on every positive normal fp32
// value, plus the values outside that range.  Counts: results that differ in
// any bit, results more than one ulp away, values checked; and flags the
// special inputs that do not give what 1/sqrt gives (0 -> inf, inf -> 0).
#include <cstdint>
#include <cuda_runtime.h>

#include "ptx.cuh"

__global__ void rsqrt_check_kernel(unsigned long long *out)  // [differ, beyond one ulp, checked, specials wrong]
{
    const uint32_t first = 0x00800000u, last = 0x7F7FFFFFu;  // the positive normal floats
    unsigned long long differ = 0, far = 0, n = 0;
    for (uint64_t b = first + static_cast<uint64_t>(blockIdx.x) * blockDim.x + threadIdx.x; b <= last;
         b += static_cast<uint64_t>(gridDim.x) * blockDim.x) {
        const float m = __uint_as_float(static_cast<uint32_t>(b));
        const uint32_t got = __float_as_uint(nqg::rsqrt_newton(m)), want = __float_as_uint(__frsqrt_rn(m));
        differ += got != want;
        far += (got > want ? got - want : want - got) > 1u;  // positive floats: ulps = bit distance
        ++n;
    }
    atomicAdd(out + 0, differ);
    atomicAdd(out + 1, far);
    atomicAdd(out + 2, n);
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        unsigned long long bad = 0;
        bad += !(nqg::rsqrt_newton(0.0f) == __int_as_float(0x7F800000));
        bad += !(nqg::rsqrt_newton(__int_as_float(0x7F800000)) == 0.0f);
        const float sub = __uint_as_float(0x00400000u);  // a subnormal: 2^-127
        bad += !(nqg::rsqrt_newton(sub) > 0.0f && nqg::rsqrt_newton(sub) < __int_as_float(0x7F800000));
        atomicAdd(out + 3, bad);
    }
}

extern "C" int rsqrt_check(unsigned long long *host_result)  // 4 counters, as above
{
    unsigned long long *d = nullptr;
    if (cudaMalloc(&d, 4 * sizeof(unsigned long long)) != cudaSuccess)
        return 1;
    cudaMemset(d, 0, 4 * sizeof(unsigned long long));
    rsqrt_check_kernel<<<1024, 256>>>(d);
    const cudaError_t e = cudaMemcpy(host_result, d, 4 * sizeof(unsigned long long), cudaMemcpyDeviceToHost);
    cudaFree(d);
    return e == cudaSuccess ? 0 : 2;
}
