// Exhaustive check of div6_rn (the combine's NVFP4 block-scale quotient)
// against the correctly rounded division, on every finite non-negative fp32
// value.  Counts, over all inputs: results that differ in any bit where the
// correctly rounded quotient is a normal float; results that differ in any
// bit where it is subnormal; and e4m3 codes (the block scale the kernel
// keeps) that differ anywhere.
#include <cstdint>
#include <cuda_runtime.h>

#include "ptx.cuh"

__global__ void div6_check_kernel(unsigned long long *out)  // [normal, subnormal, codes, checked]
{
    const uint32_t last = 0x7F7FFFFFu;  // the largest finite float
    unsigned long long bad_normal = 0, bad_sub = 0, bad_code = 0, n = 0;
    for (uint64_t b = static_cast<uint64_t>(blockIdx.x) * blockDim.x + threadIdx.x; b <= last;
         b += static_cast<uint64_t>(gridDim.x) * blockDim.x) {
        const float x = __uint_as_float(static_cast<uint32_t>(b));
        const float mine = nqg::div6_rn(x), ref = __fdiv_rn(x, 6.0f);
        if (__float_as_uint(mine) != __float_as_uint(ref)) {
            if (ref >= 0x1p-126f)
                ++bad_normal;
            else
                ++bad_sub;
        }
        bad_code += (nqg::cvt_e4m3x2(mine, 0.f) & 0xFFu) != (nqg::cvt_e4m3x2(ref, 0.f) & 0xFFu);
        ++n;
    }
    atomicAdd(out + 0, bad_normal);
    atomicAdd(out + 1, bad_sub);
    atomicAdd(out + 2, bad_code);
    atomicAdd(out + 3, n);
}

extern "C" int div6_check(unsigned long long *host_result)  // 4 counters, as above
{
    unsigned long long *d = nullptr;
    if (cudaMalloc(&d, 4 * sizeof(unsigned long long)) != cudaSuccess)
        return 1;
    cudaMemset(d, 0, 4 * sizeof(unsigned long long));
    div6_check_kernel<<<1024, 256>>>(d);
    const cudaError_t e = cudaMemcpy(host_result, d, 4 * sizeof(unsigned long long), cudaMemcpyDeviceToHost);
    cudaFree(d);
    return e == cudaSuccess ? 0 : 2;
}
