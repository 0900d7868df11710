// Exhaustive check of div_scale_rn2 (the combine's NVFP4 element quotient
// v / s) against the correctly rounded division.  For every positive e4m3
// block scale s and every non-negative float v that a block with that scale
// can hold -- v <= 16 s (amax / 6 rounds to s, so amax < 9 s even for the
// smallest subnormal scale), every finite v for the saturated scale 448 --
// it counts quotients that differ from the correctly rounded one (by where
// they fall), e2m1 codes that differ anywhere, and, for comparison, e2m1
// codes of the plain product v * RN(1/s) that differ from the quotient's.
#include <cstdint>
#include <cuda_runtime.h>

#include "ptx.cuh"

namespace {

__device__ __forceinline__ uint32_t e2m1_code(float x)
{
    uint16_t r;
    asm("{ .reg .b8 b;\n"
        "  cvt.rn.satfinite.e2m1x2.f32 b, 0f00000000, %1;\n"
        "  cvt.u16.u8 %0, b; }"
        : "=h"(r)
        : "f"(x));
    return r & 0xFu;
}

__global__ void quotient_check_kernel(unsigned long long *out)  // see the counters below
{
    const uint32_t c = blockIdx.y + 1;  // e4m3 codes 1..126 (126 = 448, the largest finite)
    const float s = nqg::e4m3_code_value(c);
    const float rs = __frcp_rn(s);
    const uint32_t last = c == 126u ? 0x7F7FFFFFu : __float_as_uint(16.0f * s);
    // [0] quotients differing, v >= 2^-100 and the quotient normal; [1]
    // quotients differing, v < 2^-100 (the remainder v - q s, about 2^-24 v,
    // can then fall below the subnormal range and round, which the theorem
    // excludes; such a quotient is below 2^-91, code 0 either way); [2]
    // quotients differing, the quotient subnormal; [3] e2m1 codes
    // differing anywhere; [4] codes of the plain product v * RN(1/s) differing
    // from the quotient's; [5] values checked; [6] the first (scale code << 32
    // | v bits) of a [0] case, or 0
    unsigned long long cnt[6] = {0, 0, 0, 0, 0, 0};
    unsigned long long first = 0;
    for (uint64_t b = static_cast<uint64_t>(blockIdx.x) * blockDim.x + threadIdx.x; b <= last;
         b += static_cast<uint64_t>(gridDim.x) * blockDim.x) {
        const float v = __uint_as_float(static_cast<uint32_t>(b));
        float q0, q1;
        nqg::div_scale_rn2(v, v, s, rs, q0, q1);
        const float ref = __fdiv_rn(v, s);
        if (__float_as_uint(q0) != __float_as_uint(ref) || __float_as_uint(q1) != __float_as_uint(ref)) {
            if (v < 0x1p-100f) {
                ++cnt[1];
            } else if (ref < 0x1p-126f) {
                ++cnt[2];
            } else {
                ++cnt[0];
                if (!first)
                    first = (static_cast<unsigned long long>(c) << 32) | b;
            }
        }
        const uint32_t want = e2m1_code(ref);
        cnt[3] += e2m1_code(q0) != want;
        cnt[4] += e2m1_code(__fmul_rn(v, rs)) != want;
        ++cnt[5];
    }
    for (int i = 0; i < 6; ++i)
        atomicAdd(out + i, cnt[i]);
    if (first)
        atomicCAS(out + 6, 0ull, first);
}

} // namespace

extern "C" int nvfp4_quotient_check(unsigned long long *host_result)  // 7 counters, as above
{
    unsigned long long *d = nullptr;
    if (cudaMalloc(&d, 7 * sizeof(unsigned long long)) != cudaSuccess)
        return 1;
    cudaMemset(d, 0, 7 * sizeof(unsigned long long));
    quotient_check_kernel<<<dim3(1024, 126), 256>>>(d);
    const cudaError_t e = cudaMemcpy(host_result, d, 7 * sizeof(unsigned long long), cudaMemcpyDeviceToHost);
    cudaFree(d);
    return e == cudaSuccess ? 0 : 2;
}

// The number of floats each scale code is checked on, for the host to
// compare with the device's count.
extern "C" unsigned long long nvfp4_quotient_expected_count()
{
    unsigned long long total = 0;
    for (uint32_t c = 1; c <= 126; ++c) {
        const uint32_t e = (c >> 3) & 15u, m = c & 7u;
        float s;
        if (e == 0) {
            s = static_cast<float>(m) / 512.0f;
        } else {
            const uint32_t bits = ((e + 120u) << 23) | (m << 20);
            __builtin_memcpy(&s, &bits, 4);
        }
        float lim = 16.0f * s;
        uint32_t last;
        __builtin_memcpy(&last, &lim, 4);
        if (c == 126u)
            last = 0x7F7FFFFFu;
        total += static_cast<unsigned long long>(last) + 1ull;
    }
    return total;
}
