// ptx.cuh -- thin inline-PTX wrappers used by the sm_103a kernels:
// mbarrier, 1-D bulk async copies (TMA engine), the global timer, and the
// hardware fp8 / fp4 / bf16 conversions.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace nqg {

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---------------------------------------------------- programmatic launch

// Blocks until the grids this one depends on (programmatic dependent launch)
// have completed and their memory operations are visible; a no-op when the
// kernel was launched without the programmatic-serialization attribute.
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Lets the grid that depends on this one begin launching (its threads still
// wait in grid_dependency_wait until this grid has completed).
__device__ __forceinline__ void allow_dependent_launch() { asm volatile("griddepcontrol.launch_dependents;"); }

// ---------------------------------------------------------------- mbarrier

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Makes the initialised barriers visible to the async proxy (bulk copies).
__device__ __forceinline__ void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("{ .reg .b64 st; mbarrier.arrive.shared::cta.b64 st, [%0]; }" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("{ .reg .b64 st; mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1; }" ::"r"(bar),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile("{ .reg .pred p;\n"
                 "  mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
                 "  selp.u32 %0, 1, 0, p; }"
                 : "=r"(ok)
                 : "r"(bar), "r"(parity)
                 : "memory");
    return ok != 0;
}

// Waits for the phase of parity `parity` to complete, for at most
// `limit_ns` of wall-clock time.  Returns false if it gave up.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, uint64_t limit_ns)
{
    if (mbar_try_wait(bar, parity))
        return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        if (mbar_try_wait(bar, parity))
            return true;
        if (globaltimer_ns() - t0 > limit_ns)
            return false;
    }
}

// Hardware barrier `id` (1..15; 0 is __syncthreads) for `count` threads of
// the CTA (a multiple of 32); every participating thread must reach it.
__device__ __forceinline__ void named_barrier_sync(uint32_t id, uint32_t count)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// ------------------------------------------------------ thread-block clusters

__device__ __forceinline__ uint32_t cluster_rank()
{
    uint32_t r;
    asm("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t cluster_size()
{
    uint32_t r;
    asm("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t cluster_id_x()
{
    uint32_t r;
    asm("mov.u32 %0, %%clusterid.x;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t cluster_count_x()
{
    uint32_t r;
    asm("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
    return r;
}

// A cluster barrier in two halves, for work placed between them: every thread
// of the cluster must alternate arrive (release) and wait (acquire), and a wait
// completes once every thread of the cluster that has not exited has arrived.
__device__ __forceinline__ void cluster_arrive_rel() { asm volatile("barrier.cluster.arrive.release;" ::: "memory"); }
__device__ __forceinline__ void cluster_wait_acq() { asm volatile("barrier.cluster.wait.acquire;" ::: "memory"); }
// An arrive that orders nothing by itself: after fence_mbar_init it is the
// pattern that publishes initialised barriers to the peers' acquiring waits.
__device__ __forceinline__ void cluster_arrive_relaxed() { asm volatile("barrier.cluster.arrive.relaxed;" ::: "memory"); }

// Address of the same shared-memory location in cluster CTA `rank`.
__device__ __forceinline__ uint32_t cluster_map(uint32_t local, uint32_t rank)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
    return r;
}

// An asynchronous store of one float into another CTA's shared memory whose
// completion counts 4 transaction bytes on an mbarrier of that CTA (both
// addresses from cluster_map): the data is visible to a thread that has seen
// the barrier's phase complete, and the storing thread does not wait.
__device__ __forceinline__ void st_async_cluster_f32(uint32_t remote, float v, uint32_t remote_bar)
{
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.f32 [%0], %1, [%2];" ::"r"(remote), "f"(v),
                 "r"(remote_bar)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile("{ .reg .pred p;\n"
                 "  mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
                 "  selp.u32 %0, 1, 0, p; }"
                 : "=r"(ok)
                 : "r"(bar), "r"(parity)
                 : "memory");
    return ok != 0;
}

// As mbar_wait_bounded, acquiring at cluster scope what the arriving CTAs
// released.
__device__ __forceinline__ bool mbar_wait_cluster_bounded(uint32_t bar, uint32_t parity, uint64_t limit_ns)
{
    if (mbar_try_wait_cluster(bar, parity))
        return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        if (mbar_try_wait_cluster(bar, parity))
            return true;
        if (globaltimer_ns() - t0 > limit_ns)
            return false;
    }
}

// ---------------------------------------------------------- bulk copies

// One contiguous global -> shared copy through the TMA engine; completion is
// signalled on `bar` as `bytes` transaction bytes.  src, dst and bytes must
// be multiples of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     dst),
                 "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}

// One contiguous shared -> global copy through the TMA engine, added to the
// issuing thread's current bulk group.  dst, src and bytes multiples of 16.
__device__ __forceinline__ void bulk_s2g(void *dst, uint32_t src, uint32_t bytes)
{
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(src), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// Waits until at most one of this thread's bulk groups still reads shared memory.
__device__ __forceinline__ void bulk_wait_read_all_but_one()
{
    asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}

// Waits until every bulk group of this thread has completed.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Orders this thread's earlier shared-memory accesses with its later
// async-proxy (bulk copy) accesses.
__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ------------------------------------------------------------ arithmetic

// x / 6 rounded to nearest even, without a division, wherever the quotient
// is a normal float: q = RN(x * RN(1/6)) is within one ulp of x / 6, the
// remainder x - 6q is exact in one fused multiply-add, and
// RN(q + (x - 6q) * RN(1/6)) is then the correctly rounded quotient
// (Markstein's theorem on FMA-corrected division; P. Markstein, IBM J. Res.
// Dev. 34(1), 1990).  The theorem assumes no underflow: below 2^-126 the
// result may differ in its last place.  Checked on every finite non-negative
// float against the correctly rounded division.
__device__ __forceinline__ float div6_rn(float x)
{
    const float c = 0x1.555556p-3f;  // RN(1/6)
    const float q = __fmul_rn(x, c);
    const float r = __fmaf_rn(-q, 6.0f, x);
    return __fmaf_rn(r, c, q);
}

// a0 / s and a1 / s rounded to nearest even, without a division, wherever
// the quotient is a normal float, given rs = RN(1/s): the same FMA-corrected
// product as div6_rn (Markstein's theorem), on two lanes at once with the
// packed fp32 instructions.  q = RN(a * rs) is within one ulp of a / s, the
// remainder a - q * s is exact in one fma, and RN(q + (a - q * s) * rs) is the
// correctly rounded quotient.  The theorem assumes the remainder does not
// underflow: for an element below 2^-100 it can, and the quotient may differ
// in its last place, but it is then below 2^-91 and its e2m1 code 0 either
// way.  Checked against the correctly rounded division for every positive
// e4m3 block scale and every float a block with that scale can hold.
__device__ __forceinline__ void div_scale_rn2(float a0, float a1, float s, float rs, float &q0, float &q1)
{
    uint64_t a, q, r, rr, ns;
    asm("mov.b64 %0, {%1, %2};" : "=l"(a) : "f"(a0), "f"(a1));
    asm("mov.b64 %0, {%1, %1};" : "=l"(rr) : "f"(rs));
    asm("mov.b64 %0, {%1, %1};" : "=l"(ns) : "f"(-s));
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(q) : "l"(a), "l"(rr));
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(q), "l"(ns), "l"(a));
    asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(q) : "l"(r), "l"(rr));
    asm("mov.b64 {%0, %1}, %2;" : "=f"(q0), "=f"(q1) : "l"(q));
}

// 1 / sqrt(m) for m > 0: the hardware's reciprocal square root (rsqrtf,
// within 2 ulps) refined by one step of Newton's method for f(r) = 1/r^2 - m,
// r' = r + r (1 - m r^2) / 2, which squares the relative error.  For m outside
// the normal range (0, subnormal, infinity) it returns rsqrtf(m) unrefined, so
// a zero sum of squares still gives infinity and an overflowed one 0.
// Checked against the correctly rounded __frsqrt_rn on every normal float.
__device__ __forceinline__ float rsqrt_newton(float m)
{
    const float r = rsqrtf(m);
    const float refined = __fmaf_rn(0.5f * r, __fmaf_rn(-m, r * r, 1.0f), r);
    return (m >= 0x1p-126f && m <= 0x1.fffffep127f) ? refined : r;
}

// ------------------------------------------------------------ conversions

// Two fp32 -> two e4m3 (round to nearest even, saturate to +-448); `lo`
// lands in the low byte.
__device__ __forceinline__ uint32_t cvt_e4m3x2(float lo, float hi)
{
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// Four fp32 -> four e4m3 bytes, element 0 in the lowest byte.
__device__ __forceinline__ uint32_t cvt_e4m3x4(float a, float b, float c, float d)
{
    return cvt_e4m3x2(a, b) | (cvt_e4m3x2(c, d) << 16);
}

// Eight fp32 -> eight e2m1 nibbles (round to nearest even, saturate to +-6),
// element 0 in the lowest nibble.
__device__ __forceinline__ uint32_t cvt_e2m1x8(const float *v)
{
    uint32_t r;
    asm("{ .reg .b8 b0, b1, b2, b3;\n"
        "  cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n"
        "  cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n"
        "  cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n"
        "  cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n"
        "  mov.b32 %0, {b0, b1, b2, b3}; }"
        : "=r"(r)
        : "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]));
    return r;
}

// Value of a non-negative e4m3 code (s.eeee.mmm, bias 7, subnormals at
// exponent field 0), built from the format's definition.
__device__ __forceinline__ float e4m3_code_value(uint32_t c)
{
    const uint32_t e = (c >> 3) & 15u, m = c & 7u;
    if (e == 0)
        return static_cast<float>(m) * 0x1p-9f;
    return __uint_as_float(((e + 120u) << 23) | (m << 20));
}

// bf16x2 (as a 32-bit word) -> two fp32, exact.
__device__ __forceinline__ void bf16x2_to_f32(uint32_t w, float &lo, float &hi)
{
    lo = __uint_as_float(w << 16);
    hi = __uint_as_float(w & 0xFFFF0000u);
}

// fp16x2 (as a 32-bit word) -> two fp32, exact.  Each half goes through the
// mixed-precision add (an fp16 operand, fp32 addend and result; PTX ISA 8.6,
// sm_100 and later) with -0 as the addend: every fp16 number is an fp32
// number and x + (-0) = x for every x, -0 and subnormals included.  Measured
// faster than two conversion instructions (cvt.f32.f16) in the combine.
__device__ __forceinline__ void f16x2_to_f32(uint32_t w, float &lo, float &hi)
{
    asm("{ .reg .b16 l, h;\n"
        "  mov.b32 {l, h}, %2;\n"
        "  add.rn.f32.f16 %0, l, 0f80000000;\n"
        "  add.rn.f32.f16 %1, h, 0f80000000; }"
        : "=f"(lo), "=f"(hi)
        : "r"(w));
}

// Two fp32 -> fp16x2, round to nearest even; `lo` in the low half.
__device__ __forceinline__ uint32_t f32x2_to_f16x2(float lo, float hi)
{
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// acc = w * x + acc on two fp32 lanes at once (packed FMA, each lane rounded
// to nearest exactly like fmaf).
__device__ __forceinline__ void fma2(float &acc_lo, float &acc_hi, float x_lo, float x_hi, float w)
{
    uint64_t a, x, ww;
    asm("mov.b64 %0, {%1, %2};" : "=l"(a) : "f"(acc_lo), "f"(acc_hi));
    asm("mov.b64 %0, {%1, %2};" : "=l"(x) : "f"(x_lo), "f"(x_hi));
    asm("mov.b64 %0, {%1, %1};" : "=l"(ww) : "f"(w));
    asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(a) : "l"(x), "l"(ww));
    asm("mov.b64 {%0, %1}, %2;" : "=f"(acc_lo), "=f"(acc_hi) : "l"(a));
}

// fp32 -> fp16 bits, round to nearest even (exact for a value that is an
// fp16 number, such as a router weight stored as fp16).
__device__ __forceinline__ unsigned short f32_to_f16_bits(float x)
{
    unsigned short r;
    asm("cvt.rn.f16.f32 %0, %1;" : "=h"(r) : "f"(x));
    return r;
}

// acc_lo += lo(x) * w and acc_hi += hi(x) * w for an fp16 pair x (a 32-bit
// word) and an fp16 weight w, without widening x: the mixed-precision fma
// (fp16 multiplicands, fp32 addend and result; PTX ISA 8.6, sm_100 and
// later).  A product of two fp16 numbers is exact in fp32, so each lane
// rounds once, as fmaf of the widened operands does.
__device__ __forceinline__ void fma2_f16(float &acc_lo, float &acc_hi, uint32_t x, unsigned short w)
{
    asm("{ .reg .b16 l, h;\n"
        "  mov.b32 {l, h}, %2;\n"
        "  fma.rn.f32.f16 %0, l, %3, %0;\n"
        "  fma.rn.f32.f16 %1, h, %3, %1; }"
        : "+f"(acc_lo), "+f"(acc_hi)
        : "r"(x), "h"(w));
}

// Two fp32 -> bf16x2, round to nearest even; `lo` in the low half.
__device__ __forceinline__ uint32_t f32x2_to_bf16x2(float lo, float hi)
{
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

} // namespace nqg
