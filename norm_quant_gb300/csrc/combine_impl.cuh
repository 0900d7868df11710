// combine_impl.cuh -- the combine kernel template, its launch plan and
// launchers, shared by combine.cu (bf16 I/O) and combine_f16.cu (fp16 I/O).
// What the kernel computes and how it is laid out is described in combine.cu.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "common.h"
#include "ptx.cuh"

namespace nqg {
namespace combine_detail {

constexpr uint64_t kWaitLimitNs = 2000000000ull;
constexpr int kMaxStages = 32;
constexpr size_t kSmemBudget = 226 * 1024;
constexpr size_t kDefaultRingBytes = 144 * 1024;

// Consumer warps allowed per CTA for each VPT (vectors of 8 elements per
// consumer thread); the CTA adds one producer warp.  Together they cover
// H <= 4096 (VPT 1), 8192 (VPT 2, 4) and 16384 (VPT 8).
template <int VPT>
__host__ __device__ constexpr int max_consumer_warps() { return VPT <= 2 ? 16 : 8; }
inline int max_consumer_warps_rt(int vpt) { return vpt <= 2 ? 16 : 8; }
// Rows a consumer loads into registers at once (its chunk of a slot),
// bounded by the registers the loads take; a slot holds up to kMaxSlotRows.
template <int VPT>
__host__ __device__ constexpr int chunk_rows() { return VPT <= 2 ? 4 : (VPT == 4 ? 2 : 1); }
constexpr int kMaxSlotRows = 12;

enum : int32_t { F_LAST = 1, F_RESID = 2 };

struct alignas(16) StageMeta {
    int32_t t;
    int32_t n;      // rows in the slot, 0..R
    int32_t flags;  // F_LAST: the token's last slot; F_RESID: its last row is the residual
    int32_t pad;
    float w[kMaxSlotRows];  // weight of each row (1 for the shared and residual rows)
};

struct Params {
    int64_t T;
    int32_t H, k;
    const uint8_t *expert_out;
    int64_t n_rows;
    const int32_t *row_map;
    const void *weights;
    const uint8_t *shared;
    const uint8_t *residual;
    const uint16_t *gamma;
    float eps, wb, gscale;
    float inv_h;           // 1 / H in fp32 (the mean of the squares is their sum times this)
    int32_t weight_dtype;  // moe_weight_dtype of router_weights
    int32_t sf_layout;
    uint16_t *combined_out, *residual_out, *norm_out;
    uint8_t *quant_out, *scales_out;
    int32_t *status;
    int32_t stages, rows;  // ring slots, rows per slot
    int32_t slot_major;    // expert_out is [k, T, H]: row of (t, j) is j * T + t
    int32_t split;         // CTAs sharing one token (the cluster size), 1 = a whole row per CTA
    int32_t hl;            // columns each CTA handles: H / split
    int64_t stall_after;   // test hook (moe_debug_stall): -1 off, else CTA 0 stages this many slots
    int64_t sf_cols, sf_cols_pad, sf_rows_pad;
};

struct SmemLayout {
    uint32_t row_stride, slot_stride, bars, meta, red, gamma, rtab, total;
};

// Shared memory of one CTA handling Hl columns of each row: the ring, its
// barriers (full[S], empty[S], the consumers' abort word, the gamma copy's
// barrier, and the two cross-CTA reduction barriers of a split
// token), the slots' StageMeta, two buffers of per-warp partial sums for
// csize CTAs, then (with a norm) the Hl gamma values, then a table of the
// e4m3 block scales' values and reciprocals (NVFP4).
__host__ __device__ inline SmemLayout smem_layout(int32_t Hl, int32_t stages, int32_t rows, int32_t ncw,
                                                  int32_t csize, bool with_gamma)
{
    SmemLayout L;
    L.row_stride = (static_cast<uint32_t>(Hl) * 2u + 127u) & ~127u;
    L.slot_stride = L.row_stride * static_cast<uint32_t>(rows);
    L.bars = static_cast<uint32_t>(stages) * L.slot_stride;
    L.meta = L.bars + (2u * stages + 4u) * 8u;
    L.red = L.meta + static_cast<uint32_t>(stages) * static_cast<uint32_t>(sizeof(StageMeta));
    L.gamma = (L.red + 2u * static_cast<uint32_t>(csize) * static_cast<uint32_t>(ncw) * 4u + 127u) & ~127u;
    L.rtab = (L.gamma + (with_gamma ? static_cast<uint32_t>(Hl) * 2u : 0u) + 15u) & ~15u;
    L.total = L.rtab + 128u * 8u;  // value and reciprocal of the 128 non-negative e4m3 codes
    return L;
}

__device__ __forceinline__ void report(int32_t *status, int32_t code)
{
    if (status)
        atomicCAS(status, 0, code);
}

__device__ __forceinline__ int64_t sf_offset(int64_t r, int64_t c, const Params &p)
{
    if (p.sf_layout == MOE_SF_LINEAR)
        return r * p.sf_cols + c;
    return (r >> 7) * (p.sf_cols_pad >> 2) * 512 + (c >> 2) * 512 + (r & 31) * 16 + ((r & 127) >> 5) * 4 + (c & 3);
}

// UE8M0 byte of a block whose absolute maximum is `amax` (>= 0, finite):
// the smallest e with amax <= 448 * 2^e -- with amax = m * 2^p, m in [1, 2),
// that is e = p - 8 when m <= 1.75 and p - 7 otherwise -- biased by 127 and
// clamped to [0, 254].
__device__ __forceinline__ int32_t ue8m0_byte(float amax)
{
    const uint32_t bits = __float_as_uint(amax);
    const int32_t ef = static_cast<int32_t>(bits >> 23);
    if (ef == 0)
        return 0;  // zero or below 2^-126: e <= -134 clamps to 0
    const int32_t p = ef - 127;
    const int32_t e = ((bits & 0x7FFFFFu) <= 0x600000u) ? p - 8 : p - 7;
    const int32_t b = e + 127;
    return b < 0 ? 0 : (b > 254 ? 254 : b);
}

// 16-bit element codecs.  IO 0 = bf16; 1 = fp16; 2 = fp16 with fp16 router
// weights (the same codecs as 1; only the weighted sum differs: the rows are
// not widened, each element takes one mixed-precision fma).
template <int IO>
__device__ __forceinline__ void unpack16x2(uint32_t w, float &lo, float &hi)
{
    if constexpr (IO == 0) {
        bf16x2_to_f32(w, lo, hi);
    } else {
        f16x2_to_f32(w, lo, hi);
    }
}

template <int IO>
__device__ __forceinline__ uint32_t pack16x2(float lo, float hi)
{
    if constexpr (IO == 0)
        return f32x2_to_bf16x2(lo, hi);
    else
        return f32x2_to_f16x2(lo, hi);
}

template <int IO>
__device__ __forceinline__ void store16x8(uint16_t *base, int64_t off, const float *v)
{
    uint4 q;
    q.x = pack16x2<IO>(v[0], v[1]);
    q.y = pack16x2<IO>(v[2], v[3]);
    q.z = pack16x2<IO>(v[4], v[5]);
    q.w = pack16x2<IO>(v[6], v[7]);
    *reinterpret_cast<uint4 *>(base + off) = q;
}

// Router weight idx as fp32: stored as fp32, bf16 or fp16 (moe_weight_dtype).
__device__ __forceinline__ float load_weight(const void *w, int64_t idx, int32_t dtype)
{
    if (dtype == MOE_WEIGHTS_FP32)
        return __ldg(static_cast<const float *>(w) + idx);
    const uint32_t b = __ldg(static_cast<const unsigned short *>(w) + idx);
    if (dtype == MOE_WEIGHTS_BF16)
        return __uint_as_float(b << 16);
    float lo, hi;
    f16x2_to_f32(b, lo, hi);
    return lo;
}

// UE8M0 byte for MXFP4: the smallest e with amax <= 6 * 2^e -- with
// amax = m * 2^p, e = p - 2 when m <= 1.5 and p - 1 otherwise -- biased by
// 127 and clamped to [0, 254].
__device__ __forceinline__ int32_t ue8m0_fp4_byte(float amax)
{
    const uint32_t bits = __float_as_uint(amax);
    const int32_t ef = static_cast<int32_t>(bits >> 23);
    if (ef == 0)
        return 0;
    const int32_t p = ef - 127;
    const int32_t e = ((bits & 0x7FFFFFu) <= 0x400000u) ? p - 2 : p - 1;
    const int32_t b = e + 127;
    return b < 0 ? 0 : (b > 254 ? 254 : b);
}

// N consecutive slot weights from shared memory (16-byte aligned for N = 4,
// 8-byte for N = 2) in one load.
template <int N>
__device__ __forceinline__ void load_weights(const float *w, float *out)
{
    if constexpr (N == 4) {
        const float4 x = *reinterpret_cast<const float4 *>(w);
        out[0] = x.x;
        out[1] = x.y;
        out[2] = x.z;
        out[3] = x.w;
    } else if constexpr (N == 2) {
        const float2 x = *reinterpret_cast<const float2 *>(w);
        out[0] = x.x;
        out[1] = x.y;
    } else {
        out[0] = w[0];
    }
}

// Position of the set bit of `mask` that has `rank` set bits below it
// (rank < popc(mask)), by halving the search window: skip the low half of the
// window when it holds no more than `rank` set bits.  A result whose bit is
// not set (impossible for a valid rank) is replaced by the lowest set bit, so
// the lane it names always holds a valid row.
__device__ __forceinline__ int nth_set_bit(uint32_t mask, int rank)
{
    uint32_t m = mask;
    int pos = 0;
#pragma unroll
    for (int b = 16; b >= 1; b >>= 1) {
        const int c = __popc(m & ((1u << b) - 1u));
        if (c <= rank) {
            rank -= c;
            m >>= b;
            pos += b;
        }
    }
    return ((mask >> pos) & 1u) ? pos : (mask ? __ffs(mask) - 1 : 0);
}

template <int VPT, int QUANT, int IO, bool SPLIT>
__global__ void __launch_bounds__((max_consumer_warps<VPT>() + 1) * 32, 1) combine_kernel(const Params p)
{
    constexpr int RCH = chunk_rows<VPT>();
    extern __shared__ __align__(128) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int ncw = (blockDim.x >> 5) - 1;
    const int NC = ncw * 32;
    const int S = p.stages;
    const int R = p.rows;
    const int32_t H = p.H, k = p.k;
    // This CTA handles columns [col0, col0 + Hl) of its tokens' rows: the
    // whole row, or with SPLIT the slice of its rank in a cluster of
    // p.split CTAs that all walk the same tokens (one token per cluster).
    const uint32_t csize = SPLIT ? static_cast<uint32_t>(p.split) : 1u;
    // work units (tokens in flight at once): CTAs, or with SPLIT clusters
    const uint32_t crank = SPLIT ? cluster_rank() : 0u;
    const int64_t unit0 = SPLIT ? cluster_id_x() : blockIdx.x;
    auto nunits = []() -> int64_t { return SPLIT ? cluster_count_x() : gridDim.x; };
    const int32_t Hl = SPLIT ? p.hl : H;
    const int32_t col0 = SPLIT ? static_cast<int32_t>(crank) * Hl : 0;
    const int32_t vec0 = col0 >> 3;  // first 8-element vector of the slice
    const int32_t nvec = Hl >> 3;
    const uint32_t row_bytes = static_cast<uint32_t>(H) * 2u;  // pitch of every input row
    const uint32_t copy_bytes = static_cast<uint32_t>(Hl) * 2u;
    const uint32_t col_bytes = static_cast<uint32_t>(col0) * 2u;
    const SmemLayout L = smem_layout(Hl, S, R, ncw, static_cast<int32_t>(csize), p.gamma != nullptr);
    const uint32_t ring = smem_u32(smem);
    const uint32_t full0 = ring + L.bars, empty0 = full0 + 8u * S;
    const uint32_t gbar = empty0 + 8u * S + 8u;  // the gamma copy
    const uint32_t xbar0 = gbar + 8u;            // two cross-CTA barriers, by token parity
    StageMeta *meta = reinterpret_cast<StageMeta *>(smem + L.meta);
    float *red = reinterpret_cast<float *>(smem + L.red);

    // set by a consumer warp whose bounded wait gave up, before it meets the
    // others at the norm's barrier; read by every consumer warp after it
    int32_t *abort_word = reinterpret_cast<int32_t *>(smem + L.bars + 16u * S);
    if (threadIdx.x == 0) {
        *abort_word = 0;
        for (int s = 0; s < S; ++s) {
            mbar_init(full0 + 8u * s, 1);
            mbar_init(empty0 + 8u * s, ncw);
        }
        mbar_init(gbar, 1);
        if constexpr (SPLIT) {
            // one local arrival a token (with the expected bytes); the peers'
            // partials complete the transaction bytes
            mbar_init(xbar0, 1);
            mbar_init(xbar0 + 8u, 1);
        }
        fence_mbar_init();
    }
    if constexpr (QUANT == MOE_QUANT_NVFP4) {
        // every non-negative e4m3 code's value and its correctly rounded fp32
        // reciprocal (0 for code 0, which is never divided by)
        float2 *rtab = reinterpret_cast<float2 *>(smem + L.rtab);
        for (uint32_t c = threadIdx.x; c < 128u; c += blockDim.x)
            rtab[c] = make_float2(e4m3_code_value(c), c ? __frcp_rn(e4m3_code_value(c)) : 0.f);
    }
    __syncthreads();
    // with SPLIT, every CTA's barriers are initialised before any peer arrives
    // on them: each thread arrives on the cluster barrier here and waits on it
    // only before its first access to a peer's shared memory (the norm's
    // exchange), so the barrier's latency hides behind the rows' copies.  The
    // init was published by thread 0's fence_mbar_init, so the arrive is
    // relaxed (a release here cost about 400 cycles)
    bool cl_waited = !SPLIT, cl_arrived2 = !SPLIT;
    if constexpr (SPLIT)
        cluster_arrive_relaxed();
    // launched as a programmatic dependent: nothing before this line touches
    // global memory, so the setup above overlaps the previous kernel's tail
    grid_dependency_wait();

    if (warp == ncw) {
        // ------------------------------------------------------- producer
        [&]() {
            int stage = 0;
            uint32_t phase = 0;
            int64_t issued = 0;
            bool ok = true, stalled = false;
            int64_t t = unit0;
            int32_t r_next = -1;
            float w_next = 0.f;
            auto row_of = [&](int64_t tt) {
                return p.slot_major ? static_cast<int32_t>(lane * p.T + tt) : __ldg(p.row_map + tt * k + lane);
            };
            if (p.gamma && lane == 0) {
                mbar_arrive_expect_tx(gbar, copy_bytes);
                bulk_g2s(ring + L.gamma, p.gamma + col0, copy_bytes, gbar);
            }
            if (t < p.T && lane < k) {
                r_next = row_of(t);
                w_next = load_weight(p.weights, t * k + lane, p.weight_dtype);
            }
            for (; t < p.T && ok && !stalled; t += nunits()) {
                const int32_t r = r_next;
                const float w = w_next;
                const int64_t tn = t + nunits();
                if (tn < p.T && lane < k) {
                    r_next = row_of(tn);
                    w_next = load_weight(p.weights, tn * k + lane, p.weight_dtype);
                }
                bool valid = lane < k && r >= 0;
                if (valid && r >= p.n_rows) {
                    report(p.status, MOE_ERR_ROW_OUT_OF_RANGE);
                    valid = false;
                }
                const uint32_t mval = __ballot_sync(0xffffffffu, valid);
                const int n_exp = __popc(mval);
                const bool has_sh = p.shared != nullptr, has_res = p.residual != nullptr;
                const int n = n_exp + (has_sh ? 1 : 0) + (has_res ? 1 : 0);
                // the token's rows spread evenly over ceil(n / R) slots (9 rows
                // at R = 4 as 3 + 3 + 3, not 4 + 4 + 1); a token with no rows
                // still gets one slot
                const int nslots = n > 0 ? (n + R - 1) / R : 1;
                int i = 0, si = 0;
                do {
                    if (p.stall_after >= 0 && blockIdx.x == 0 && issued >= p.stall_after) {
                        // test hook: CTA 0 stages nothing more, so that its
                        // consumers' bounded waits run out
                        stalled = true;
                        break;
                    }
                    const int left = nslots - si;
                    const int ns = (n - i + left - 1) / left;
                    // lane q stages row i + q: the (i + q)-th valid expert slot in
                    // ascending j, then the shared row, then the residual row
                    const int ii = i + lane;
                    const bool mine = lane < ns;
                    const int j = nth_set_bit(mval, ii < n_exp ? ii : 0);
                    const int32_t rj = __shfl_sync(0xffffffffu, r, j);
                    const float wj = __shfl_sync(0xffffffffu, w, j);
                    const uint8_t *src = nullptr;
                    if (mine) {
                        if (ii < n_exp)
                            src = p.expert_out + static_cast<int64_t>(rj) * row_bytes + col_bytes;
                        else if (has_sh && ii == n_exp)
                            src = p.shared + t * row_bytes + col_bytes;
                        else
                            src = p.residual + t * row_bytes + col_bytes;
                    }
                    const bool last = (i + ns >= n);
                    bool good = true;
                    if (lane == 0)
                        good = mbar_wait_bounded(empty0 + 8u * stage, phase ^ 1u, kWaitLimitNs);
                    good = __shfl_sync(0xffffffffu, good, 0);
                    if (!good) {
                        ok = false;
                        break;
                    }
                    // each lane copies its own row and records its weight; lane 0
                    // then publishes the slot and arms its barrier.  Until lane
                    // 0 arrives the phase has an arrival pending, so copies that
                    // land before the expected bytes are set cannot complete it.
                    const uint32_t full = full0 + 8u * stage;
                    StageMeta &m = meta[stage];
                    if (mine) {
                        m.w[lane] = ii < n_exp ? wj : 1.f;
                        bulk_g2s(ring + static_cast<uint32_t>(stage) * L.slot_stride +
                                     static_cast<uint32_t>(lane) * L.row_stride,
                                 src, copy_bytes, full);
                    }
                    __syncwarp();
                    if (lane == 0) {
                        m.t = static_cast<int32_t>(t);
                        m.n = ns;
                        m.flags = (last ? F_LAST : 0) | ((last && has_res && ns > 0) ? F_RESID : 0);
                        if (ns > 0)
                            mbar_arrive_expect_tx(full, static_cast<uint32_t>(ns) * copy_bytes);
                        else
                            mbar_arrive(full);
                    }
                    ++issued;
                    if (++stage == S) {
                        stage = 0;
                        phase ^= 1u;
                    }
                    i += ns;
                    ++si;
                } while (i < n);
            }
            if (!ok && lane == 0) {
                // a slot never freed up: record it, then let every copy this
                // warp started land before the CTA's shared memory goes away
                report(p.status, MOE_ERR_DEVICE_TIMEOUT);
                if (p.gamma)
                    mbar_wait_bounded(gbar, 0, kWaitLimitNs);
                const int64_t nn = issued < S ? issued : S;
                for (int64_t s = 0; s < nn; ++s) {
                    const int64_t times = (issued - 1 - s) / S + 1;
                    mbar_wait_bounded(full0 + 8u * static_cast<uint32_t>(s), static_cast<uint32_t>((times - 1) & 1),
                                      kWaitLimitNs);
                }
            }
        }();
    } else {
        // ----------------------------------------------------------- consumers
        [&]() {
            const int tid = threadIdx.x;
            // pad rows of a swizzled scale matrix are written as zero.  They
            // are rows T % 128 .. 127 of the last 128-row tile.  In that
            // layout the 512 bytes of one column group of a tile hold, at
            // 16 * L, the 4 columns of rows L, L + 32, L + 64 and L + 96: a
            // warp clears a column group with lane L storing its 16 bytes, or
            // only the 4-byte cells of pad rows where the lane holds real rows
            if (QUANT != MOE_QUANT_NONE && p.sf_layout == MOE_SF_SWIZZLED_128x4 && p.sf_rows_pad > p.T) {
                const uint32_t groups = static_cast<uint32_t>(p.sf_cols_pad >> 2);
                const uint32_t r0 = static_cast<uint32_t>(p.T & 127);
                uint8_t *const tile = p.scales_out + (p.T >> 7) * static_cast<int64_t>(groups) * 512;
                const uintptr_t base = reinterpret_cast<uintptr_t>(p.scales_out);
                const bool v16 = (base & 15u) == 0, w4 = (base & 3u) == 0;
                for (uint32_t g = blockIdx.x * static_cast<uint32_t>(ncw) + warp; g < groups;
                     g += gridDim.x * static_cast<uint32_t>(ncw)) {
                    uint8_t *const cell = tile + g * 512u + static_cast<uint32_t>(lane) * 16u;
                    if (static_cast<uint32_t>(lane) >= r0 && v16) {
                        *reinterpret_cast<uint4 *>(cell) = make_uint4(0u, 0u, 0u, 0u);
                        continue;
                    }
#pragma unroll
                    for (uint32_t q = 0; q < 4; ++q) {
                        if (static_cast<uint32_t>(lane) + 32u * q < r0)
                            continue;  // a real row: its scales are the epilogue's
                        if (w4) {
                            *reinterpret_cast<uint32_t *>(cell + 4u * q) = 0u;
                        } else {
                            cell[4u * q] = 0;
                            cell[4u * q + 1] = 0;
                            cell[4u * q + 2] = 0;
                            cell[4u * q + 3] = 0;
                        }
                    }
                }
            }
            const bool do_norm = p.gamma != nullptr;
            const int max_slots = k + 3;  // a token never needs more slots than rows + 1
            // Without SPLIT, the consumer warps meet at a named hardware barrier
            // once per token, for the norm.  A warp whose bounded wait gives up
            // must still meet the others there, or they would wait forever: it
            // raises abort_word, arrives at the barrier of the token it is in,
            // and leaves; every warp reads abort_word after that barrier and
            // leaves before its next store.  A warp reaches a token's barrier
            // only once that token's slots have all filled, so the barrier the
            // warp that gave up arrives at is the one every other warp is bound
            // for.
            const bool meets = !SPLIT && do_norm;
            auto give_up = [&]() {
                if (meets) {
                    if (lane == 0)
                        *reinterpret_cast<volatile int32_t *>(abort_word) = 1;
                    named_barrier_sync(1, NC);
                }
                report(p.status, MOE_ERR_DEVICE_TIMEOUT);
            };
            // gamma's slice, copied to shared memory once by the producer
            if (do_norm && __any_sync(0xffffffffu, !mbar_wait_bounded(gbar, 0, kWaitLimitNs))) {
                give_up();
                return;
            }

            int stage = 0;
            uint32_t phase = 0;
            uint32_t tok = 0;
            for (int64_t t = unit0; t < p.T; t += nunits(), ++tok) {
                float acc[VPT][8];
#pragma unroll
                for (int s = 0; s < VPT; ++s)
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        acc[s][i] = 0.f;
                bool combined_done = false;
                for (int it = 0; it < max_slots; ++it) {
                    // a give-up is taken by the whole warp, so that no lane is
                    // left behind in the warp-wide shuffles below
                    if (__any_sync(0xffffffffu, !mbar_wait_bounded(full0 + 8u * stage, phase, kWaitLimitNs))) {
                        give_up();
                        return;
                    }
                    // the slot's header (t, n, flags) in one 16-byte load
                    const int4 hdr = *reinterpret_cast<const int4 *>(&meta[stage]);
                    const int mn = hdr.y, mflags = hdr.z;
                    const uint8_t *slot = smem + static_cast<uint32_t>(stage) * L.slot_stride;
                    // the slot's rows in chunks of RCH: all of a chunk's loads
                    // first, then its sums in row order
#pragma unroll
                    for (int c0 = 0; c0 < kMaxSlotRows; c0 += RCH) {
                        if (c0 >= mn)
                            break;
                        uint4 q[RCH][VPT];
                        // the chunk's weights in one vector load (beyond the
                        // slot's rows they are stale and unused)
                        float wr[RCH];
                        load_weights<RCH>(meta[stage].w + c0, wr);
#pragma unroll
                        for (int rr = 0; rr < RCH; ++rr) {
                            const int row = c0 + rr;
#pragma unroll
                            for (int s = 0; s < VPT; ++s) {
                                const int v = s * NC + tid;
                                q[rr][s] = make_uint4(0, 0, 0, 0);
                                if (row < mn && v < nvec)
                                    q[rr][s] = *reinterpret_cast<const uint4 *>(slot + row * L.row_stride + 16 * v);
                            }
                        }
#pragma unroll
                        for (int rr = 0; rr < RCH; ++rr) {
                            const int row = c0 + rr;
                            if (row >= mn)
                                break;
                            if ((mflags & F_RESID) && row == mn - 1 && p.combined_out) {
#pragma unroll
                                for (int s = 0; s < VPT; ++s) {
                                    const int v = s * NC + tid;
                                    if (v < nvec)
                                        store16x8<IO>(p.combined_out, t * H + col0 + 8 * v, acc[s]);
                                }
                                combined_done = true;
                            }
#pragma unroll
                            for (int s = 0; s < VPT; ++s) {
                                const int v = s * NC + tid;
                                if (v < nvec) {
                                    const uint32_t qw[4] = {q[rr][s].x, q[rr][s].y, q[rr][s].z, q[rr][s].w};
                                    if constexpr (IO == 2) {
                                        // the weight is an fp16 number (or the
                                        // 1 of the shared / residual row)
                                        const unsigned short wh = f32_to_f16_bits(wr[rr]);
#pragma unroll
                                        for (int i = 0; i < 4; ++i)
                                            fma2_f16(acc[s][2 * i], acc[s][2 * i + 1], qw[i], wh);
                                    } else {
#pragma unroll
                                        for (int i = 0; i < 4; ++i) {
                                            float lo, hi;
                                            unpack16x2<IO>(qw[i], lo, hi);
                                            fma2(acc[s][2 * i], acc[s][2 * i + 1], lo, hi, wr[rr]);
                                        }
                                    }
                                }
                            }
                        }
                    }
                    __syncwarp();
                    if (lane == 0)
                        mbar_arrive(empty0 + 8u * stage);
                    if (++stage == S) {
                        stage = 0;
                        phase ^= 1u;
                    }
                    if (mflags & F_LAST)
                        break;
                }

                // -------------------------------------------------- epilogue
                const int64_t row0 = t * H + col0;  // element offset of this CTA's slice of row t
                auto store_sums = [&]() {
                    if (p.combined_out && !combined_done) {
#pragma unroll
                        for (int s = 0; s < VPT; ++s) {
                            const int v = s * NC + tid;
                            if (v < nvec)
                                store16x8<IO>(p.combined_out, row0 + 8 * v, acc[s]);
                        }
                    }
                    if (p.residual_out) {
#pragma unroll
                        for (int s = 0; s < VPT; ++s) {
                            const int v = s * NC + tid;
                            if (v < nvec)
                                store16x8<IO>(p.residual_out, row0 + 8 * v, acc[s]);
                        }
                    }
                };
                // with SPLIT and a norm, the sums are stored after this thread's
                // release operations toward the peers (below), so that those
                // do not wait for the stores to drain
                if (!(SPLIT && do_norm))
                    store_sums();
                if (do_norm) {
                    uint4 gq[VPT];
#pragma unroll
                    for (int s = 0; s < VPT; ++s) {
                        const int v = s * NC + tid;
                        gq[s] = (v < nvec) ? *reinterpret_cast<const uint4 *>(smem + L.gamma + 16 * v)
                                           : make_uint4(0, 0, 0, 0);
                    }
                    float ss = 0.f;
#pragma unroll
                    for (int s = 0; s < VPT; ++s)
#pragma unroll
                        for (int i = 0; i < 8; ++i)
                            ss = fmaf(acc[s][i], acc[s][i], ss);  // vectors past the slice hold 0
#pragma unroll
                    for (int d = 16; d > 0; d >>= 1)
                        ss += __shfl_xor_sync(0xffffffffu, ss, d);
                    const float *part;
                    int np;
                    int32_t aborted = 0;
                    if constexpr (SPLIT) {
                        // every warp of every CTA of the cluster sends its partial
                        // to slot [rank][warp] of every CTA (lane r to CTA r) as
                        // an asynchronous store that completes on that CTA's
                        // exchange barrier; each CTA then adds all csize * ncw
                        // of them in the same order, so the whole token sees one
                        // norm.  Buffers and barriers alternate with the token's
                        // parity: a CTA can run at most one token ahead of a peer
                        // that has not yet read its partials.
                        const uint32_t par = tok & 1u;
                        part = red + par * csize * static_cast<uint32_t>(ncw);
                        if (!cl_waited) {
                            cluster_wait_acq();
                            cl_waited = true;
                        }
                        // this token's partials from every warp of every CTA
                        // arrive as transaction bytes (the count can run below
                        // zero before this arrival sets it, and the phase still
                        // waits for the arrival)
                        if (warp == 0 && lane == 0)
                            mbar_arrive_expect_tx(xbar0 + 8u * par, csize * static_cast<uint32_t>(ncw) * 4u);
                        __syncwarp();
                        if (static_cast<uint32_t>(lane) < csize) {
                            const uint32_t mine = smem_u32(part + crank * ncw + warp);
                            st_async_cluster_f32(cluster_map(mine, lane), ss, cluster_map(xbar0 + 8u * par, lane));
                        }
                        if (t + nunits() >= p.T) {
                            // the CTA's last exchange: this thread has written
                            // into its peers' shared memory for the last time,
                            // so it arrives on the exit barrier now and waits on
                            // it at the very end.  The barrier completes only
                            // once every peer has arrived too, each after its
                            // own last stores into this CTA; the release orders
                            // those stores before the arrival (a relaxed arrive,
                            // measured faster, would not).
                            cluster_arrive_rel();
                            cl_arrived2 = true;
                        }
                        store_sums();
                        if (__any_sync(0xffffffffu,
                                       !mbar_wait_cluster_bounded(xbar0 + 8u * par, (tok >> 1) & 1u, kWaitLimitNs))) {
                            report(p.status, MOE_ERR_DEVICE_TIMEOUT);
                            return;
                        }
                        np = static_cast<int>(csize) * ncw;
                    } else {
                        float *mine = red + (tok & 1u) * ncw;
                        if (lane == 0)
                            mine[warp] = ss;
                        named_barrier_sync(1, NC);  // the consumer warps only
                        aborted = *abort_word;      // checked before the next store
                        part = mine;
                        np = ncw;
                    }
                    // the partials, strided over the lanes and then added by a
                    // butterfly: each step adds the same two values in every
                    // lane (addition commutes), so all lanes of all warps end
                    // with one identical total
                    float total = 0.f;
                    for (int w = lane; w < np; w += 32)
                        total += part[w];
#pragma unroll
                    for (int d = 16; d > 0; d >>= 1)
                        total += __shfl_xor_sync(0xffffffffu, total, d);
                    const float rinv = rsqrt_newton(fmaf(total, p.inv_h, p.eps));
#pragma unroll
                    for (int s = 0; s < VPT; ++s) {
                        const uint32_t gv[4] = {gq[s].x, gq[s].y, gq[s].z, gq[s].w};
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            float lo, hi;
                            unpack16x2<IO>(gv[i], lo, hi);
                            acc[s][2 * i] = acc[s][2 * i] * rinv * (lo + p.wb);
                            acc[s][2 * i + 1] = acc[s][2 * i + 1] * rinv * (hi + p.wb);
                        }
                    }
                    if (aborted)  // a warp gave up (and has reported)
                        return;
                    if (p.norm_out) {
#pragma unroll
                        for (int s = 0; s < VPT; ++s) {
                            const int v = s * NC + tid;
                            if (v < nvec)
                                store16x8<IO>(p.norm_out, row0 + 8 * v, acc[s]);
                        }
                    }
                }

                if constexpr (QUANT == MOE_QUANT_MXFP8) {
#pragma unroll
                    for (int s = 0; s < VPT; ++s) {
                        const int v = s * NC + tid;
                        const bool vv = v < nvec;
                        float amax = 0.f;
#pragma unroll
                        for (int i = 0; i < 8; ++i)
                            amax = fmaxf(amax, fabsf(acc[s][i]));
                        amax = vv ? amax : 0.f;
                        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
                        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
                        const int32_t byte = ue8m0_byte(amax);
                        const float scale = __uint_as_float(static_cast<uint32_t>(254 - byte) << 23);  // 2^-e
                        if (vv) {
                            uint2 qv;
                            qv.x = cvt_e4m3x4(acc[s][0] * scale, acc[s][1] * scale, acc[s][2] * scale,
                                              acc[s][3] * scale);
                            qv.y = cvt_e4m3x4(acc[s][4] * scale, acc[s][5] * scale, acc[s][6] * scale,
                                              acc[s][7] * scale);
                            *reinterpret_cast<uint2 *>(p.quant_out + row0 + 8 * v) = qv;
                            if ((lane & 3) == 0) {
                                const int64_t c = (vec0 + v) >> 2;
                                p.scales_out[sf_offset(t, c, p)] = static_cast<uint8_t>(byte);
                                if (c == p.sf_cols - 1)
                                    for (int64_t cp = p.sf_cols; cp < p.sf_cols_pad; ++cp)
                                        p.scales_out[sf_offset(t, cp, p)] = 0;
                            }
                        }
                    }
                } else if constexpr (QUANT == MOE_QUANT_MXFP4) {
#pragma unroll
                    for (int s = 0; s < VPT; ++s) {
                        const int v = s * NC + tid;
                        const bool vv = v < nvec;
                        float amax = 0.f;
#pragma unroll
                        for (int i = 0; i < 8; ++i)
                            amax = fmaxf(amax, fabsf(acc[s][i]));
                        amax = vv ? amax : 0.f;
                        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
                        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
                        const int32_t byte = ue8m0_fp4_byte(amax);
                        const float scale = __uint_as_float(static_cast<uint32_t>(254 - byte) << 23);  // 2^-e
                        if (vv) {
                            float qv[8];
#pragma unroll
                            for (int i = 0; i < 8; ++i)
                                qv[i] = acc[s][i] * scale;
                            *reinterpret_cast<uint32_t *>(p.quant_out + (row0 >> 1) + 4 * v) = cvt_e2m1x8(qv);
                            if ((lane & 3) == 0) {
                                const int64_t c = (vec0 + v) >> 2;
                                p.scales_out[sf_offset(t, c, p)] = static_cast<uint8_t>(byte);
                                if (c == p.sf_cols - 1)
                                    for (int64_t cp = p.sf_cols; cp < p.sf_cols_pad; ++cp)
                                        p.scales_out[sf_offset(t, cp, p)] = 0;
                            }
                        }
                    }
                } else if constexpr (QUANT == MOE_QUANT_NVFP4) {
#pragma unroll
                    for (int s = 0; s < VPT; ++s) {
                        const int v = s * NC + tid;
                        const bool vv = v < nvec;
                        float g[8];
                        float amax = 0.f;
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            g[i] = acc[s][i] * p.gscale;
                            amax = fmaxf(amax, fabsf(g[i]));
                        }
                        amax = vv ? amax : 0.f;
                        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
                        const uint32_t sc = cvt_e4m3x2(div6_rn(amax), 0.f) & 0xFFu;
                        if (vv) {
                            uint32_t packed = 0;
                            if (sc != 0u) {
                                // each element divided by the block scale, the
                                // quotient correctly rounded to fp32 (from the
                                // scale's value and reciprocal in the table)
                                const float2 sr = reinterpret_cast<const float2 *>(smem + L.rtab)[sc];
                                float qv[8];
#pragma unroll
                                for (int i = 0; i < 8; i += 2)
                                    div_scale_rn2(g[i], g[i + 1], sr.x, sr.y, qv[i], qv[i + 1]);
                                packed = cvt_e2m1x8(qv);
                            }
                            *reinterpret_cast<uint32_t *>(p.quant_out + (row0 >> 1) + 4 * v) = packed;
                            if ((lane & 1) == 0) {
                                const int64_t c = (vec0 + v) >> 1;
                                p.scales_out[sf_offset(t, c, p)] = static_cast<uint8_t>(sc);
                                if (c == p.sf_cols - 1)
                                    for (int64_t cp = p.sf_cols; cp < p.sf_cols_pad; ++cp)
                                        p.scales_out[sf_offset(t, cp, p)] = 0;
                            }
                        }
                    }
                }
            }
        }();
    }
    // with SPLIT, no CTA leaves while a peer may still write into its shared
    // memory or arrive on its barriers.  Every wait above is bounded, so every
    // thread gets here; one that left its work early (a wait gave up, or the
    // producer) completes its arrive-wait-arrive sequence here.
    if constexpr (SPLIT) {
        if (!cl_waited)
            cluster_wait_acq();
        if (!cl_arrived2)
            cluster_arrive_rel();
        cluster_wait_acq();
    }
}

// ------------------------------------------------------------------- host

// Process-wide plan overrides set by moe_tuning_set (0 = automatic).
struct Tuning {
    int vpt = 0, rows = 0, ring_kib = 0, ctas_per_sm = 0, split = 0;
    int64_t stall_after = -1;  // moe_debug_stall
};
extern Tuning g_tuning;

struct Plan {
    int vpt, ncw, rows, stages, ctas_per_sm;
    int split, hl;  // CTAs per token (cluster size) and the columns each handles
    SmemLayout smem;
};

constexpr int kMaxSplit = 16;
constexpr int kMaxSplitCols = 4096;  // a slice fits 16 consumer warps at one vector each

// Whether `c` CTAs can share a row of H: equal slices that hold whole quant
// blocks and at most kMaxSplitCols columns.
inline bool split_ok(int32_t H, int32_t quant, int c)
{
    const int blk = quant == MOE_QUANT_NVFP4 ? 16 : (quant == MOE_QUANT_NONE ? 8 : 32);
    return c >= 2 && c <= kMaxSplit && H % (c * blk) == 0 && H / c <= kMaxSplitCols;
}

// CTAs per token.  moe_tuning_set may ask for a cluster size (or 1, whole
// rows); otherwise small batches split their rows over a thread-block cluster
// while every CTA of it finds an SM of its own and keeps a slice of at least
// 1792 columns: 4 CTAs a token up to sms / 4 tokens, 2 up to sms / 2; whole
// rows otherwise.  Measured on GB300 (graphs of 50 launches, k = 8):
//   H = 7168, residual + norm, bf16 out: T = 1: 4.34 us whole, 3.74 in 4s;
//     T = 38: 4.42, 4.14 in 4s; T = 64: 4.47, 4.42 in pairs; T = 100: 4.59
//     whole, 8.11 in pairs (more clusters than SMs);
//   H = 7168, shared + residual + norm + MXFP8: T = 1: 5.45, 4.04 in 4s;
//     T = 64: 5.61, 4.75 in pairs;
//   H = 4096, NVFP4: no gain past T = 8 (T = 64: 4.30 whole, 4.42 in pairs).
// A split token's CTAs each stage and sum a slice of every row, which halves
// or quarters one SM's copy intake and consumer work; the slices' sums of
// squares cost one exchange through distributed shared memory.
inline int choose_split(int32_t H, int64_t T, int32_t quant, int forced)
{
    if (forced >= 2)
        return split_ok(H, quant, forced) ? forced : 1;
    if (forced == 1)
        return 1;
    const int64_t sms = sm_count();
    if (T * 4 <= sms && H / 4 >= 1792 && split_ok(H, quant, 4))
        return 4;
    if (T * 2 <= sms && H / 2 >= 3584 && split_ok(H, quant, 2))
        return 2;
    return 1;
}

// Whole rows (split 1): vectors per consumer thread, the smallest of 1, 2,
// 4, 8 that needs at most 16 consumer warps.  Measured on GB300: at H = 7168,
// 14 warps x 2 vectors reach 93 % of HBM copy bandwidth against 73 % for 7
// warps x 4 (latency-bound) and 80 % for 28 warps x 1 (per-row overhead); at
// H = 4096, 16 warps x 1 beat 8 x 2.  Rows per ring slot: the fewest slots
// per token that leave room for three slots (measured, Gemma NVFP4 at
// H = 4096, 9 rows a token: one slot of 9 rows 0.93 of copy bandwidth, two of
// 5 + 4 rows 0.85, three of 3 rows 0.78, 8-row slots with only two in the
// ring 0.79; prefill at H = 7168, 10 rows: two slots of 5 rows 0.99).  Ring:
// about kDefaultRingBytes of rows, at least 3 slots where they fit, within
// the shared-memory budget.
// Split rows (when requested): one vector per thread over the H / split
// columns, and a ring that holds a whole token, so that the producer never
// waits inside a token and several CTAs fit on one SM.
inline Plan make_plan(int32_t H, int64_t T, int32_t rows_per_token, int32_t quant, bool with_gamma,
                      int split_request)
{
    const Tuning tu = g_tuning;
    Plan pl{};
    pl.split = choose_split(H, T, quant, split_request);
    pl.hl = H / pl.split;
    const int nvec = pl.hl / 8;
    auto covers = [&](int v) { return (nvec + 32 * v - 1) / (32 * v) <= max_consumer_warps_rt(v); };
    pl.vpt = 8;
    if (pl.split > 1) {
        pl.vpt = 1;
    } else if (tu.vpt && covers(tu.vpt)) {
        pl.vpt = tu.vpt;
    } else {
        for (int v : {1, 2, 4, 8}) {
            if (covers(v) && (nvec + 32 * v - 1) / (32 * v) <= 16) {
                pl.vpt = v;
                break;
            }
        }
    }
    pl.ncw = (nvec + 32 * pl.vpt - 1) / (32 * pl.vpt);
    pl.ctas_per_sm = tu.ctas_per_sm ? tu.ctas_per_sm : 1;
    // one CTA keeps kSmemBudget; several share the SM's 228 KB (1 KB reserved each)
    const size_t budget = pl.ctas_per_sm == 1 ? kSmemBudget : (224 * 1024) / pl.ctas_per_sm - 2048;
    if (tu.rows) {
        pl.rows = tu.rows < kMaxSlotRows ? tu.rows : kMaxSlotRows;
    } else {
        // as few slots per token as still leave room for three slots in the
        // ring: each slot costs the consumers a wait and a release, and
        // three let the producer stay a slot ahead of the one being summed
        // (with one token per CTA, a single slot holding the whole token was
        // measured slower: 4.9 against 4.7 us at T = 64, H = 7168, since the
        // consumers then wait for every row before summing the first)
        pl.rows = 1;
        for (int ns = 1; ns <= rows_per_token; ++ns) {
            const int r = (rows_per_token + ns - 1) / ns;
            if (r <= kMaxSlotRows && smem_layout(pl.hl, 3, r, pl.ncw, pl.split, with_gamma).total <= budget) {
                pl.rows = r;
                break;
            }
        }
    }
    // fewer rows per slot where two slots would not fit
    SmemLayout one = smem_layout(pl.hl, 1, pl.rows, pl.ncw, pl.split, with_gamma);
    while (pl.rows > 1 && one.total + one.slot_stride + 16 + sizeof(StageMeta) > budget) {
        --pl.rows;
        one = smem_layout(pl.hl, 1, pl.rows, pl.ncw, pl.split, with_gamma);
    }
    const size_t per_slot = one.slot_stride + 16 + sizeof(StageMeta);
    const size_t fixed = one.total - per_slot;
    int s;
    if (tu.ring_kib) {
        s = static_cast<int>((static_cast<size_t>(tu.ring_kib) * 1024 + one.slot_stride / 2) / one.slot_stride);
    } else if (pl.split > 1) {
        s = (rows_per_token + pl.rows - 1) / pl.rows;
    } else {
        s = static_cast<int>((kDefaultRingBytes + one.slot_stride / 2) / one.slot_stride);
        s = s < 3 ? 3 : s;
    }
    const int fit = budget > fixed ? static_cast<int>((budget - fixed) / per_slot) : 0;
    s = s > fit ? fit : s;
    s = s > kMaxStages ? kMaxStages : s;
    pl.stages = s < 2 ? 2 : s;
    pl.smem = smem_layout(pl.hl, pl.stages, pl.rows, pl.ncw, pl.split, with_gamma);
    return pl;
}

template <int VPT, int QUANT, int IO, bool SPLIT>
moe_status launch_t(const Params &p, const Plan &pl, cudaStream_t stream)
{
    auto kern = combine_kernel<VPT, QUANT, IO, SPLIT>;
    static SmemLimit smem_limit;  // per instantiation
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return MOE_ERR_CUDA;
    const int need = static_cast<int>(pl.smem.total);
    if (need > 227 * 1024)
        return MOE_ERR_UNSUPPORTED;
    if (ensure_dynamic_smem(kern, dev, need, smem_limit) != cudaSuccess ||
        (SPLIT && cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess)) {
        cudaGetLastError();
        return MOE_ERR_CUDA;
    }
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(pl.split);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    // programmatic dependent launch: the kernel may be scheduled while the
    // previous kernel on the stream finishes; it waits for it before reading
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.blockDim = dim3((pl.ncw + 1) * 32);
    cfg.dynamicSmemBytes = pl.smem.total;
    cfg.stream = stream;
    if (SPLIT) {
        // a cluster that no GPC can hold is reported as unsupported (the
        // caller then falls back to whole rows); the answer is kept per
        // device, cluster size and shared-memory size
        static int fits_split[64][5], fits_smem[64][5];
        static std::mutex fits_mu;
        std::lock_guard<std::mutex> guard(fits_mu);
        int li = 0;
        while ((2 << li) < pl.split)
            ++li;
        if (dev < 0 || dev >= 64 || fits_smem[dev][li] != need) {
            cfg.gridDim = dim3(static_cast<unsigned>(pl.split));
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            int n = 0;
            if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
                cudaGetLastError();
                n = 0;
            }
            if (dev < 0 || dev >= 64) {
                if (n < 1)
                    return MOE_ERR_UNSUPPORTED;
            } else {
                fits_split[dev][li] = n;
                fits_smem[dev][li] = need;
            }
        }
        if (dev >= 0 && dev < 64 && fits_split[dev][li] < 1)
            return MOE_ERR_UNSUPPORTED;
    }
    const int64_t sms = sm_count();
    if (sms <= 0)
        return MOE_ERR_CUDA;
    int64_t grid;
    if (SPLIT) {
        // one cluster per token, up to four clusters' worth of CTAs per SM;
        // clusters never wait on one another, so any that do not fit at
        // once simply start later
        const int64_t most = (4 * sms) / pl.split;
        grid = (p.T < most ? p.T : most) * pl.split;
    } else {
        const int64_t ctas = sms * pl.ctas_per_sm;
        grid = p.T < ctas ? p.T : ctas;
    }
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.attrs = SPLIT ? attr : attr + 1;
    cfg.numAttrs = SPLIT ? 2 : 1;
    if (cudaLaunchKernelEx(&cfg, kern, p) != cudaSuccess) {
        cudaGetLastError();
        return MOE_ERR_CUDA;
    }
    return MOE_OK;
}

template <int QUANT, int IO>
moe_status launch_q(const Params &p, const Plan &pl, cudaStream_t stream)
{
    if (pl.split > 1)
        return launch_t<1, QUANT, IO, true>(p, pl, stream);
    switch (pl.vpt) {
    case 1: return launch_t<1, QUANT, IO, false>(p, pl, stream);
    case 2: return launch_t<2, QUANT, IO, false>(p, pl, stream);
    case 4: return launch_t<4, QUANT, IO, false>(p, pl, stream);
    default: return launch_t<8, QUANT, IO, false>(p, pl, stream);
    }
}

// Every kernel of one I/O form; each form is compiled in its own translation
// unit (combine.cu: bf16, combine_f16.cu: fp16, combine_f16w.cu: fp16 with
// fp16 router weights).
template <int IO>
moe_status launch_io(const Params &p, const Plan &pl, int32_t quant, cudaStream_t stream)
{
    switch (quant) {
    case MOE_QUANT_MXFP8: return launch_q<MOE_QUANT_MXFP8, IO>(p, pl, stream);
    case MOE_QUANT_NVFP4: return launch_q<MOE_QUANT_NVFP4, IO>(p, pl, stream);
    case MOE_QUANT_MXFP4: return launch_q<MOE_QUANT_MXFP4, IO>(p, pl, stream);
    default: return launch_q<MOE_QUANT_NONE, IO>(p, pl, stream);
    }
}

} // namespace combine_detail
} // namespace nqg
