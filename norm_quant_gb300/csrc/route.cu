// route.cu -- routing build: per-expert histogram, exclusive scan and stable
// scatter to row_map (Struct_ep_combine_skip_a2a: topk_ids, src_info,
// recv_count_ptrs; flashinfer.megamoe.nvfp4_mega_moe: num_tokens padding
// with -1 and cumulative_local_expert_recv_stats).
//
// The N = T * top_k slots are cut into chunks of kChunk consecutive slots,
// one warp per chunk:
//   K1 route_hist     hist[c][e] = slots of chunk c routed to e
//   K2 route_scan     counts[e] = sum_c hist[c][e]; offsets = exclusive scan
//                     of counts; base[c][e] = offsets[e] + sum_{c'<c} hist[c'][e]
//                     (written over hist)
//   K3 route_scatter  row_map[i] = base[c][e] + rank of slot i among the slots
//                     of chunk c before it with the same expert
// Ranks come from __match_any_sync over 32 slots at a time plus a running
// per-expert count in shared memory, so the result is deterministic and
// bit-exact: no atomics decide a position.  No kernel waits on another CTA.
//
// For N <= kFusedMaxSlots and E <= kFusedMaxExperts the three steps run as
// ONE launch (route_fused_kernel): a thread-block cluster of up to 16 CTAs
// (8 where 16 cannot be placed) of 32 warps, one chunk per warp.  Each warp
// counts its chunk into its own column of an expert-major shared histogram;
// each slot's rank inside its chunk comes from warp ballots over the bits of
// the expert ids (no atomics); one warp per 8 experts turns the columns into
// prefixes with shuffle scans and stores each per-expert total straight into
// every CTA's shared memory (distributed shared memory; a cluster barrier
// split around the first phase guarantees every CTA has started); one more
// cluster barrier makes the totals visible, and each CTA derives counts,
// offsets and its bases locally and scatters.  Batches of up to
// kSmallMaxSlots slots use one CTA of 8 warps instead (route_small_kernel).
// Cluster barriers are hardware barriers over co-scheduled CTAs, so nothing
// spins.
//
// Both single-launch kernels are launched as programmatic dependents of the
// previous kernel on the stream (typically the previous layer's combine,
// which reads the row_map this build overwrites, or the router that writes
// the ids).  They clear their shared histograms first and touch global
// memory only after grid_dependency_wait, which returns once that kernel has
// completed and its writes are visible; so their launch and set-up overlap
// its tail.  The three-kernel path is launched plainly.
#include <cstdint>
#include <cuda_runtime.h>

#include "common.h"
#include "ptx.cuh"

namespace nqg {
namespace {

constexpr int kChunk = 1024;           // slots per warp-chunk
constexpr int kPerLane = kChunk / 32;  // slots per lane per chunk
constexpr int kScanMaxGroups = 32;     // route_scan uses up to 32 warps
constexpr size_t kScanSmemBudget = 200 * 1024;

struct WorkspaceLayout {
    int64_t chunks;
    size_t hist_off, err_off, total;
};

WorkspaceLayout layout_for(int64_t N, int32_t E)
{
    WorkspaceLayout L;
    L.chunks = (N + kChunk - 1) / kChunk;
    L.err_off = 0;  // error word first, padded to 16 bytes
    L.hist_off = 16;
    L.total = L.hist_off + static_cast<size_t>(L.chunks) * static_cast<size_t>(E) * sizeof(int32_t);
    L.total = (L.total + 255) / 256 * 256;
    return L;
}

__device__ __forceinline__ uint32_t smem_addr(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

int warps_per_cta(int32_t E)
{
    int w = static_cast<int>((48 * 1024) / (static_cast<size_t>(E) * sizeof(int32_t)));
    return w < 1 ? 1 : (w > 8 ? 8 : w);
}

__global__ void route_hist_kernel(const int32_t *__restrict__ ids, int64_t N, int32_t E,
                                  int32_t *__restrict__ hist, int64_t chunks, int32_t *__restrict__ err)
{
    extern __shared__ int32_t sh[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t c = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + warp;
    if (c >= chunks)
        return;
    int32_t *h = sh + static_cast<size_t>(warp) * E;
    for (int e = lane; e < E; e += 32)
        h[e] = 0;
    __syncwarp();
    const int64_t base = c * kChunk;
    int32_t v[kPerLane];
#pragma unroll
    for (int it = 0; it < kPerLane; ++it) {
        const int64_t i = base + it * 32 + lane;
        v[it] = (i < N) ? __ldg(ids + i) : -1;
    }
    bool bad = false;
#pragma unroll
    for (int it = 0; it < kPerLane; ++it) {
        const int32_t e = v[it];
        if (e >= 0 && e < E)
            atomicAdd(&h[e], 1);
        else if (e != -1)
            bad = true;
    }
    __syncwarp();
    int32_t *out = hist + c * E;
    for (int e = lane; e < E; e += 32)
        out[e] = h[e];
    if (__any_sync(0xffffffffu, bad) && lane == 0)
        atomicOr(err, 1);
}

// Warps of route_scan: as many as fit the shared-memory budget, up to 32.
int scan_groups(int32_t E)
{
    const size_t tiles = (static_cast<size_t>(E) + 31) / 32;
    const size_t per_group = tiles * 32 * sizeof(int32_t);
    const size_t g = (kScanSmemBudget - (static_cast<size_t>(E) + 1) * sizeof(int32_t)) / per_group;
    return static_cast<int>(g < 1 ? 1 : (g > kScanMaxGroups ? kScanMaxGroups : g));
}

// One CTA of 32 * ngroups threads.  Thread (g, lane) with g = threadIdx.x / 32
// owns, for every tile of 32 experts, expert tile*32 + lane over the chunk
// range of group g.
__global__ void __launch_bounds__(kScanMaxGroups * 32) route_scan_kernel(int32_t *__restrict__ hist,
                                                                        int64_t chunks, int32_t E,
                                                                        int32_t *__restrict__ counts,
                                                                        int32_t *__restrict__ offsets)
{
    extern __shared__ int32_t sh[];
    const int g = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int ngroups = blockDim.x >> 5;
    const int tiles = (E + 31) / 32;
    const int64_t per = (chunks + ngroups - 1) / ngroups;
    const int64_t c0 = g * per, c1 = (c0 + per < chunks) ? c0 + per : chunks;
    int32_t *part = sh;                                             // [tiles][ngroups][32]
    int32_t *tot = sh + static_cast<size_t>(tiles) * ngroups * 32;  // [E + 1]

    // 1. per-(group, expert) sums of the group's chunks
    for (int tile = 0; tile < tiles; ++tile) {
        const int e = tile * 32 + lane;
        int32_t s = 0;
        if (e < E) {
#pragma unroll 8
            for (int64_t c = c0; c < c1; ++c)
                s += hist[c * E + e];
        }
        part[(tile * ngroups + g) * 32 + lane] = s;
    }
    __syncthreads();
    // 2. exclusive scan over groups per expert; expert totals
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        const int tile = e >> 5, l = e & 31;
        int32_t run = 0;
        for (int gg = 0; gg < ngroups; ++gg) {
            int32_t *p = &part[(tile * ngroups + gg) * 32 + l];
            const int32_t v = *p;
            *p = run;
            run += v;
        }
        tot[e] = run;
        counts[e] = run;
    }
    __syncthreads();
    // 3. exclusive scan over experts: each lane of warp 0 takes a contiguous
    //    range, then a warp scan of the range sums
    if (threadIdx.x < 32) {
        const int per_e = (E + 31) / 32;
        const int e0 = lane * per_e, e1 = (e0 + per_e < E) ? e0 + per_e : E;
        int32_t s = 0;
        for (int e = e0; e < e1; ++e)
            s += tot[e];
        int32_t incl = s;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int32_t o = __shfl_up_sync(0xffffffffu, incl, d);
            if (lane >= d)
                incl += o;
        }
        int32_t run = incl - s;
        for (int e = e0; e < e1; ++e) {
            const int32_t v = tot[e];
            tot[e] = run;
            offsets[e] = run;
            run += v;
        }
        if (lane == 31)
            offsets[E] = incl;
    }
    __syncthreads();
    // 4. base[c][e] = offsets[e] + group prefix + running sum inside the group
    for (int tile = 0; tile < tiles; ++tile) {
        const int e = tile * 32 + lane;
        if (e >= E)
            continue;
        int32_t run = tot[e] + part[(tile * ngroups + g) * 32 + lane];
        for (int64_t c = c0; c < c1; ++c) {
            const int32_t v = hist[c * E + e];
            hist[c * E + e] = run;
            run += v;
        }
    }
}

__global__ void route_scatter_kernel(const int32_t *__restrict__ ids, int64_t N, int32_t E,
                                     const int32_t *__restrict__ base, int64_t chunks,
                                     int32_t *__restrict__ row_map, int32_t *__restrict__ src_row)
{
    extern __shared__ int32_t sh[];
    allow_dependent_launch();  // the combine may start its setup now
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t c = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + warp;
    if (c >= chunks)
        return;
    int32_t *run = sh + static_cast<size_t>(warp) * E;
    const int32_t *b = base + c * E;
    for (int e = lane; e < E; e += 32)
        run[e] = b[e];
    const int64_t first = c * kChunk;
    int32_t v[kPerLane];
#pragma unroll
    for (int it = 0; it < kPerLane; ++it) {
        const int64_t i = first + it * 32 + lane;
        v[it] = (i < N) ? __ldg(ids + i) : -1;
    }
    __syncwarp();
    const uint32_t lt = (1u << lane) - 1u;
#pragma unroll
    for (int it = 0; it < kPerLane; ++it) {
        const int64_t i = first + it * 32 + lane;
        const int32_t e = v[it];
        const bool valid = (e >= 0) && (e < E);
        const uint32_t peers = __match_any_sync(0xffffffffu, valid ? e : -1);
        const int rank = __popc(peers & lt);
        if (valid) {
            const int32_t r = run[e] + rank;
            row_map[i] = r;
            if (src_row)
                src_row[r] = static_cast<int32_t>(i);
        } else if (i < N) {
            row_map[i] = -1;
        }
        __syncwarp();
        if (valid && rank == 0)
            run[e] += __popc(peers);
        __syncwarp();
    }
}


int g_route_cluster = 0;  // see set_route_cluster

constexpr int kFusedThreads = 1024;
constexpr int kFusedWarps = kFusedThreads / 32;
constexpr int kFusedMaxCtas = 16;                // non-portable cluster size where allowed
constexpr int kFusedMaxPerLane = 16;             // chunk <= 512 slots per warp
constexpr int64_t kFusedMaxSlots = int64_t(kFusedMaxCtas) * kFusedWarps * 32 * kFusedMaxPerLane;
constexpr int kFusedMaxExperts = 512;
constexpr int kHistPitch = kFusedWarps + 1;      // hist[e][w] at e * 33 + w: banks (e + w) % 32
constexpr int kScanIlp = 8;                      // experts scanned together by one warp

struct FusedPlan {
    int ctas, per_lane;  // cluster size; slots per lane (chunk = 32 * per_lane per warp)
    size_t smem;
};

size_t fused_smem(int32_t E)
{
    // hist[E][33] + all_tot[16][E] + base[E] + off[E + 1] + wsum[32] + the CTA's error flag
    // + the CTAs' flags (CTA 0)
    return (static_cast<size_t>(kHistPitch + kFusedMaxCtas + 2) * E + 1 + 32 + 1 + kFusedMaxCtas) *
           sizeof(int32_t);
}

__device__ __forceinline__ uint32_t cluster_ctarank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ void cluster_sync_all()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Stores v at the same shared-memory offset as `local` in CTA `rank`.
__device__ __forceinline__ void st_dsmem(int32_t *local, uint32_t rank, int32_t v)
{
    uint32_t remote;
    asm("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_addr(local)), "r"(rank));
    asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(remote), "r"(v) : "memory");
}

// Stores four int32 (16-byte aligned `local`) at the same offset in CTA `rank`.
__device__ __forceinline__ void st_dsmem_v4(int32_t *local, uint32_t rank, int32_t a, int32_t b, int32_t c,
                                            int32_t d)
{
    uint32_t remote;
    asm("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_addr(local)), "r"(rank));
    asm volatile("st.shared::cluster.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(remote), "r"(a), "r"(b), "r"(c), "r"(d)
                 : "memory");
}

// The two halves of a cluster barrier, for a thread that has work to do in
// between (arrive without ordering; wait with acquire).
__device__ __forceinline__ void cluster_arrive_relaxed()
{
    asm volatile("barrier.cluster.arrive.relaxed;" ::: "memory");
}

__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire;" ::: "memory"); }

// One cluster of gridDim.x CTAs (the whole grid), 32 warps each; warp w of
// CTA b owns the chunk of PL * 32 consecutive slots starting at
// (b * 32 + w) * PL * 32, taken 32 at a time in order.  Every thread
// reaches every barrier.
template <int PL>
__global__ void __launch_bounds__(kFusedThreads, 1)
    route_fused_kernel(const int32_t *__restrict__ ids, int64_t N, int32_t E, int32_t *__restrict__ counts,
                       int32_t *__restrict__ offsets, int32_t *__restrict__ row_map,
                       int32_t *__restrict__ src_row, int32_t *__restrict__ err)
{
    extern __shared__ int32_t sh[];
    int32_t *hist = sh;                                               // [E][33]: warp counts, then prefixes
    int32_t *all_tot = hist + static_cast<size_t>(kHistPitch) * E;    // [16][E]
    int32_t *base = all_tot + static_cast<size_t>(kFusedMaxCtas) * E;  // [E]: offsets + lower CTAs
    int32_t *off = base + E;                                          // [E + 1]
    int32_t *wsum = off + E + 1;                                      // [32]
    int32_t &cta_bad = wsum[32];                                      // an id outside [-1, E) seen here
    int32_t *flags = wsum + 33;                                       // [16]: each CTA's cta_bad (CTA 0)
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const int nctas = static_cast<int>(gridDim.x);
    const int64_t first = (static_cast<int64_t>(rank) * kFusedWarps + warp) * (PL * 32);
    const uint32_t lt = (1u << lane) - 1u;
    allow_dependent_launch();  // the combine may start its setup now
    // the CTAs push their totals into one another's shared memory later; a
    // cluster barrier split around phase 1 makes sure every CTA has started
    if (nctas > 1)
        cluster_arrive_relaxed();

    // 1. each warp counts its chunk into its own column of hist and ranks
    //    every slot among the earlier slots of the chunk with the same expert.
    //    Per 32 slots, a lane's peers (lanes holding the same expert) come
    //    from one ballot per bit of the expert id; its rank is the running
    //    count plus the peers below it, and the lowest peer alone advances
    //    the count (the column is this warp's, so no atomics are needed)
    for (int e = lane; e < E; e += 32)
        hist[e * kHistPitch + warp] = 0;
    grid_dependency_wait();  // nothing above touches global memory
    int32_t v[PL], rk[PL];
#pragma unroll
    for (int it = 0; it < PL; ++it) {
        const int64_t i = first + it * 32 + lane;
        v[it] = (i < N) ? __ldg(ids + i) : -1;
    }
    const int key_bits = 32 - __clz(E);  // ids 0..E-1 and the key E of an invalid slot
    __syncwarp();
    bool bad = false;
#pragma unroll
    for (int it = 0; it < PL; ++it) {
        const int32_t e = v[it];
        const bool valid = e >= 0 && e < E;
        bad |= !valid && e != -1;
        const uint32_t key = valid ? static_cast<uint32_t>(e) : static_cast<uint32_t>(E);
        uint32_t peers = 0xffffffffu;
        for (int b = 0; b < key_bits; ++b) {
            const bool bit = (key >> b) & 1u;
            const uint32_t on = __ballot_sync(0xffffffffu, bit);
            peers &= bit ? on : ~on;
        }
        rk[it] = valid ? hist[e * kHistPitch + warp] + __popc(peers & lt) : 0;
        __syncwarp();
        if (valid && (peers & lt) == 0)  // the lowest lane of the group
            hist[e * kHistPitch + warp] += __popc(peers);
        __syncwarp();
    }
    // whether any slot of this CTA held an id outside [-1, E); CTA 0 gathers
    // the CTAs' flags with their totals and writes the error word once, at
    // the end (a global store before a cluster barrier would make its
    // release wait for the store to reach L2)
    {
        const int32_t b = __syncthreads_or(bad ? 1 : 0);
        if (nctas > 1)
            cluster_wait();
        if (threadIdx.x == 0) {
            cta_bad = b;
            if (nctas > 1)
                st_dsmem(&flags[rank], 0, b);
            else
                flags[0] = b;
        }
    }
    // 2. per expert: exclusive prefix over the 32 warp columns (a shuffle
    //    scan, kScanIlp experts at a time per warp) and the CTA's total
    for (int e0 = warp * kScanIlp; e0 < E; e0 += kFusedWarps * kScanIlp) {
        int32_t x[kScanIlp], incl[kScanIlp];
#pragma unroll
        for (int q = 0; q < kScanIlp; ++q) {
            x[q] = (e0 + q < E) ? hist[(e0 + q) * kHistPitch + lane] : 0;
            incl[q] = x[q];
        }
#pragma unroll
        for (int d = 1; d < 32; d <<= 1)
#pragma unroll
            for (int q = 0; q < kScanIlp; ++q) {
                const int32_t o = __shfl_up_sync(0xffffffffu, incl[q], d);
                if (lane >= d)
                    incl[q] += o;
            }
        int32_t tot[kScanIlp];
#pragma unroll
        for (int q = 0; q < kScanIlp; ++q) {
            const int e = e0 + q;
            tot[q] = __shfl_sync(0xffffffffu, incl[q], 31);
            if (e < E)
                hist[e * kHistPitch + lane] = incl[q] - x[q];
        }
        // this CTA's totals go into row `rank` of every CTA's all_tot: lane
        // b stores them in CTA b, 16 bytes at a time where E allows
        if (nctas == 1) {
            if (lane == 0) {
#pragma unroll
                for (int q = 0; q < kScanIlp; ++q)
                    if (e0 + q < E)
                        all_tot[e0 + q] = tot[q];
            }
        } else if (lane < nctas) {
            int32_t *row = &all_tot[rank * E + e0];
            if (E % kScanIlp == 0) {
                st_dsmem_v4(row, static_cast<uint32_t>(lane), tot[0], tot[1], tot[2], tot[3]);
                st_dsmem_v4(row + 4, static_cast<uint32_t>(lane), tot[4], tot[5], tot[6], tot[7]);
            } else {
#pragma unroll
                for (int q = 0; q < kScanIlp; ++q)
                    if (e0 + q < E)
                        st_dsmem(row + q, static_cast<uint32_t>(lane), tot[q]);
            }
        }
    }
    // 3. one barrier makes every CTA's pushed totals and flags visible; no
    //    CTA touches another's shared memory after it.  A lone CTA needs only
    //    its own barrier.
    if (nctas > 1)
        cluster_sync_all();
    else
        __syncthreads();
    int32_t any_bad = 0;
    if (rank == 0 && warp == 0)
        any_bad = __any_sync(0xffffffffu, lane < nctas && flags[lane] != 0) ? 1 : 0;
    if (rank == 0 && threadIdx.x == 0)
        *err = any_bad;
    // 4. counts, exclusive scan over experts, this CTA's base per expert
    {
        const int per_t = (E + kFusedThreads - 1) / kFusedThreads;  // 1 for E <= 1024
        const int ea = threadIdx.x * per_t, eb = (ea + per_t < E) ? ea + per_t : E;
        int32_t s = 0;
        for (int e = ea; e < eb; ++e) {
            int32_t all = 0, before = 0;
            for (int b = 0; b < nctas; ++b) {
                const int32_t x = all_tot[b * E + e];
                all += x;
                before += (b < static_cast<int>(rank)) ? x : 0;
            }
            off[e] = all;      // the count, for now
            base[e] = before;  // lower CTAs' share, for now
            s += all;
        }
        int32_t incl = s;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int32_t o = __shfl_up_sync(0xffffffffu, incl, d);
            if (lane >= d)
                incl += o;
        }
        if (lane == 31)
            wsum[warp] = incl;
        __syncthreads();
        if (warp == 0) {
            const int32_t ws = wsum[lane];
            int32_t wi = ws;
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const int32_t o = __shfl_up_sync(0xffffffffu, wi, d);
                if (lane >= d)
                    wi += o;
            }
            wsum[lane] = wi - ws;  // exclusive prefix of warp sums
            if (lane == 31)
                off[E] = wi;
        }
        __syncthreads();
        int32_t run = wsum[warp] + incl - s;
        for (int e = ea; e < eb; ++e) {
            const int32_t c = off[e];
            if (rank == 0) {
                counts[e] = c;
                offsets[e] = run;
            }
            off[e] = run;
            base[e] += run;
            run += c;
        }
        if (rank == 0 && threadIdx.x == 0)
            offsets[E] = off[E];
    }
    __syncthreads();
    // 5. scatter: row = offsets + lower CTAs + lower warps + rank in the chunk
#pragma unroll
    for (int it = 0; it < PL; ++it) {
        const int64_t i = first + it * 32 + lane;
        const int32_t e = v[it];
        if (e >= 0 && e < E) {
            const int32_t row = base[e] + hist[e * kHistPitch + warp] + rk[it];
            row_map[i] = row;
            if (src_row)
                src_row[row] = static_cast<int32_t>(i);
        } else if (i < N) {
            row_map[i] = -1;
        }
    }
}

// Small builds (N <= kSmallMaxSlots, decode-sized batches): one CTA of 8
// warps, launched without a cluster.  Warp w owns the PL * 32 consecutive
// slots from w * PL * 32 and ranks them with ballots as above; one thread per
// expert turns the 8 warp columns into exclusive prefixes and the expert's
// count; a block scan over the experts gives the offsets.  The error word is
// written once, at the end.
constexpr int kSmallThreads = 256;
constexpr int kSmallWarps = kSmallThreads / 32;
constexpr int kSmallPitch = kSmallWarps + 1;  // hist[e][w] at e * 9 + w
constexpr int kSmallMaxPerLane = 8;  // measured: at 4096 slots (16 a lane) a 16-CTA cluster is faster
constexpr int64_t kSmallMaxSlots = int64_t(kSmallThreads) * kSmallMaxPerLane;
constexpr int kSmallMaxExperts = 1024;

size_t small_smem(int32_t E)
{
    // hist[E][9] + off[E] + wsum[8]
    return (static_cast<size_t>(kSmallPitch + 1) * E + kSmallWarps) * sizeof(int32_t);
}

template <int PL>
__global__ void __launch_bounds__(kSmallThreads, 1)
    route_small_kernel(const int32_t *__restrict__ ids, int64_t N, int32_t E, int32_t *__restrict__ counts,
                       int32_t *__restrict__ offsets, int32_t *__restrict__ row_map,
                       int32_t *__restrict__ src_row, int32_t *__restrict__ err)
{
    extern __shared__ int32_t sh[];
    int32_t *hist = sh;                            // [E][9]: warp counts, then prefixes
    int32_t *off = hist + static_cast<size_t>(kSmallPitch) * E;  // [E]: counts, then offsets
    int32_t *wsum = off + E;                       // [8]
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t first = static_cast<int64_t>(warp) * (PL * 32);
    const uint32_t lt = (1u << lane) - 1u;
    allow_dependent_launch();  // the combine may start its setup now

    // 1. ranks within each warp's slots, counts in the warp's column
    for (int e = lane; e < E; e += 32)
        hist[e * kSmallPitch + warp] = 0;
    grid_dependency_wait();  // nothing above touches global memory
    int32_t v[PL], rk[PL];
#pragma unroll
    for (int it = 0; it < PL; ++it) {
        const int64_t i = first + it * 32 + lane;
        v[it] = (i < N) ? __ldg(ids + i) : -1;
    }
    const int key_bits = 32 - __clz(E);
    __syncwarp();
    // the ballots of a lane's PL slots are independent, so they interleave
    bool bad = false;
    uint32_t key[PL], peers[PL];
#pragma unroll
    for (int it = 0; it < PL; ++it) {
        const int32_t e = v[it];
        const bool valid = e >= 0 && e < E;
        bad |= !valid && e != -1;
        key[it] = valid ? static_cast<uint32_t>(e) : static_cast<uint32_t>(E);
        peers[it] = 0xffffffffu;
    }
    for (int b = 0; b < key_bits; ++b) {
#pragma unroll
        for (int it = 0; it < PL; ++it) {
            const bool bit = (key[it] >> b) & 1u;
            const uint32_t on = __ballot_sync(0xffffffffu, bit);
            peers[it] &= bit ? on : ~on;
        }
    }
    // ranks and counts, slot by slot (the running count orders them)
#pragma unroll
    for (int it = 0; it < PL; ++it) {
        const int32_t e = v[it];
        const bool valid = e >= 0 && e < E;
        rk[it] = valid ? hist[e * kSmallPitch + warp] + __popc(peers[it] & lt) : 0;
        __syncwarp();
        if (valid && (peers[it] & lt) == 0)
            hist[e * kSmallPitch + warp] += __popc(peers[it]);
        __syncwarp();
    }
    const int32_t any_bad = __syncthreads_or(bad ? 1 : 0);

    // 2. per expert (a contiguous run of experts per thread): exclusive
    //    prefix over the warp columns, and the count
    const int per_t = (E + kSmallThreads - 1) / kSmallThreads;
    const int ea = tid * per_t, eb = (ea + per_t < E) ? ea + per_t : E;
    int32_t s = 0;
    for (int e = ea; e < eb; ++e) {
        int32_t c = 0;
#pragma unroll
        for (int w = 0; w < kSmallWarps; ++w) {
            const int32_t x = hist[e * kSmallPitch + w];
            hist[e * kSmallPitch + w] = c;
            c += x;
        }
        off[e] = c;
        s += c;
    }
    // 3. exclusive scan of the counts over the experts
    int32_t incl = s;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const int32_t o = __shfl_up_sync(0xffffffffu, incl, d);
        if (lane >= d)
            incl += o;
    }
    if (lane == 31)
        wsum[warp] = incl;
    __syncthreads();
    // every warp adds up the totals of the warps below it itself (8 reads of
    // shared memory instead of one more barrier)
    int32_t below = 0, total = 0;
#pragma unroll
    for (int w = 0; w < kSmallWarps; ++w) {
        const int32_t x = wsum[w];
        total += x;
        below += (w < warp) ? x : 0;
    }
    if (tid == 0) {
        offsets[E] = total;
        *err = any_bad;
    }
    int32_t run = below + incl - s;
    for (int e = ea; e < eb; ++e) {
        const int32_t c = off[e];
        counts[e] = c;
        offsets[e] = run;
        off[e] = run;
        run += c;
    }
    __syncthreads();
    // 4. scatter: row = offset + lower warps + rank
#pragma unroll
    for (int it = 0; it < PL; ++it) {
        const int64_t i = first + it * 32 + lane;
        const int32_t e = v[it];
        if (e >= 0 && e < E) {
            const int32_t row = off[e] + hist[e * kSmallPitch + warp] + rk[it];
            row_map[i] = row;
            if (src_row)
                src_row[row] = static_cast<int32_t>(i);
        } else if (i < N) {
            row_map[i] = -1;
        }
    }
}

using SmallFn = decltype(&route_small_kernel<1>);

// Slots per lane of the small build for N slots, or 0 where it does not
// apply (too many slots or experts, or a routing path chosen by tuning).
int small_plan(int64_t N, int32_t E)
{
    if (N > kSmallMaxSlots || E > kSmallMaxExperts || g_route_cluster != 0)
        return 0;
    int pl = 1;
    while (int64_t(kSmallThreads) * pl < N)
        pl *= 2;
    return pl;
}

SmallFn small_fn(int per_lane)
{
    switch (per_lane) {
    case 1: return route_small_kernel<1>;
    case 2: return route_small_kernel<2>;
    case 4: return route_small_kernel<4>;
    default: return route_small_kernel<8>;
    }
}

using FusedFn = void (*)(const int32_t *, int64_t, int32_t, int32_t *, int32_t *, int32_t *, int32_t *, int32_t *);

FusedFn fused_fn(int per_lane)
{
    switch (per_lane) {
    case 1: return route_fused_kernel<1>;
    case 2: return route_fused_kernel<2>;
    case 4: return route_fused_kernel<4>;
    case 8: return route_fused_kernel<8>;
    default: return route_fused_kernel<16>;
    }
}

// Whether one cluster of `ctas` CTAs with `smem` bytes can be placed on this
// device; cached per device, kernel, cluster size and 32 KiB smem bucket.
bool fused_fits(FusedFn fn, int per_lane, int ctas, size_t smem)
{
    // answers and attribute state, shared by host threads (static storage:
    // they start at zero)
    static std::atomic<signed char> cache[64][6][kFusedMaxCtas + 1][8];  // 0 unknown, 1 yes, -1 no
    static std::atomic<bool> attr_set[64][6];
    static std::mutex attr_mu;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return false;
    const int pl_idx = per_lane == 1 ? 0 : per_lane == 2 ? 1 : per_lane == 4 ? 2 : per_lane == 8 ? 3 : 4;
    const int bucket = static_cast<int>((smem + 32 * 1024 - 1) / (32 * 1024));
    if (bucket >= 8 || static_cast<size_t>(bucket) * 32 * 1024 > 227 * 1024)
        return false;
    std::atomic<signed char> &c = cache[dev][pl_idx][ctas][bucket];
    const signed char known = c.load(std::memory_order_acquire);
    if (known)
        return known > 0;
    if (!attr_set[dev][pl_idx].load(std::memory_order_acquire)) {
        std::lock_guard<std::mutex> guard(attr_mu);
        if (!attr_set[dev][pl_idx].load(std::memory_order_relaxed)) {
            if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024) != cudaSuccess ||
                cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess) {
                cudaGetLastError();
                return false;
            }
            attr_set[dev][pl_idx].store(true, std::memory_order_release);
        }
    }
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = ctas;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(ctas);
    cfg.blockDim = dim3(kFusedThreads);
    cfg.dynamicSmemBytes = static_cast<size_t>(bucket) * 32 * 1024;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    const bool ok = cudaOccupancyMaxActiveClusters(&n, reinterpret_cast<const void *>(fn), &cfg) == cudaSuccess && n > 0;
    cudaGetLastError();
    c.store(ok ? 1 : -1, std::memory_order_release);
    return ok;
}

// Cluster size and slots per lane: enough CTAs that each holds at most
// 32 * 32 * per_lane slots with the fewest slots per lane, preferring 16 CTAs
// (or 8 where 16 cannot be placed); per_lane a power of two up to 32.
bool fused_plan(int64_t N, int32_t E, FusedPlan *out)
{
    if (N > kFusedMaxSlots || E > kFusedMaxExperts || g_route_cluster < 0)
        return false;
    const size_t smem = fused_smem(E);
    for (int max_ctas : {16, 8}) {
        if (g_route_cluster > 0 && max_ctas > g_route_cluster)
            max_ctas = g_route_cluster;
        const int64_t per_cta_min = int64_t(kFusedWarps) * 32;  // one slot per lane
        int ctas = static_cast<int>((N + per_cta_min - 1) / per_cta_min);
        ctas = ctas < 1 ? 1 : (ctas > max_ctas ? max_ctas : ctas);
        int per_lane = 1;
        while (int64_t(ctas) * kFusedWarps * 32 * per_lane < N)
            per_lane *= 2;
        if (per_lane > kFusedMaxPerLane)
            continue;
        if (fused_fits(fused_fn(per_lane), per_lane, ctas, smem)) {
            *out = FusedPlan{ctas, per_lane, smem};
            return true;
        }
    }
    return false;
}
} // namespace

void set_route_cluster(int v) { g_route_cluster = v; }

} // namespace nqg

using namespace nqg;

extern "C" moe_status moe_build_row_map_workspace_size(int64_t T, int32_t top_k, int32_t E, size_t *bytes)
{
    if (!bytes || T < 0 || top_k < 1 || E < 1)
        return MOE_ERR_INVALID_ARG;
    if (top_k > MOE_MAX_TOP_K || E > MOE_MAX_EXPERTS || T * top_k >= (int64_t(1) << 31))
        return MOE_ERR_UNSUPPORTED;
    *bytes = layout_for(T * top_k, E).total;
    return MOE_OK;
}

extern "C" moe_status moe_build_row_map_launches(int64_t T, int32_t top_k, int32_t E, int32_t *launches)
{
    if (!launches || T < 0 || top_k < 1 || E < 1)
        return MOE_ERR_INVALID_ARG;
    if (top_k > MOE_MAX_TOP_K || E > MOE_MAX_EXPERTS || T * top_k >= (int64_t(1) << 31))
        return MOE_ERR_UNSUPPORTED;
    FusedPlan f;
    *launches = T == 0 ? 0 : ((small_plan(T * top_k, E) || fused_plan(T * top_k, E, &f)) ? 1 : 3);
    return MOE_OK;
}

extern "C" moe_status moe_build_row_map(const int32_t *topk_ids, int64_t T, int32_t top_k, int32_t E,
                                        int32_t *counts, int32_t *offsets, int32_t *row_map,
                                        int32_t *src_row, void *workspace, size_t workspace_bytes,
                                        moe_stream_t stream)
{
    if (T < 0 || top_k < 1 || E < 1 || !counts || !offsets)
        return MOE_ERR_INVALID_ARG;
    if (top_k > MOE_MAX_TOP_K || E > MOE_MAX_EXPERTS || T * top_k >= (int64_t(1) << 31))
        return MOE_ERR_UNSUPPORTED;
    if (T > 0 && (!topk_ids || !row_map))
        return MOE_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(topk_ids) | reinterpret_cast<uintptr_t>(counts) |
         reinterpret_cast<uintptr_t>(offsets) | reinterpret_cast<uintptr_t>(row_map) |
         reinterpret_cast<uintptr_t>(src_row)) & 3u)
        return MOE_ERR_INVALID_ARG;
    const int64_t N = T * top_k;
    const WorkspaceLayout L = layout_for(N, E);
    if (!workspace)
        return MOE_ERR_WORKSPACE;
    if (!aligned16(workspace))
        return MOE_ERR_INVALID_ARG;
    if (workspace_bytes < L.total)
        return MOE_ERR_WORKSPACE;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    char *ws = static_cast<char *>(workspace);
    int32_t *err = reinterpret_cast<int32_t *>(ws + L.err_off);
    int32_t *hist = reinterpret_cast<int32_t *>(ws + L.hist_off);
    if (N == 0) {
        if (cudaMemsetAsync(err, 0, sizeof(int32_t), s) != cudaSuccess ||
            cudaMemsetAsync(counts, 0, sizeof(int32_t) * E, s) != cudaSuccess ||
            cudaMemsetAsync(offsets, 0, sizeof(int32_t) * (E + 1), s) != cudaSuccess)
            return MOE_ERR_CUDA;
        return MOE_OK;
    }
    // the single-launch kernels go out as programmatic dependents (see the
    // top of this file); a cluster dimension is added for a fused cluster
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (const int pl = small_plan(N, E)) {
        cfg.gridDim = dim3(1);
        cfg.blockDim = dim3(kSmallThreads);
        cfg.dynamicSmemBytes = small_smem(E);
        if (cudaLaunchKernelEx(&cfg, small_fn(pl), topk_ids, N, E, counts, offsets, row_map, src_row, err) !=
            cudaSuccess) {
            cudaGetLastError();
            return MOE_ERR_CUDA;
        }
        return MOE_OK;
    }
    FusedPlan f;
    if (fused_plan(N, E, &f)) {
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = f.ctas;
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        cfg.gridDim = dim3(f.ctas);
        cfg.blockDim = dim3(kFusedThreads);
        cfg.dynamicSmemBytes = f.smem;
        cfg.numAttrs = f.ctas > 1 ? 2 : 1;  // a lone CTA is launched without a cluster
        if (cudaLaunchKernelEx(&cfg, fused_fn(f.per_lane), topk_ids, N, E, counts, offsets, row_map, src_row,
                               err) != cudaSuccess) {
            cudaGetLastError();
            return MOE_ERR_CUDA;
        }
        return MOE_OK;
    }
    if (cudaMemsetAsync(err, 0, sizeof(int32_t), s) != cudaSuccess)
        return MOE_ERR_CUDA;
    const int wpc = warps_per_cta(E);
    const int grid = static_cast<int>((L.chunks + wpc - 1) / wpc);
    const size_t sh = static_cast<size_t>(wpc) * E * sizeof(int32_t);
    route_hist_kernel<<<grid, wpc * 32, sh, s>>>(topk_ids, N, E, hist, L.chunks, err);
    const int tiles = (E + 31) / 32;
    const int groups = scan_groups(E);
    const size_t sh_scan = (static_cast<size_t>(tiles) * groups * 32 + E + 1) * sizeof(int32_t);
    if (sh_scan > 48 * 1024 &&
        cudaFuncSetAttribute(route_scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(sh_scan)) != cudaSuccess)
        return MOE_ERR_CUDA;
    route_scan_kernel<<<1, groups * 32, sh_scan, s>>>(hist, L.chunks, E, counts, offsets);
    route_scatter_kernel<<<grid, wpc * 32, sh, s>>>(topk_ids, N, E, hist, L.chunks, row_map, src_row);
    return launch_status();
}

extern "C" moe_status moe_build_row_map_check(const void *workspace, moe_stream_t stream)
{
    if (!workspace)
        return MOE_ERR_INVALID_ARG;
    int32_t err = 0;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (cudaMemcpyAsync(&err, workspace, sizeof(err), cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return MOE_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess)
        return MOE_ERR_CUDA;
    return err ? MOE_ERR_INVALID_EXPERT : MOE_OK;
}
