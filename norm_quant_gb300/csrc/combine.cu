// combine.cu -- the MoE combine/finalize kernel and its C entry points.
//
// What it computes (Struct_ep_combine_skip_a2a, execute: weighted sum of
// routed expert outputs; fused_shared_expert; flashinfer.comm.
// trtllm_moe_allreduce_fusion: residual_in/out, rms_gamma, rms_eps,
// weight_bias, norm_out, quant_out, scale_out, layout_code;
// flashinfer.comm.moe_a2a_combine: output_dtype float8_e4m3fn with UE8M0
// output_scales per 32, output_scalar_scale for NVFP4, sf_layout):
//
//   s = sum_j w[t,j] * expert_out[row_map[t,j]]  (fp32, ascending j) + shared[t]
//   x = s + residual[t]
//   y = x / sqrt(mean(x^2) + eps) * (gamma + weight_bias)
//   MXFP8: per 32 elements, e = smallest integer with amax <= 448 * 2^e,
//          byte = clamp(e + 127, 0, 254), code = e4m3_rn_sat(y * 2^-e)
//   NVFP4: v = g * y; per 16 elements s = e4m3_rn_sat(amax(v) / 6),
//          code = e2m1_rn_sat(rn(v / s)) (0 when s == 0)
//   MXFP4: per 32 elements, e = smallest integer with amax <= 6 * 2^e,
//          byte = clamp(e + 127, 0, 254), code = e2m1_rn_sat(y * 2^-e)
// Inputs and outputs are bf16 or fp16 (io_dtype); router weights fp32,
// bf16 or fp16 (weight_dtype); accumulation is fp32 throughout.  With fp16
// rows and fp16 weights each product is formed by a mixed-precision fma
// (fp16 x fp16 + fp32), which is exact, so the result is the same bits.
//
// Design (an HBM-bound gather; no tensor cores -- nothing here is a
// contraction):
//   * persistent CTAs, one per SM by default; token t goes to CTA t mod grid;
//   * one producer warp walks the CTA's tokens.  A token needs its valid
//     expert rows in ascending j, then the shared row, then the residual row;
//     they are spread evenly over as few slots of a shared-memory ring as the
//     slot capacity R (up to 12 rows) allows.  Lane q of the producer stages
//     row q of a slot: one cp.async.bulk of the 2H-byte row, completing on the
//     slot's "full" mbarrier, and the row's weight beside the slot; lane 0
//     then publishes the slot's count and flags and arms the barrier.
//     row_map / weights of the next token are prefetched meanwhile;
//   * consumer warps own 8-element vectors v = slot * NC + thread of the row;
//     per ring slot they wait once, then take its rows in register chunks
//     (all of a chunk's 16-byte shared loads, with its weights in one vector
//     load, before its sums), accumulate fp32 in row order, and release the
//     slot on its "empty" mbarrier;
//   * after a token's last slot: bf16 stores, a sum of squares reduced by
//     warp shuffles and a cross-warp sum at a named barrier of the
//     consumer warps, the norm (its scale 1 / sqrt(mean + eps) from rsqrt
//     refined by one Newton step, within one ulp of the correctly rounded
//     value), and the block quantiser (an MXFP8 block is 4 consecutive lanes,
//     NVFP4 2; NVFP4 elements divided by their block scale, the quotient
//     correctly rounded);
//   * for small batches, or on request (moe_tuning_set), a token is split by
//     columns over a thread-block cluster of 2..16 CTAs (each copies, sums,
//     normalises and quantises its own slice of every row); the slices' sums of squares
//     meet through distributed shared memory: each warp sends its partial to
//     every CTA of the cluster as an asynchronous store that completes on that
//     CTA's mbarrier, and each CTA adds the partials in one fixed order.  This
//     is the automatic plan for small batches (at H >= 7168, 4 CTAs a token
//     while T * 4 <= the SM count, 2 while T * 2 <= it), where it halves or
//     quarters one SM's copies and sums;
//   * gamma's slice is copied to shared memory once per CTA, and the
//     per-warp partial sums of squares are added by a butterfly that gives
//     every lane the same total.
// Every mbarrier wait is bounded (kWaitLimitNs); a wait that gives up records
// MOE_ERR_DEVICE_TIMEOUT and the CTA drains its own copies and finishes (a
// consumer warp that gives up first meets the others at the norm's barrier
// with an abort flag, so that none waits there forever).
#include <cstdint>
#include <cuda_runtime.h>

#include "combine_impl.cuh"

namespace nqg {
namespace combine_detail {

Tuning g_tuning;

// the fp16 kernels are instantiated in combine_f16.cu
extern template moe_status launch_io<1>(const Params &, const Plan &, int32_t, cudaStream_t);
extern template moe_status launch_io<2>(const Params &, const Plan &, int32_t, cudaStream_t);
template moe_status launch_io<0>(const Params &, const Plan &, int32_t, cudaStream_t);

} // namespace combine_detail
} // namespace nqg

using namespace nqg;
using namespace nqg::combine_detail;


extern "C" moe_status moe_tuning_set(int32_t vpt, int32_t rows_per_slot, int32_t ring_kib, int32_t ctas_per_sm,
                                     int32_t route_cluster, int32_t combine_split)
{
    if (route_cluster < -1 || route_cluster > 16)
        return MOE_ERR_INVALID_ARG;
    if (!(vpt == 0 || vpt == 1 || vpt == 2 || vpt == 4 || vpt == 8))
        return MOE_ERR_INVALID_ARG;
    if (rows_per_slot < 0 || rows_per_slot > kMaxSlotRows || ring_kib < 0 || ring_kib > 224 || ctas_per_sm < 0 ||
        ctas_per_sm > 4)
        return MOE_ERR_INVALID_ARG;
    if (!(combine_split == 0 || combine_split == 1 || combine_split == 2 || combine_split == 4 ||
          combine_split == 8 || combine_split == 16))
        return MOE_ERR_INVALID_ARG;
    nqg::set_route_cluster(route_cluster);
    g_tuning.vpt = vpt;
    g_tuning.rows = rows_per_slot;
    g_tuning.ring_kib = ring_kib;
    g_tuning.ctas_per_sm = ctas_per_sm;
    g_tuning.split = combine_split;
    return MOE_OK;
}

int64_t nqg::debug_stall_slots() { return g_tuning.stall_after; }

extern "C" moe_status moe_debug_stall(int64_t slots)
{
    if (slots < -1)
        return MOE_ERR_INVALID_ARG;
    g_tuning.stall_after = slots;
    return MOE_OK;
}

extern "C" moe_status moe_combine(const moe_combine_args *a, moe_stream_t stream)
{
    if (!a)
        return MOE_ERR_INVALID_ARG;
    if (a->T < 0 || (a->expert_layout != MOE_LAYOUT_GROUPED && a->expert_layout != MOE_LAYOUT_SLOT_MAJOR))
        return MOE_ERR_INVALID_ARG;
    if (a->H < 8 || a->H % 8 != 0 || a->top_k < 1)
        return MOE_ERR_INVALID_ARG;
    if (a->H > MOE_MAX_HIDDEN || a->top_k > MOE_MAX_TOP_K)
        return MOE_ERR_UNSUPPORTED;
    if (a->T == 0)
        return MOE_OK;  // an empty batch: empty tensors may carry NULL pointers
    const bool slot_major = a->expert_layout == MOE_LAYOUT_SLOT_MAJOR;
    if ((!slot_major && !a->row_map) || !a->router_weights || a->n_expert_rows < 0)
        return MOE_ERR_INVALID_ARG;
    if (slot_major && (a->n_expert_rows != a->T * a->top_k || a->T * a->top_k >= (int64_t(1) << 31)))
        return MOE_ERR_INVALID_ARG;
    if (a->n_expert_rows > 0 && !a->expert_out)
        return MOE_ERR_INVALID_ARG;
    if (a->quant != MOE_QUANT_NONE && a->quant != MOE_QUANT_MXFP8 && a->quant != MOE_QUANT_NVFP4 &&
        a->quant != MOE_QUANT_MXFP4)
        return MOE_ERR_INVALID_ARG;
    if ((a->io_dtype != MOE_IO_BF16 && a->io_dtype != MOE_IO_FP16) ||
        (a->weight_dtype != MOE_WEIGHTS_FP32 && a->weight_dtype != MOE_WEIGHTS_BF16 &&
         a->weight_dtype != MOE_WEIGHTS_FP16))
        return MOE_ERR_INVALID_ARG;
    if (a->quant != MOE_QUANT_NONE) {
        if (a->sf_layout != MOE_SF_LINEAR && a->sf_layout != MOE_SF_SWIZZLED_128x4)
            return MOE_ERR_INVALID_ARG;
        if (!a->quant_out || !a->scales_out)
            return MOE_ERR_INVALID_ARG;
        if ((a->quant == MOE_QUANT_MXFP8 || a->quant == MOE_QUANT_MXFP4) && a->H % 32 != 0)
            return MOE_ERR_INVALID_ARG;
        if (a->quant == MOE_QUANT_NVFP4 &&
            (a->H % 16 != 0 || !(a->global_scale > 0.f) || !(a->global_scale < 3.0e38f)))
            return MOE_ERR_INVALID_ARG;
    }
    if (a->norm_out && !a->gamma)
        return MOE_ERR_INVALID_ARG;
    if (!(a->eps >= 0.f) || !(a->eps < 3.0e38f) || !(a->weight_bias == a->weight_bias))
        return MOE_ERR_INVALID_ARG;
    if (!a->combined_out && !a->residual_out && !a->norm_out && a->quant == MOE_QUANT_NONE)
        return MOE_ERR_INVALID_ARG;
    const void *must16[] = {a->expert_out, a->shared_out, a->residual, a->gamma, a->combined_out,
                            a->residual_out, a->norm_out, a->quant_out};
    for (const void *q : must16)
        if (q && !aligned16(q))
            return MOE_ERR_INVALID_ARG;
    const uintptr_t walign = a->weight_dtype == MOE_WEIGHTS_FP32 ? 3u : 1u;
    if ((reinterpret_cast<uintptr_t>(a->row_map) & 3u) || (reinterpret_cast<uintptr_t>(a->router_weights) & walign) ||
        (reinterpret_cast<uintptr_t>(a->status) & 3u))
        return MOE_ERR_INVALID_ARG;

    Params p{};
    p.T = a->T;
    p.H = a->H;
    p.k = a->top_k;
    p.expert_out = static_cast<const uint8_t *>(a->expert_out);
    p.n_rows = a->n_expert_rows;
    p.row_map = slot_major ? nullptr : a->row_map;
    p.slot_major = slot_major ? 1 : 0;
    p.weights = a->router_weights;
    p.weight_dtype = a->weight_dtype;
    p.shared = static_cast<const uint8_t *>(a->shared_out);
    p.residual = static_cast<const uint8_t *>(a->residual);
    p.gamma = static_cast<const uint16_t *>(a->gamma);
    p.eps = a->eps;
    p.inv_h = 1.0f / static_cast<float>(a->H);
    p.wb = a->weight_bias;
    p.gscale = a->global_scale;
    p.sf_layout = a->sf_layout;
    p.combined_out = static_cast<uint16_t *>(a->combined_out);
    p.residual_out = static_cast<uint16_t *>(a->residual_out);
    p.norm_out = static_cast<uint16_t *>(a->norm_out);
    p.quant_out = static_cast<uint8_t *>(a->quant_out);
    p.scales_out = static_cast<uint8_t *>(a->scales_out);
    p.status = a->status;
    if (a->quant != MOE_QUANT_NONE) {
        p.sf_cols = a->H / (a->quant == MOE_QUANT_NVFP4 ? 16 : 32);
        p.sf_cols_pad = a->sf_layout == MOE_SF_LINEAR ? p.sf_cols : (p.sf_cols + 3) / 4 * 4;
        p.sf_rows_pad = a->sf_layout == MOE_SF_LINEAR ? p.T : (p.T + 127) / 128 * 128;
    }
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    auto launch = [&](const Plan &pl) {
        p.stages = pl.stages;
        p.rows = pl.rows;
        p.split = pl.split;
        p.hl = pl.hl;
        p.stall_after = g_tuning.stall_after;
        if (a->io_dtype == MOE_IO_BF16)
            return launch_io<0>(p, pl, a->quant, s);
        // fp16 rows with fp16 weights: products exact without widening the rows
        return a->weight_dtype == MOE_WEIGHTS_FP16 ? launch_io<2>(p, pl, a->quant, s)
                                                   : launch_io<1>(p, pl, a->quant, s);
    };
    // rows a token may need: its valid expert rows, the shared row, the residual row
    const int rows_per_token = a->top_k + (a->shared_out ? 1 : 0) + (a->residual ? 1 : 0);
    const bool with_gamma = a->gamma != nullptr;
    const Plan pl = make_plan(a->H, a->T, rows_per_token, a->quant, with_gamma, g_tuning.split);
    const moe_status st = launch(pl);
    if (st == MOE_ERR_UNSUPPORTED && pl.split > 1)  // no room for the cluster: whole rows
        return launch(make_plan(a->H, a->T, rows_per_token, a->quant, with_gamma, 1));
    return st;
}
