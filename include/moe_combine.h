/*
 * moe_combine.h -- C ABI of the single-GPU MoE combine/finalize step
 * (GB300, sm_103a).
 *
 * The library turns per-expert output rows, stored grouped by expert, back
 * into per-token hidden states:
 *
 *   routing build   topk_ids [T, k] -> counts [E], offsets [E+1],
 *                   row_map [T, k], src_row [N_valid]
 *   combine         s[t]  = sum_j w[t, j] * expert_out[row_map[t, j]]  (fp32, ascending j)
 *                           + shared_out[t]                             (optional, weight 1)
 *                   x[t]  = s[t] + residual[t]                          (optional)
 *                   y[t]  = x[t] / sqrt(mean(x[t]^2) + eps) * (gamma + weight_bias)  (optional)
 *                   quant = MXFP8 (e4m3, UE8M0 per 32) or NVFP4 (e2m1, e4m3 per 16,
 *                           global scale g) of y, scales linear or 128x4-swizzled
 *
 * Sources (page title -- section):
 *  - Struct_ep_combine_skip_a2a -- execute: weighted sum of routed expert
 *    outputs per token; args router_weights [num_tokens, top_k], topk_ids
 *    [num_tokens, top_k], src_info (originating token of each received row),
 *    recv_count_ptrs (tokens received per expert); parameter
 *    fused_shared_expert (adds the shared expert's output); parameter
 *    has_epilogue_fusion (elementwise epilogue after the combined output).
 *  - flashinfer.megamoe.nvfp4_mega_moe -- parameters num_tokens (padding
 *    rows are routed to -1), cumulative_local_expert_recv_stats (int32
 *    receive count per expert), y (caller-owned output, first num_tokens
 *    rows written in place); Notes (contiguous tensors on the device).
 *  - flashinfer.comm.trtllm_moe_allreduce_fusion -- residual_in,
 *    residual_out, rms_gamma, rms_eps, weight_bias (None -> 0.0, 1.0 -> the
 *    Gemma form (1 + gamma)), scale_factor, norm_out, quant_out, scale_out,
 *    layout_code; each output tensor is optional.
 *  - flashinfer.comm.moe_a2a_combine -- output_dtype (bf16 or
 *    float8_e4m3fn), output_scales (UE8M0 in uint8, vector size 32),
 *    output_scalar_scale (per-tensor global scale applied before FP4 block
 *    scaling), sf_layout (linear by default, or swizzled), output
 *    (caller-provided, contiguous, same device).
 *
 * Conventions for every entry point:
 *  - Pointers named "device" are CUDA device pointers owned by the caller;
 *    the library allocates nothing and keeps no state between calls.
 *  - All work is enqueued on `stream` (a cudaStream_t; NULL is the legacy
 *    default stream) and returns without synchronising, except
 *    moe_build_row_map_check, which synchronises `stream`.
 *  - Stream order holds as for any kernel.  The combine, the dispatch
 *    permute and the single-launch routing builds are launched with
 *    programmatic dependent launch: they may be scheduled while the previous
 *    kernel on `stream` is still running, but they read and write global
 *    memory only after it has completed and its writes are visible.
 *  - Arguments are validated on the host before anything is launched; an
 *    invalid call returns an error status and enqueues nothing.
 *  - A failed kernel launch returns MOE_ERR_CUDA.
 *  - Inputs must be finite (no NaN / Inf); they are not checked.
 */
#ifndef MOE_COMBINE_H
#define MOE_COMBINE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MOE_ABI_VERSION 4

/* Limits of this implementation (validated on the host). */
#define MOE_MAX_TOP_K 32
#define MOE_MAX_EXPERTS 8192
#define MOE_MAX_HIDDEN 16384

/* cudaStream_t without including the CUDA headers (same type). */
typedef struct CUstream_st *moe_stream_t;

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,    /* null / misaligned pointer, bad size or enum */
    MOE_ERR_UNSUPPORTED = 2,    /* valid request outside this library's limits */
    MOE_ERR_WORKSPACE = 3,      /* workspace missing or too small */
    MOE_ERR_INVALID_EXPERT = 4, /* a topk id outside [-1, E) (device-detected) */
    MOE_ERR_CUDA = 5,           /* a CUDA runtime call or launch failed */
    MOE_ERR_ROW_OUT_OF_RANGE = 6, /* a row_map entry >= n_expert_rows (device-detected) */
    MOE_ERR_DEVICE_TIMEOUT = 7  /* a bounded device-side wait gave up (device-detected) */
} moe_status;

typedef enum {
    MOE_QUANT_NONE = 0,
    MOE_QUANT_MXFP8 = 1, /* e4m3 codes [T, H] bytes + UE8M0 scale per 32 elements */
    MOE_QUANT_NVFP4 = 2, /* e2m1 codes [T, H/2] bytes (element 2i in the low nibble)
                            + e4m3 scale s = e4m3(amax(g * y) / 6) per 16 elements,
                            with global scale g; code = e2m1 of the quotient
                            (g * y) / s, correctly rounded to fp32 */
    MOE_QUANT_MXFP4 = 3  /* e2m1 codes [T, H/2] bytes (element 2i in the low nibble)
                            + UE8M0 scale per 32 elements: the smallest e with
                            amax <= 6 * 2^e, biased by 127 (global_scale ignored) */
} moe_quant_kind;

/* Element type of every 16-bit tensor of a combine call: expert_out,
 * shared_out, residual, gamma and the combined / residual / norm outputs
 * (Struct_ep_combine_skip_a2a -- combine_dtype; trtllm_moe_allreduce_fusion --
 * "fp16/bf16 -> fp4"). */
typedef enum {
    MOE_IO_BF16 = 0,
    MOE_IO_FP16 = 1
} moe_io_dtype;

/* Element type of router_weights (Struct_ep_combine_skip_a2a --
 * router_weights_dtype); weights are widened to fp32 exactly.  fp16 weights
 * with fp16 I/O take a kernel that multiplies the fp16 row elements by the
 * fp16 weight directly (the product is exact in fp32): the same results. */
typedef enum {
    MOE_WEIGHTS_FP32 = 0,
    MOE_WEIGHTS_BF16 = 1,
    MOE_WEIGHTS_FP16 = 2
} moe_weight_dtype;

typedef enum {
    MOE_LAYOUT_GROUPED = 0,    /* expert_out rows grouped by expert; row_map[t, j] gives
                                  the row of (token t, slot j), -1 = padded slot */
    MOE_LAYOUT_SLOT_MAJOR = 1  /* expert_out is [top_k, T, H]: slot j of token t is row
                                  j * T + t, every slot present, row_map unused
                                  (trtllm_moe_allreduce_fusion --
                                  moe_reduction_active_experts_token_input, with
                                  moe_reduction_scale_input as router_weights and
                                  moe_reduction_token_input as shared_out) */
} moe_expert_layout;

typedef enum {
    MOE_SF_LINEAR = 0,         /* scale (row r, column c) at byte r*C + c */
    MOE_SF_SWIZZLED_128x4 = 1  /* 128-row x 4-column tiles of 512 bytes, tiles in
                                  row-tile-major order, column tiles fastest; inside a
                                  tile (r%32)*16 + ((r%128)/32)*4 + c%4.  Rows padded
                                  to a multiple of 128, columns to a multiple of 4;
                                  the library writes the pad bytes as 0. */
} moe_sf_layout;

/* MOE_ABI_VERSION of the loaded library. */
int moe_abi_version(void);

/* A static, human-readable name for a moe_status value. */
const char *moe_status_string(int status);

/* sizeof(moe_combine_args) as compiled into the library (ABI check). */
size_t moe_combine_args_size(void);

/* ------------------------------------------------------------------------
 * Routing build (Struct_ep_combine_skip_a2a: topk_ids, src_info,
 * recv_count_ptrs; nvfp4_mega_moe: num_tokens padding with -1,
 * cumulative_local_expert_recv_stats).
 *
 * Given topk_ids (int32, [T, top_k] row-major, device), computes
 *   counts[e]    number of slots routed to expert e              int32 [E]
 *   offsets[e]   sum of counts[e'] for e' < e; offsets[E] = N_valid  int32 [E+1]
 *   row_map[t,j] row of the expert-grouped buffer holding token t's output
 *                from slot j: offsets[e] + the number of earlier slots
 *                (t', j') < (t, j), in row-major order, routed to the same
 *                expert e; -1 for a padded slot                    int32 [T, top_k]
 *   src_row[r]   t * top_k + j of the slot stored in row r, for r < N_valid
 *                (optional, NULL to skip; capacity T * top_k)     int32
 * The result is unique and deterministic (bit-identical across runs).
 * An id of -1 is padding.  Any other id outside [0, E) is treated as padding
 * too and recorded in the workspace's error word; moe_build_row_map_check
 * then returns MOE_ERR_INVALID_EXPERT.
 * All arrays are device memory.  `workspace` is caller-owned device memory of
 * at least moe_build_row_map_workspace_size(...) bytes, 16-byte aligned; it
 * must not be shared by calls that may overlap on the GPU.
 * Limits: 1 <= top_k <= MOE_MAX_TOP_K, 1 <= E <= MOE_MAX_EXPERTS,
 * T * top_k < 2^31.  T == 0 writes counts = 0 and offsets = 0.
 * ---------------------------------------------------------------------- */
moe_status moe_build_row_map_workspace_size(int64_t T, int32_t top_k, int32_t E,
                                            size_t *bytes);

moe_status moe_build_row_map(const int32_t *topk_ids, int64_t T, int32_t top_k, int32_t E,
                             int32_t *counts, int32_t *offsets, int32_t *row_map,
                             int32_t *src_row, void *workspace, size_t workspace_bytes,
                             moe_stream_t stream);

/* Synchronises `stream`, then reads the error word that the last
 * moe_build_row_map on `workspace` left there: MOE_OK or
 * MOE_ERR_INVALID_EXPERT (or MOE_ERR_CUDA if the read fails). */
moe_status moe_build_row_map_check(const void *workspace, moe_stream_t stream);

/* Kernels that moe_build_row_map(T, top_k, E) launches on the current device
 * with the current tuning: 1 (one thread-block cluster does the histogram,
 * scan and scatter), 3 (histogram, scan, scatter kernels over the
 * workspace) or 0 (T == 0: only memsets).  Launches nothing.  Returns
 * MOE_OK, MOE_ERR_INVALID_ARG or MOE_ERR_UNSUPPORTED as
 * moe_build_row_map_workspace_size does.  (No counterpart on the pages.) */
moe_status moe_build_row_map_launches(int64_t T, int32_t top_k, int32_t E, int32_t *launches);

/* ------------------------------------------------------------------------
 * Routing build without a workspace (no counterpart on the pages: an
 * addition of this library for callers that cannot allocate).
 *
 * Some callers cannot hand the library a workspace: plug-ins or extensions
 * running inside a host framework that owns all device memory through its
 * own allocator and offers them none, or latency-critical loops that may not
 * call cudaMalloc / cudaFree, because those calls can synchronise the device
 * or fail under memory pressure.  This entry point computes exactly what
 * moe_build_row_map computes (same outputs, bit for bit) but keeps its
 * scratch in a fixed array of MOE_NOALLOC_SCRATCH_BYTES bytes that the
 * library holds on every GPU where it is loaded, until the process exits.
 * It allocates nothing and calls no allocating routine.
 *
 *  - Limit: moe_build_row_map_workspace_size(T, top_k, E) must not exceed
 *    MOE_NOALLOC_SCRATCH_BYTES (1 MiB: for example T * top_k up to about one
 *    million slots with E = 256); larger problems return MOE_ERR_UNSUPPORTED.
 *  - The first call in each CUDA context looks up the array's device
 *    address there (cudaGetSymbolAddress, with that device current) and
 *    remembers it under the context's id; make that first call before any
 *    stream capture.  A context created later on the same device (after
 *    cudaDeviceReset, or a caller's own driver-API context) gets its own
 *    lookup on its first call.
 *  - All calls on a device share the one array, and it keeps whatever the
 *    last call left in it; every call rewrites the parts it reads.  Calls
 *    that may overlap on the GPU (different streams, or host threads) race
 *    on the array and must be serialised by the caller.
 *  - error_flag: device int32 or NULL.  When given it receives 0, or a
 *    nonzero value if an id outside [-1, E) was met (such ids are treated as
 *    padding, as in moe_build_row_map).
 * Other arguments, validation and return values as for moe_build_row_map.
 * ---------------------------------------------------------------------- */
#define MOE_NOALLOC_SCRATCH_BYTES (1u << 20)

moe_status moe_build_row_map_noalloc(const int32_t *topk_ids, int64_t T, int32_t top_k, int32_t E,
                                     int32_t *counts, int32_t *offsets, int32_t *row_map,
                                     int32_t *src_row, int32_t *error_flag, moe_stream_t stream);

/* ------------------------------------------------------------------------
 * Combine + residual + RMSNorm + quantisation, one call.
 * ---------------------------------------------------------------------- */
typedef struct moe_combine_args {
    int64_t T;                    /* tokens (rows of every [T, *] tensor); 0 = no-op */
    int32_t H;                    /* hidden size; multiple of 8, <= MOE_MAX_HIDDEN */
    int32_t top_k;                /* slots per token, 1..MOE_MAX_TOP_K */
    const void *expert_out;       /* device [n_expert_rows, H] (io_dtype): grouped by expert,
                                     or [top_k, T, H] slot-major (see expert_layout) */
    int64_t n_expert_rows;        /* rows in expert_out (row_map entries must be below;
                                     exactly top_k * T for the slot-major layout) */
    const int32_t *row_map;       /* device int32 [T, top_k], -1 = padded slot; unused
                                     (may be NULL) for the slot-major layout */
    const void *router_weights;   /* device [T, top_k] (weight_dtype), used as given */
    const void *shared_out;       /* device [T, H] (io_dtype) or NULL: shared-expert row, weight 1 */
    const void *residual;         /* device [T, H] (io_dtype) or NULL */
    const void *gamma;            /* device [H] (io_dtype) or NULL = no RMSNorm */
    float eps;                    /* RMSNorm epsilon, >= 0, inside the square root */
    float weight_bias;            /* added to gamma: 0 standard, 1 Gemma form */
    int32_t quant;                /* moe_quant_kind */
    int32_t sf_layout;            /* moe_sf_layout (ignored when quant == NONE) */
    float global_scale;           /* NVFP4 g > 0: codes encode g * y (ignored otherwise) */
    int32_t expert_layout;        /* moe_expert_layout */
    void *combined_out;           /* device [T, H] (io_dtype) or NULL: s rounded */
    void *residual_out;           /* device [T, H] (io_dtype) or NULL: x rounded */
    void *norm_out;               /* device [T, H] (io_dtype) or NULL: y rounded; needs gamma */
    void *quant_out;              /* device uint8: [T, H] MXFP8 / [T, H/2] NVFP4, MXFP4; needs quant */
    void *scales_out;             /* device uint8, moe_scales_bytes(...) bytes; needs quant */
    int32_t *status;              /* device int32 or NULL: set to a nonzero moe_status
                                     if the kernel meets a row_map entry >= n_expert_rows
                                     (that slot is skipped) or a bounded wait gives up;
                                     the caller zeroes it beforehand */
    int32_t io_dtype;             /* moe_io_dtype (0: bf16) */
    int32_t weight_dtype;         /* moe_weight_dtype (0: fp32) */
} moe_combine_args;

/* Enqueues the combine on `stream`.
 * x is the unrounded fp32 sum; residual_out = bf16(x); the RMSNorm and the
 * quantiser read the unrounded x (or y), not a bf16 copy.  Without gamma
 * the quantiser reads x directly.  Without residual, x = s.
 * Padded tokens (all slots -1) are still written: s = shared (or 0).
 * Host-side validation, before any launch:
 *   args non-NULL; T >= 0; expert_layout in {GROUPED, SLOT_MAJOR};
 *   H % 8 == 0 and 8 <= H <= MOE_MAX_HIDDEN; 1 <= top_k <= MOE_MAX_TOP_K;
 *   T == 0 then returns MOE_OK without looking at any pointer (empty tensors
 *   may carry NULL); otherwise router_weights non-NULL; row_map non-NULL for
 *   the grouped layout; n_expert_rows == top_k * T < 2^31 for the slot-major one;
 *   expert_out non-NULL when n_expert_rows > 0; every bf16 / byte tensor
 *   pointer 16-byte aligned; at least one output requested;
 *   norm_out needs gamma; quant in {NONE, MXFP8, NVFP4, MXFP4}; MXFP8 and
 *   MXFP4 need H % 32 == 0, NVFP4 needs H % 16 == 0 and a finite
 *   global_scale > 0; io_dtype and weight_dtype valid (weights 4-byte
 *   aligned if fp32, 2-byte otherwise);
 *   quant needs quant_out and scales_out; sf_layout in {LINEAR, SWIZZLED}.
 * Returns MOE_OK (enqueued), MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED or
 * MOE_ERR_CUDA. */
moe_status moe_combine(const moe_combine_args *args, moe_stream_t stream);

/* Overrides the combine kernel's launch plan for the rest of the process
 * (performance only: every plan computes identical results).  Each argument
 * 0 restores the automatic choice:
 *   vpt            8-element vectors per consumer thread: 1, 2, 4 or 8
 *                  (ignored where it cannot cover H; at most 16, 16, 8, 8
 *                  consumer warps respectively, so 1 covers H <= 4096);
 *   rows_per_slot  most rows staged per ring slot, 1..12 (a token's rows are
 *                  spread evenly over as few slots as that allows; fewer
 *                  where two slots would not fit in shared memory);
 *   ring_kib       shared-memory ring size in KiB, 1..224 (capped to what fits);
 *   ctas_per_sm    resident CTAs per SM the grid is sized for, 1..4;
 *   route_cluster  routing build: 0 automatic, -1 the three-kernel path,
 *                  1..16 the largest thread-block cluster its single-launch
 *                  path may use;
 *   combine_split  CTAs that share one token's row, as a thread-block
 *                  cluster that splits the columns: 0 automatic (for
 *                  H >= 7168, 4 CTAs a token while T * 4 <= the SM count
 *                  and 2 while T * 2 <= the SM count; whole rows
 *                  otherwise), 1 never, 2, 4, 8 or 16
 *                  always where H allows it (slices of equal width holding
 *                  whole quant blocks, at most 4096 columns each; otherwise
 *                  whole rows).  vpt, rows_per_slot and ctas_per_sm apply
 *                  to whole rows only.
 * Not synchronised with calls in flight on other host threads.  Returns
 * MOE_OK or MOE_ERR_INVALID_ARG.  (No counterpart on the pages: a tuning
 * hook of this implementation.) */
moe_status moe_tuning_set(int32_t vpt, int32_t rows_per_slot, int32_t ring_kib, int32_t ctas_per_sm,
                          int32_t route_cluster, int32_t combine_split);

/* Test hook for failure detection, for the rest of the process: with
 * slots >= 0, CTA 0 of the combine stops staging rows after that many ring
 * slots, and CTA 0 of the dispatch permute stops loading token rows after
 * that many tokens, so that their bounded waits run out (about 2 s) and the
 * call records MOE_ERR_DEVICE_TIMEOUT in its status word; the other CTAs
 * finish normally.  Nothing faults, and the CUDA context stays usable.
 * -1 (the default) turns it off.  Returns MOE_OK or MOE_ERR_INVALID_ARG.
 * (No counterpart on the pages.) */
moe_status moe_debug_stall(int64_t slots);

/* ------------------------------------------------------------------------
 * Dispatch-side permute: the step before the expert computation, the
 * inverse of the combine's gather (flashinfer.comm.moe_a2a_combine: combine
 * is the inverse of moe_a2a_dispatch; Struct_ep_combine_skip_a2a: src_info).
 *
 * Copies token t's row x[t] (device bf16 [T, H]) to every row row_map[t, j]
 * >= 0 of x_grouped (device bf16 [n_rows, H]), so that x_grouped holds the
 * tokens grouped by expert in the order moe_build_row_map defines.  Rows no
 * slot names are not written.  H % 8 == 0, 8 <= H <= MOE_MAX_HIDDEN,
 * 1 <= top_k <= MOE_MAX_TOP_K; x and x_grouped 16-byte aligned.  A row_map
 * entry >= n_rows is skipped and reported in *status (device int32 or NULL,
 * zeroed by the caller) as MOE_ERR_ROW_OUT_OF_RANGE.  T == 0 is a no-op.
 * ---------------------------------------------------------------------- */
moe_status moe_dispatch_permute(const void *x, int64_t T, int32_t H, const int32_t *row_map,
                                int32_t top_k, void *x_grouped, int64_t n_rows, int32_t *status,
                                moe_stream_t stream);

/* Bytes of the scale matrix for T rows of H elements: linear T * C, swizzled
 * roundup(T, 128) * roundup(C, 4), with C = H / 32 (MXFP8, MXFP4) or H / 16
 * (NVFP4). */
moe_status moe_scales_bytes(int64_t T, int32_t H, int32_t quant, int32_t sf_layout,
                            size_t *bytes);

#ifdef __cplusplus
}
#endif

#endif /* MOE_COMBINE_H */
