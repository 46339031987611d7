/*
 * moe.h -- C ABI of a GB300 (sm_103a) sparse Mixture-of-Experts expert layer.
 *
 * One layer call runs, on one CUDA stream of one GPU:
 *   router matmul -> top-k gating (softmax or sigmoid scoring, optional group
 *   stage, zero-computation experts) -> stable re-sort of the token picks by
 *   expert -> grouped SwiGLU expert FFN (GEMV-style streaming for lightly loaded
 *   experts, tensor-core tiles for loaded ones) -> weighted combine, plus an
 *   optional always-on shared expert.
 *
 * Sources (web pages; cited by title and section):
 *  [LC-A3]   "基于Atlas 900 A3 SuperPoD的LongCat-Flash模型推理性能优化实践",
 *            section 背景介绍 (zero-computation experts: a token routed to one
 *            passes through unchanged) and section 优化措施三：权重预取 (Router
 *            Matmul, QuantBatchMatmul).
 *  [LC-CANN] "LongCat-Flash与GLM-4.6V，昇腾CANN异构计算深水区突围详解",
 *            section 拆解MoE困局 (768 experts = 512 routed + 256 zero-computation;
 *            token dispatch and combine).
 *  [PANGU]   "华为技术披露集 VOL.12：昇腾×盘古" (Pangu Pro MoE), opening section
 *            (grouped experts, MoGE), section 分层混合并行（H2P） (grouped routed
 *            experts, shared expert) and section SwiftGMM (grouped expert matmul
 *            that switches between GEMV and GEMM by load).
 *  [DS-ASC]  DeepSeek-V3/R1 on Ascend (Huxiu article): deployment paragraph
 *            (routed experts + 1 shared expert), section "2. 模型侧并发优化"
 *            (quantised activations sent with their scales), section
 *            "2. MOE 算子优化" (InitialRouting re-sorts tokens by expert).
 *
 * Conventions for every entry point
 *  - All tensor pointers are DEVICE pointers owned by the caller, row-major,
 *    16-byte aligned (MOE_ERR_ALIGNMENT otherwise).  The library never
 *    allocates or frees device memory and never synchronises the stream, except
 *    moe_check_device_status and moe_timing_collect, which say so.
 *  - Work is enqueued asynchronously on `stream` (a cudaStream_t; NULL = legacy
 *    default stream).  Calls keep no state between them; concurrent calls on
 *    different streams need different workspaces.
 *  - The library's kernels are launched with programmatic dependent launch: each
 *    may be scheduled while the kernel before it on the stream is finishing, and
 *    waits for that kernel to complete before it reads or writes device memory,
 *    so results and stream order are those of plain launches.  The environment
 *    variable MOE_PDL=0, read once per process, turns this off.
 *  - Small-batch routing runs its matmul on tensor cores where the batch gives
 *    enough parallel work; MOE_ROUTER_TC=0 (read once) keeps it on CUDA cores.
 *    The smallest layers (T x (E_r + E_z) x H at most 2^20 multiply-adds, x and
 *    w_router within one CTA's shared memory) route in one CTA on CUDA cores,
 *    inside moe_layer_forward's re-sort kernel unless MOE_FOLDS=0.  All paths
 *    compute fp32-class logits (routing ids do not depend on the choice beyond
 *    ties closer than the logits' rounding).
 *  - bf16 tensors are passed as `const void*` holding IEEE bfloat16 values.
 *  - Expert indices 0 .. n_routed-1 are FFN experts; n_routed .. n_routed+n_zero-1
 *    are zero-computation experts (no weights; their pick contributes w * x_t).
 *  - Host-detectable errors return a status before anything is enqueued.  Data
 *    errors found on the device (an expert id out of range, a bounded wait that
 *    ran out) set bits of a status word kept in the workspace; kernels skip the
 *    bad items and never trap.  moe_check_device_status reports them.
 *  - Nothing crosses the ABI as a C++ exception.
 */
#ifndef MOE_H
#define MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* moe_stream_t; /* identical to cudaStream_t */

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,         /* NULL pointer, bad size or inconsistent config */
  MOE_ERR_UNSUPPORTED = 2,         /* valid request outside what the library implements */
  MOE_ERR_ALIGNMENT = 3,           /* a pointer is not 16-byte aligned (workspace: 256) */
  MOE_ERR_WORKSPACE_TOO_SMALL = 4, /* ws_bytes < moe_workspace_size() */
  MOE_ERR_CUDA = 5,                /* a CUDA runtime call or launch failed */
  MOE_ERR_DEVICE_CHECK = 6,        /* device status word: bad data (e.g. id out of range) */
  MOE_ERR_DEVICE_TIMEOUT = 7       /* device status word: a bounded wait gave up */
} moe_status;

typedef enum { MOE_SCORE_SOFTMAX = 0, MOE_SCORE_SIGMOID = 1 } moe_score_fn;

typedef enum {
  MOE_BIAS_NONE = 0,
  MOE_BIAS_LOGIT = 1, /* bias[e] added to the logit before scoring (moves weights too) */
  MOE_BIAS_SELECT = 2 /* bias[e] added to the score for selection only */
} moe_bias_mode;

/* How moe_layer_forward returns the expert outputs to their tokens. */
typedef enum {
  MOE_COMBINE_DEFAULT = 0, /* the library's choice (MOE_COMBINE_FUSED) */
  MOE_COMBINE_ORDERED = 1, /* the down projection writes one fp32 row per pick; a
                              combine kernel adds each token's picks in slot order
                              (deterministic: the same bits on every call) */
  MOE_COMBINE_FUSED = 2    /* the down projection's epilogue adds w * y into the
                              token's fp32 accumulator (atomic adds; the order of
                              a token's picks, and so the last bits, can change
                              from call to call) */
} moe_combine_mode;

/* How the bf16 grouped FFN launches its tensor-core passes. */
typedef enum {
  MOE_FFN_LAUNCH_DEFAULT = 0, /* the library's tile-parameter table decides */
  MOE_FFN_LAUNCH_TWO = 1,     /* gate/up, then down: two persistent launches */
  MOE_FFN_LAUNCH_ONE = 2,     /* one persistent launch: a down tile starts as soon as
                                 its expert's gate/up tiles have stored h */
  MOE_FFN_LAUNCH_ONE_WIDE = 3 /* one persistent launch whose down tiles span 256 output
                                 channels: two 128-channel weight boxes share each
                                 activation box, so h rows are read half as often
                                 (pays off with many rows per expert) */
} moe_ffn_launch;

typedef enum {
  MOE_W_BF16 = 0, /* bf16 weights and activations, fp32 accumulation */
  MOE_W8A8 = 1    /* int8 weights + per-output-channel fp32 scales; per-row int8 activations */
} moe_wdtype;

/* Layer description.  Zero-initialise, then fill.  Group modes:
 *   n_group == 1                      : flat top-k over all experts;
 *   n_group > 1, per_group_k == 0     : a group scores the sum of its two best
 *                                       keys; the topk_group best groups stay
 *                                       eligible, then top-k ([PANGU] H2P);
 *   n_group > 1, per_group_k > 0      : exactly per_group_k winners per group,
 *                                       top_k == n_group * per_group_k (MoGE).
 * Groups are contiguous blocks of (n_routed + n_zero) / n_group experts. */
typedef struct {
  int32_t hidden;        /* H, multiple of 8 */
  int32_t inter;         /* I (routed experts), multiple of 8 */
  int32_t n_routed;      /* E_r >= 0 */
  int32_t n_zero;        /* E_z >= 0; 1 <= E_r + E_z <= 4096 */
  int32_t top_k;         /* 1 <= k <= min(32, E_r + E_z) */
  int32_t n_group;       /* >= 1, divides E_r + E_z, <= 64 */
  int32_t topk_group;
  int32_t per_group_k;
  int32_t score;         /* moe_score_fn */
  int32_t renormalize;   /* 1: weights divided by the sum of the k picked scores */
  float routed_scale;    /* multiplies every routed weight (0 is read as 1) */
  int32_t bias_mode;     /* moe_bias_mode */
  int32_t shared_inter;  /* I_s of the always-on shared expert (weight 1); 0 = none */
  int32_t wdtype;        /* moe_wdtype */
  int32_t out_fp32;      /* moe_layer_forward `out`: 1 = fp32, 0 = bf16 */
  int32_t gemv_max_rows; /* experts with <= this many rows take the streaming GEMV
                            path (bf16 FMA, or int8 dp4a for MOE_W8A8), the rest
                            tensor-core tiles.  0 = the library's tile-parameter
                            table (moe_tile_choice), < 0 = never GEMV.  Fixed with
                            the workspace size: W8A8 streaming needs int8 copies
                            of the sorted activations. */
  int32_t combine;       /* moe_combine_mode; fixed with the workspace size */
  int32_t ffn_launch;    /* moe_ffn_launch (bf16 layers) */
} moe_config;

/* Human-readable name of a status. Never NULL. */
const char* moe_status_string(moe_status s);

/* Bytes of device workspace needed by any entry point below for (cfg, T).
 * The same workspace serves every stage; its first 4096 bytes hold the device
 * status word and the router's tile counters, which the caller must zero once
 * (cudaMemset) before first use; the library leaves the counters zero after
 * every call. */
moe_status moe_workspace_size(const moe_config* cfg, int32_t T, size_t* bytes);

/* Router + top-k gating.  [LC-A3] 优化措施三 (Router Matmul), [PANGU] opening
 * section and H2P (grouped experts), [LC-CANN] 拆解MoE困局 (zero experts compete
 * in the same top-k).
 *  x         bf16 [T, H]
 *  w_router  fp32 [E_r + E_z, H]
 *  bias      fp32 [E_r + E_z] (required unless bias_mode == NONE, else ignored)
 *  topk_ids  int32 [T, k] out: slot j = j-th largest key, ties to the lower index
 *  topk_w    fp32  [T, k] out: score of the pick (renormalised / scaled per cfg) */
moe_status moe_route(const moe_config* cfg, int32_t T, const void* x, const float* w_router,
                     const float* bias, int32_t* topk_ids, float* topk_w, void* ws,
                     size_t ws_bytes, moe_stream_t stream);

/* Stable re-sort of the T*k picks by expert, InitialRouting style ([DS-ASC]
 * "2. MOE 算子优化"), and gather of the picked token rows.
 *  topk_ids            int32 [T, k]; an id outside [0, E_r+E_z) sets the device
 *                      status word (MOE_ERR_DEVICE_CHECK) and the pick is dropped
 *  x                   bf16 [T, H]
 *  counts              int32 [E_r + E_z] out
 *  offsets             int32 [E_r + E_z + 1] out (exclusive scan; offsets[E] = T*k)
 *  sorted_to_expanded  int32 [T*k] out: sorted position p -> expanded index t*k + j
 *  expanded_to_sorted  int32 [T*k] out: inverse permutation
 *  x_perm              out, rows in sorted order, only the picks of FFN experts
 *                      (positions < offsets[E_r]); capacity T*k rows.
 *                      bf16 [T*k, H] (MOE_W_BF16) or int8 [T*k, H] (MOE_W8A8)
 *  x_perm_scale        fp32 [T*k] out (MOE_W8A8: per-row scale; may be NULL for bf16) */
moe_status moe_permute(const moe_config* cfg, int32_t T, const int32_t* topk_ids, const void* x,
                       int32_t* counts, int32_t* offsets, int32_t* sorted_to_expanded,
                       int32_t* expanded_to_sorted, void* x_perm, float* x_perm_scale, void* ws,
                       size_t ws_bytes, moe_stream_t stream);

/* Grouped SwiGLU FFN over the sorted rows ([PANGU] SwiftGMM): for each FFN
 * expert e, rows offsets[e] .. offsets[e+1]-1 of x_perm go through
 * y = W_down[e] (silu(W_gate[e] x) * (W_up[e] x)).
 *  offsets   int32 [E_r + E_z + 1] as written by moe_permute
 *  x_perm    as written by moe_permute (bf16 or int8 rows)
 *  w_gate, w_up  [E_r, I, H]; w_down [E_r, H, I]  (bf16, or int8 for MOE_W8A8)
 *  s_gate, s_up  fp32 [E_r, I]; s_down fp32 [E_r, H]  (MOE_W8A8 only, else NULL)
 *  y_perm    fp32 [T*k, H] out, row p = expert output of sorted pick p
 *            (rows >= offsets[E_r] are not written) */
moe_status moe_grouped_ffn(const moe_config* cfg, int32_t T, const int32_t* offsets,
                           const void* x_perm, const float* x_perm_scale, const void* w_gate,
                           const void* w_up, const void* w_down, const float* s_gate,
                           const float* s_up, const float* s_down, float* y_perm, void* ws,
                           size_t ws_bytes, moe_stream_t stream);

/* Weighted combine ([LC-CANN] 拆解MoE困局 "Combine"; [LC-A3] 背景介绍 for
 * zero-computation experts):
 *   out[t] = sum_j topk_w[t,j] * (id < E_r ? y_perm[expanded_to_sorted[t*k+j]] : x[t])
 *            + shared_out[t]
 * summed in slot order, then the shared expert.
 *  shared_out  fp32 [T, H] or NULL
 *  out         bf16 [T, H] (cfg->out_fp32 == 0) or fp32 [T, H] */
moe_status moe_combine(const moe_config* cfg, int32_t T, const float* y_perm,
                       const int32_t* expanded_to_sorted, const int32_t* topk_ids,
                       const float* topk_w, const void* x, const float* shared_out, void* out,
                       moe_stream_t stream);

/* The whole layer: route -> permute -> grouped FFN (+ shared expert) -> combine.
 *  x, w_router, bias, w_gate/w_up/w_down, s_* as above
 *  ws_gate, ws_up [I_s, H], ws_down [H, I_s]: shared expert, NULL when
 *  cfg->shared_inter == 0 ([DS-ASC] deployment paragraph: 1 shared expert).
 *  bf16, or int8 for MOE_W8A8: the shared expert then takes the same per-token
 *  int8 codes as the routed experts ([DS-ASC] "2. 模型侧并发优化": activations
 *  are quantised before they are gathered for the MoE layer), and its
 *  per-output-channel scales follow the routed experts' in s_gate / s_up
 *  ([E_r * I + I_s] each) and s_down ([E_r * H + H]).
 *  out       bf16 or fp32 [T, H] per cfg->out_fp32 */
moe_status moe_layer_forward(const moe_config* cfg, int32_t T, const void* x,
                             const float* w_router, const float* bias, const void* w_gate,
                             const void* w_up, const void* w_down, const float* s_gate,
                             const float* s_up, const float* s_down, const void* ws_gate,
                             const void* ws_up, const void* ws_down, void* out, void* ws,
                             size_t ws_bytes, moe_stream_t stream);

/* Router + top-k without any caller memory besides the tensors (the pages have
 * no counterpart; this is a library convenience).  For callers that cannot
 * provide a workspace: a host framework that hands an operator only its input
 * and output buffers, or a decode loop that must not call cudaMalloc (it can
 * synchronise the device and take milliseconds).  Same arguments as moe_route,
 * minus the workspace, and the same results for batches below 1024 tokens.
 * Nothing is allocated: the router's logits live in a 4 MiB array compiled
 * into the library, present on every GPU that loads it until the process exits.
 *  - It always takes moe_route's small-batch router.  For T >= 1024 with H a
 *    multiple of 64, where moe_route may switch to its large-batch router, the
 *    two sum the same products in a different order: ids are equal unless two
 *    keys are closer than the logits' rounding, weights agree to ~1e-5 relative.
 *  - Rejects, with MOE_ERR_WORKSPACE_TOO_SMALL, any (cfg, T) whose logits need
 *    more than 4 MiB: T x (E_r + E_z) x 4 bytes, times (1 + the router's split-K
 *    count) when the CUDA-core router runs and splits K (the tensor-core router,
 *    taken where H is a multiple of 64 and the batch has enough tiles, needs no
 *    partials); e.g. T = 64 with 768 experts needs 196 KB, T = E = 1024 4 MiB.
 *  - The first call on a device looks up the array's device address
 *    (cudaGetSymbolAddress); make that first call before any stream capture.
 *  - Every call on a device shares the array: calls whose work overlaps on the
 *    GPU (other streams, other host threads) race on it and may give wrong
 *    results.  Serialise them.  Device-side data checks are not reported. */
moe_status moe_route_noalloc(const moe_config* cfg, int32_t T, const void* x,
                             const float* w_router, const float* bias, int32_t* topk_ids,
                             float* topk_w, moe_stream_t stream);

/* The grouped FFN's tiling choices for (cfg, T): the GEMV / tensor-core switch
 * point and whether a bf16 FFN runs as one persistent launch (1) or two (0).
 * They come from cfg where it sets them, else from the tile-parameter table the
 * library was built with ([PANGU] SwiftGMM: tiling chosen from measured
 * history, by expert load): the entry of the same weight type nearest in load
 * bucket (expected picks per expert, T * k / (E_r + E_z)), then in H * I. */
moe_status moe_tile_choice(const moe_config* cfg, int32_t T, int32_t* gemv_max_rows,
                           int32_t* ffn_one_launch);
/* *ffn_one_launch: 0 = two launches, 1 = one launch, 2 = one launch with
 * 256-channel down tiles (MOE_FFN_LAUNCH_ONE_WIDE). */

/* Synchronises `stream`, reads and clears the device status word in `ws`.
 * MOE_OK, MOE_ERR_DEVICE_CHECK or MOE_ERR_DEVICE_TIMEOUT (or MOE_ERR_CUDA). */
moe_status moe_check_device_status(void* ws, moe_stream_t stream);

/* ---- Diagnostics ---- */

/* Exercises the device-side failure path without faulting the GPU: one thread
 * waits on a barrier that nothing completes, gives up after `limit_cycles` SM
 * cycles (1 .. 2e9), records MOE_ERR_DEVICE_TIMEOUT in the status word of `ws`
 * (>= 256 bytes, 256-byte aligned, first 8 bytes zero) and returns.  Every
 * bounded wait of the library reports a timeout the same way; read it with
 * moe_check_device_status. */
moe_status moe_selftest_wait_timeout(void* ws, int64_t limit_cycles, moe_stream_t stream);

/* Kernels of the library, for timing and launch counts. */
typedef enum {
  MOE_K_ROUTER = 0,
  MOE_K_TOPK,
  MOE_K_PERM_COUNT,
  MOE_K_PERM_SCAN,
  MOE_K_PERM_SCATTER,
  MOE_K_PERM_GATHER,
  MOE_K_WORKLIST,
  MOE_K_GEMV_GATE_UP,
  MOE_K_GEMV_DOWN,
  MOE_K_TC_GATE_UP,
  MOE_K_TC_DOWN,
  MOE_K_QUANT_H,
  MOE_K_COMBINE,
  MOE_K_W8_EXACT,
  MOE_K_SORT,  /* small batches: count, scan, scatter and work list in one launch */
  MOE_K_COUNT
} moe_kernel_kind;

/* Grouped int8 x int8 -> int32 matmul on the W8A8 path's kernels, exposing the
 * exact integer accumulators (QuantBatchMatmul, [LC-A3] 优化措施三):
 *   acc[r, n] = sum_k a[r, k] * w[e, n, k]   for offsets[e] <= r < offsets[e+1].
 *  a        int8 [R, K] rows sorted by expert; w int8 [n_experts, N, K]
 *  offsets  int32 [n_experts + 1], device, offsets[n_experts] <= R
 *  acc      int32 [R, N] out (rows >= offsets[n_experts] untouched)
 * K must be a multiple of 16 (<= 131071).  Exact for every int8 input: tiles
 * whose partial sums could reach 2^24 are recomputed with integer arithmetic. */
moe_status moe_qgemm_s8_workspace_size(int32_t n_experts, int32_t K, int32_t N, int32_t R,
                                       size_t* bytes);
moe_status moe_qgemm_s8(int32_t n_experts, int32_t K, int32_t N, int32_t R, const int32_t* offsets,
                        const void* a, const void* w, int32_t* acc, void* ws, size_t ws_bytes,
                        moe_stream_t stream);

const char* moe_kernel_name(int32_t kind);

/* enable != 0: every later launch of the library is bracketed by CUDA events on
 * its stream (costs two event records per launch).  Process-wide. */
moe_status moe_timing_enable(int32_t enable);

/* Waits for the recorded events (host synchronisation), adds each kernel kind's
 * elapsed milliseconds and launch count since the last collect into
 * ms[kind] / launches[kind] (arrays of n >= MOE_K_COUNT entries), then resets. */
moe_status moe_timing_collect(float* ms, int32_t* launches, int32_t n);

/* Launches made since process start, per kind (always counted). */
moe_status moe_launch_counts(int64_t* launches, int32_t n);

#ifdef __cplusplus
}
#endif
#endif /* MOE_H */
