// Host-side interface between the C ABI (abi.cu) and the kernel files.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "moe.h"

namespace moe {

struct DevStatus;

// One unit of grouped-FFN work: a contiguous run of sorted rows of one expert.
// expert >= 0 indexes the routed weight stacks; expert == -1 is the shared
// expert (its rows index the token matrix directly).  Tensor-core tasks carry
// (chunk index << 16 | chunks of the same expert) in `chunk`.
struct FfnTask {
  int32_t expert;
  int32_t row0;
  int32_t nrows;
  int32_t chunk;
};

// Tensor-core tile -> (task, channel tile).  The tiles of one expert's tasks
// form one contiguous range, enumerated channel tile outer, token chunk inner,
// so the CTAs working on an expert at the same time read the same weight tile
// (one HBM read, the rest from L2) instead of re-streaming it per chunk.
__device__ __forceinline__ void tc_tile_of(const FfnTask* tasks, const int32_t* start,
                                           int ntasks, int tile, int* task, int* ct) {
  int lo = 0, hi = ntasks - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (start[mid] <= tile)
      lo = mid;
    else
      hi = mid - 1;
  }
  const int c = tasks[lo].chunk;
  const int first = lo - (c >> 16), nt = c & 0xffff;
  const int u = tile - start[first];
  *task = first + u % nt;
  *ct = u / nt;
}

// The down projection's outputs added straight into the tokens' fp32
// accumulators (the combine fused into the down epilogue; acc == nullptr:
// store the y rows instead, for the ordered combine).  Sorted row p adds
// w[r] * y to acc[r / k], r = s2e[p]; a row of the shared expert is the token
// itself and adds y at weight 1.
struct ScatterAdd {
  float* acc;          // [T, H] fp32
  const int32_t* s2e;  // sorted position -> expanded index t * k + j (nullptr: the
                       // rows are the tokens themselves, at weight 1)
  const float* w;      // [T * k] routing weights
  int k;
};
__device__ __forceinline__ void scatter_target(const ScatterAdd& s, int row, bool shared,
                                               int* tok, float* wt) {
  if (shared || s.s2e == nullptr) {
    *tok = row;
    *wt = 1.f;
  } else {
    const int r = s.s2e[row];
    *tok = r / s.k;
    *wt = s.w[r];
  }
}

// Slots of the device work-list counter array.
enum {
  kWlGemvTasks = 0,
  kWlGemvItemsGU,
  kWlGemvItemsDN,
  kWlTcTasks,
  kWlTcTilesGU,
  kWlTcTilesDN,
  kWlSchedGU,   // dynamic tile counters of the two tensor-core passes (zeroed
  kWlSchedDN,   // by the kernel that writes the work list)
  kWlCount
};

struct WorkList {
  FfnTask* gemv_tasks;
  int32_t* gemv_start_gu;  // first item of each task, gate/up pass
  int32_t* gemv_start_dn;  // first item of each task, down pass
  FfnTask* tc_tasks;
  int32_t* tc_start_gu;
  int32_t* tc_start_dn;
  int32_t* counts;  // kWlCount ints
  int32_t capacity; // max tasks of each kind
  int32_t* redo_gu; // W8A8 guard-failure lists (count word zeroed here), or nullptr
  int32_t* redo_dn;
  int32_t* gu_done; // single-launch FFN: per tensor-core task counter, zeroed here
};

// Geometry of the streaming (GEMV) path.
constexpr int kGemvMaxRows = 8;    // most activation rows one GEMV task carries
constexpr int kGemvChGU = 8;       // output channels per gate/up item
constexpr int kGemvChDN = 16;      // output channels per down item
constexpr int kGemvI8Ch = 128;     // output channels per W8A8 streaming item (both passes)
// Geometry of the tensor-core path (swap-AB: weights are M, tokens are N).
constexpr int kTcM = 128;          // weight rows per tile
constexpr int kTcMaxN = 128;       // token rows per task
constexpr int kW8MaxN = 256;       // token rows per W8A8 task
// Measured on GB300 (LongCat/DSv3/Pangu-shaped decode layers): tensor-core
// tiles with N = 16 stream expert weights at ~6.9 TB/s, above the CUDA-core GEMV
// at every row count (6.4 TB/s at one row, less with more), so by default every
// unit takes the tensor-core path; gemv_max_rows > 0 selects the GEMV path.
constexpr int kDefaultGemvMaxRows = 0;
// W8A8: the int8 GEMV (dp4a, no conversion) beats the converting tensor-core
// tiles on light experts.  Measured on GB300 (tensor cores only / GEMV for <= 2,
// 4, 8, 16 rows): a LongCat-shaped W8A8 decode layer 3.31 / 2.03 / 1.77 / 1.71 /
// 1.75 ms; the Zipf-loaded prefill layer 7.74 / - / 7.57 / 7.47 / 7.76 ms.
constexpr int kDefaultGemvMaxRowsW8 = 8;

struct Launch {
  cudaStream_t stream;
  int num_sms;
  DevStatus* status;
};

// Router + top-k (route.cu).  With split-K (splits > 1) the router needs the
// partial buffer [splits, T, E] and one counter per tile (router_tiles), which
// must be zero before the first call; the kernel leaves them zero again.
constexpr int kRouterCounterBytes = 3840;  // counters kept right after the status word
int router_tiles(const moe_config& c, int T);
int router_splits(const moe_config& c, int T, int num_sms);
// The CUDA-core router's split-K count as every entry point sizes its scratch
// (the split aims at about two CTAs on each of 152 SMs).
int router_splits_default(const moe_config& c, int T);
// Whether launch_route runs the decode router on tensor cores for (c, T): H a
// multiple of 64, enough parallel work, and MOE_ROUTER_TC not set to 0.  That
// router needs neither the split-K partials nor the tile counters.  (If its
// tensor maps cannot be encoded, launch_route falls back to the CUDA-core
// router with the split count it was given.)
bool router_tc_decode_chosen(const moe_config& c, int T);
// Router matmul then top-k gating (one launch when the decode router on tensor
// cores holds all experts in one tile and picks the top-k itself; logits are
// then not written).
void launch_route(const Launch& L, const moe_config& c, int T, const void* x, const float* w_r,
                  const float* bias, float* partial, int splits, float* logits, int* counters,
                  int32_t* ids, float* w);
// Top-k gating of given logits.
void launch_topk_only(const Launch& L, const moe_config& c, int T, const float* logits,
                      const float* bias, int32_t* ids, float* w);
// Top-k gating arguments (one warp per token; topk.cuh).
struct TopkArgs {
  const float* logits;
  const float* bias;
  int32_t* ids;
  float* w;
  DevStatus* status;
  int T, E, k;
  int n_group, topk_group, per_group_k;
  int score, renorm, bias_mode;
  float scale;
};
TopkArgs topk_args(const Launch& L, const moe_config& c, int T, const float* logits,
                   const float* bias, int32_t* ids, float* w);
// Small layers: the router's x and W_r fit one CTA's shared memory and the work
// (T * E * H multiply-adds) is at most kSmallRouteWork, so one CTA of
// kSmallRouteWarps warps computes the logits and the top-k.  The one-CTA
// re-sort runs that code before its own work when folds are on; otherwise
// launch_route runs it as a kernel of its own: the same bits either way.
constexpr int kSmallRouteWarps = 32;
constexpr long long kSmallRouteWork = 1LL << 20;
struct SmallRoute {
  const uint16_t* x;  // bf16 [T, H], 16-byte aligned
  const float* w_r;   // fp32 [E, H], 16-byte aligned
  int H;
};
bool route_small_fits(const moe_config& c, int T);
size_t route_small_smem(const moe_config& c, int T);
// Large batches: the router as a tensor-core GEMM over the exact three-term
// bf16 split of W_r ([E, 3H], written by launch_router_split).
bool router_on_tensor_cores(const moe_config& c, int T);
void launch_router_split(const Launch& L, const float* w_r, int E, int H, uint16_t* out);

// Permutation (permute.cu)
constexpr int kPermTokens = 256;  // tokens per permutation block
void launch_perm_count(const Launch& L, int T, int k, int E, const int32_t* ids, int32_t* bc);
void launch_perm_scan(const Launch& L, int T, int E, int32_t* bc, int32_t* counts,
                      int32_t* offsets);
void launch_perm_scatter(const Launch& L, int T, int k, int E, const int32_t* ids,
                         const int32_t* bc, int32_t* s2e, int32_t* e2s);
void launch_perm_gather(const Launch& L, const moe_config& c, int T, const int32_t* ids,
                        const int32_t* e2s, const void* x, void* x_perm, float* x_perm_scale,
                        const float* w = nullptr, float* acc = nullptr);
// dn_ch: output channels of a tensor-core down tile (0: the weight type's own,
// kTcM for bf16, 2 * kTcM for W8A8).
void launch_worklist(const Launch& L, const moe_config& c, int T, const int32_t* offsets,
                     const WorkList& wl, int gemv_max_rows, int gemv_chunk, int tc_chunk,
                     int dn_ch = 0);
// Small batches (one CTA holds the [expert][token] pick bitmap): count, scan and
// stable scatter in one launch, plus the work list when wl is not nullptr.
// Outputs equal those of the count / scan / scatter / work-list launches.
constexpr int kSortSmallMaxT = 1024;
constexpr int kSortSmallSmem = 96 * 1024;
bool sort_small_fits(int T, int E);
// The bf16 row gather (and the fused combine's accumulator start) done by the
// one-CTA sort itself, for layers whose gathered rows and accumulators are
// small (kSmallGatherBytes at most): one launch fewer.
constexpr size_t kSmallGatherBytes = 256 * 1024;
struct SmallGather {
  const uint16_t* x;  // bf16 [T, H]
  uint16_t* x_perm;   // bf16 [T * k, H] (nullptr: no gather)
  const float* w;     // routing weights (fused combine), or nullptr
  float* acc;         // the tokens' accumulators (fused combine), or nullptr
  int H, E_r;
};
// With route != nullptr (route_small_fits(c, T)) the CTA first routes the
// tokens itself (tk: where the ids and weights go) and then sorts those ids.
void launch_sort_small(const Launch& L, const moe_config& c, int T, const int32_t* ids,
                       int32_t* counts, int32_t* offsets, int32_t* s2e, int32_t* e2s,
                       const WorkList* wl, int gemv_max_rows, int gemv_chunk, int tc_chunk,
                       const SmallGather* gather = nullptr, const SmallRoute* route = nullptr,
                       const TopkArgs* tk = nullptr, int dn_ch = 0);

// Grouped FFN, streaming path (gemv.cu)
struct GemvPass {
  const FfnTask* tasks;
  const int32_t* item_start;
  const int32_t* counts;  // work-list counters
  int task_slot, item_slot;
  const uint16_t* w0;     // gate (gate/up pass) or down weights, routed stack [E, N, K]
  const uint16_t* w1;     // up weights (gate/up pass), else nullptr
  const uint16_t* act;    // routed activation rows [*, K]
  uint16_t* out_h;        // gate/up pass: bf16 [*, N]
  float* out_y;           // down pass: fp32 [*, N]
  const uint16_t* sw0;    // shared expert counterparts (may be nullptr)
  const uint16_t* sw1;
  const uint16_t* sact;
  uint16_t* sout_h;
  float* sout_y;
  int K, Ks;              // reduction length, routed / shared
  int N, Ns;              // output channels, routed / shared
  int max_rows;           // rows per task (1, 2, 4 or 8); the work list chunks by it
  ScatterAdd sc;          // down pass: acc != nullptr adds into the tokens' rows
};
void launch_gemv_gate_up(const Launch& L, const GemvPass& p);
void launch_gemv_down(const Launch& L, const GemvPass& p);

// W8A8 streaming path (gemv_i8.cu): int8 weights x int8 codes with dp4a, items
// of <= 8 rows x 128 channels.  Returns false if a tensor map could not be
// encoded (nothing launched).
struct GemvI8Pass {
  const FfnTask* tasks;
  const int32_t* item_start;
  const int32_t* counts;
  int task_slot, item_slot;
  const int8_t* w0;         // int8 weights [E, N, K] (gate or down)
  const int8_t* w1;         // int8 up weights (gate/up pass)
  int n_experts;
  const float* s0;          // per-channel scales [E, N]
  const float* s1;
  const int8_t* act;        // int8 activation codes [act_rows, K]
  int64_t act_rows;
  const float* row_scale;   // [rows]
  float* out_f32;           // gate/up: h [rows, N]; down: y [rows, N]
  int K, N;
  ScatterAdd sc;            // down pass: acc != nullptr adds into the tokens' rows
};
bool launch_gemv_i8_gate_up(const Launch& L, const GemvI8Pass& p);
bool launch_gemv_i8_down(const Launch& L, const GemvI8Pass& p);

// Small layers with the fused combine: the down pass's last CTA to finish
// rounds the tokens' fp32 accumulators to the bf16 output (ctr != nullptr), in
// place of the finalize launch.  ctr is a zero word of the workspace head; the
// last CTA leaves it zero.
constexpr int kSmallFinalizeElems = 64 * 1024;
struct SmallFinalize {
  int* ctr;
  const float* acc;
  uint16_t* out;
  int n8;  // T * H / 8
};
constexpr size_t kFinalizeCtrOffset = 64;  // in the workspace's 256-byte status block

// Grouped FFN, tensor-core path (gemm_tc.cu).  Returns false if a tensor map
// could not be encoded (nothing launched).
struct TcPass {
  const FfnTask* tasks;
  const int32_t* tile_start;
  const int32_t* counts;
  int task_slot, tile_slot, sched_slot;
  const void* w0;          // routed weights [n_experts, N, K] (gate or down)
  const void* w1;          // routed up weights (gate/up pass)
  int n_experts;
  const void* act;         // routed activation rows [act_rows, K]
  int64_t act_rows;
  uint16_t* out_h;         // gate/up pass output, bf16 [*, N]
  float* out_y;            // down pass output, fp32 [*, N]
  const void* sw0;         // shared expert [Ns, Ks] (nullptr: none)
  const void* sw1;
  const void* sact;        // shared activation rows [sact_rows, Ks]
  int64_t sact_rows;
  uint16_t* sout_h;
  float* sout_y;
  int K, Ks, N, Ns;
  int b_kmod;              // > 0: activation K coordinate taken modulo b_kmod
  ScatterAdd sc;           // down pass: acc != nullptr adds into the tokens' rows
  SmallFinalize fin;       // down pass of a small layer: the last CTA rounds the output
  int dn_wide;             // one-launch FFN: a down tile spans 2 x kTcM channels
  int task_cap;            // entries the work-list arrays hold (0: unknown)
};
bool launch_tc_gate_up(const Launch& L, const TcPass& p);
bool launch_tc_down(const Launch& L, const TcPass& p);
// Both passes in one persistent launch: every gate/up tile, then every down
// tile; a down tile waits (bounded) until its task's gate/up tiles have stored
// their h rows, counted in gu_done [tasks] (zeroed by the work-list kernel).
// gu.tile_slot / dn.tile_slot count the tiles of each pass, gu.sched_slot is
// the one claim counter.  Timed and counted as MOE_K_TC_GATE_UP.
bool launch_tc_ffn(const Launch& L, const TcPass& gu, const TcPass& dn, int32_t* gu_done);
// logits[T, E] = x[T, H] . [W3 | W2 | W1]^T on tensor cores (K = 3H, the token
// rows read three times); tasks/start/counts are its own small work list.
bool launch_tc_router(const Launch& L, const moe_config& c, int T, const void* x,
                      const uint16_t* w_split, FfnTask* tasks, int32_t* start, int32_t* counts,
                      float* logits);

// W8A8 grouped FFN (w8a8.cu): tensor-core tiles on integer-valued fp16 operands
// with an exactness guard, then an exact CUDA-core pass over guard failures.
enum { kW8GateUp = 0, kW8Down = 1, kW8Raw = 2 };
struct W8Pass {
  int mode;                 // kW8GateUp: h = silu(g)*u (fp32); kW8Down: y (fp32);
                            // kW8Raw: int32 accumulators
  const FfnTask* tasks;
  const int32_t* tile_start;
  const int32_t* counts;
  int task_slot, tile_slot, sched_slot;
  const void* w0;           // int8 weights [n_experts, N, K] (gate or down)
  const void* w1;           // int8 up weights (gate/up mode)
  int n_experts;
  const float* s0;          // per-channel scales [n_experts, N]
  const float* s1;
  const void* act;          // integer-valued fp16 activation rows [act_rows, K]
  int64_t act_rows;
  const int32_t* row_norm2; // [act_rows] sum of squared codes
  const float* row_scale;   // [act_rows]
  float* out_f32;
  int32_t* out_i32;
  int32_t* redo;            // [0] count (zeroed by the work-list kernel), [1..cap]
  int redo_cap;
  int K, N;
  ScatterAdd sc;            // down mode: acc != nullptr adds into the tokens' rows
};
bool launch_w8a8(const Launch& L, const W8Pass& p);
void launch_i8_rows_to_f16(const Launch& L, const int8_t* src, uint16_t* dst, int32_t* norm2,
                           int R, int K, const int32_t* nrows);
// Layer path: quantise each token once and write its codes, scale and sum of
// squares to the sorted rows of its FFN-expert picks.  A row of an expert of at
// most gemv_max rows (offsets give the loads) gets int8 codes in x8, any other
// row integer-valued fp16 codes in x16; x8 nullptr sends every row to x16.
struct QuantGatherOut {
  uint16_t* x16;       // sorted rows, integer-valued fp16 codes
  int8_t* x8;          // sorted rows of streamed experts, int8 codes (or nullptr)
  float* scale;        // [R] per sorted row
  int32_t* norm2;      // [R]
  uint16_t* tok16;     // W8A8 shared expert: one fp16 code row per token (or nullptr)
  float* tok_scale;    // [T]
  int32_t* tok_norm2;  // [T]
};
void launch_quant_gather(const Launch& L, const moe_config& c, int T, const void* x,
                         const int32_t* ids, const int32_t* e2s, const int32_t* offsets,
                         int gemv_max, const QuantGatherOut& o, const float* w = nullptr,
                         float* acc = nullptr);
// The first offsets[n_experts] of R fp32 rows (all R when offsets is nullptr)
// -> codes, by the same rule: int8 into dst8 for rows of experts of at most
// gemv_max rows, else fp16 into dst; dst8 nullptr sends every row to dst.
void launch_quant_rows(const Launch& L, const float* src, uint16_t* dst, int8_t* dst8,
                       float* scale, int32_t* norm2, int R, int K, const int32_t* offsets,
                       int n_experts, int gemv_max);

// Combine (combine.cu)
void launch_combine(const Launch& L, const moe_config& c, int T, const float* y_perm,
                    const int32_t* e2s, const int32_t* ids, const float* w, const void* x,
                    const float* shared_out, void* out);

// Fused combine (combine.cu): the tokens' fp32 accumulators [T, H] rounded to
// the bf16 output.  (Their zero-computation picks are added by the gather
// kernels, which write every accumulator row first; the down passes add the
// expert outputs.)
void launch_finalize(const Launch& L, int T, int H, const float* acc, void* out);
// Zero-computation picks of token t: acc[t] = sum over such slots j, in slot
// order, of w[t, j] * x[t] (zero when there are none); elements 8i .. 8i + 7
// of the row for i = first, first + stride, ... below H / 8.
__device__ __forceinline__ void zero_pick_init(const int32_t* ids, const float* w, int t, int k,
                                               int E_r, int E, const uint16_t* xrow, float* arow,
                                               int H, int first, int stride) {
  for (int i = first; i < H / 8; i += stride) {
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int j = 0; j < k; ++j) {
      const int e = ids[(size_t)t * k + j];
      if (e < E_r || e >= E) continue;
      const float wj = w[(size_t)t * k + j];
      const uint4 v = reinterpret_cast<const uint4*>(xrow)[i];
      const uint32_t q[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        acc[2 * u] += wj * __uint_as_float(q[u] << 16);
        acc[2 * u + 1] += wj * __uint_as_float(q[u] & 0xffff0000u);
      }
    }
    float4* o = reinterpret_cast<float4*>(arow) + 2 * i;
    o[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
    o[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
  }
}

// Failure-path self-test (combine.cu): a bounded wait that is never satisfied.
void launch_wait_timeout_selftest(const Launch& L, long long limit_cycles);

// Raise a kernel's dynamic shared-memory limit once per device (abi.cu).
enum {
  kAttrTopk = 0,
  kAttrPermScatter,
  kAttrTcGU,
  kAttrTcDN,
  kAttrTcRouter,
  kAttrGemvBase,                 // 8 slots: (gate/up, down) x row cap 1, 2, 4, 8
  kAttrW8Base = kAttrGemvBase + 8,  // 3 slots: W8A8 modes
  kAttrGemvI8Base = kAttrW8Base + 3, // 8 slots: W8A8 GEMV (gate/up, down) x row cap
  kAttrRouter = kAttrGemvI8Base + 8,
  kAttrRouterTc,
  kAttrSortSmall,
  kAttrTcFfn,
  kAttrRouteSmall,
  kAttrSlots
};
void set_smem_attr_once(const void* func, int bytes, int slot);

// Per-launch bookkeeping (abi.cu): call before/after each kernel launch.
void launch_begin(const Launch& L, int kind);
void launch_end(const Launch& L, int kind);
// Records a launch's error for launch_status_take (the first one wins).
void launch_note(cudaError_t e);
// Programmatic dependent launch of the library's kernels: on unless the
// environment sets MOE_PDL=0 (read once).
bool pdl_enabled();

// Small-layer folds (router + top-k in one launch, re-sort + gather in one CTA,
// the output rounded by the down pass's last CTA): on unless the environment
// sets MOE_FOLDS=0 (read once).
bool folds_enabled();

// Launches a library kernel so that it may start while the previous kernel of
// the stream is still running (the kernel waits, pdl_wait, before it touches
// global memory).
template <typename... P, typename... A>
void launch_kernel(void (*kernel)(P...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                   A&&... args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_enabled() ? 1 : 0;
  launch_note(cudaLaunchKernelEx(&cfg, kernel, static_cast<A&&>(args)...));
}
// The same with a cluster shape given at launch (for kernels whose cluster size
// is chosen at run time).
template <typename... P, typename... A>
void launch_kernel_cluster(void (*kernel)(P...), dim3 grid, dim3 cluster, dim3 block, size_t smem,
                           cudaStream_t stream, A&&... args) {
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cluster.x;
  attr[0].val.clusterDim.y = cluster.y;
  attr[0].val.clusterDim.z = cluster.z;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_enabled() ? 2 : 1;
  launch_note(cudaLaunchKernelEx(&cfg, kernel, static_cast<A&&>(args)...));
}
// Status of the launches since the last call (MOE_OK or MOE_ERR_CUDA); resets it.
moe_status launch_status_take();

}  // namespace moe
