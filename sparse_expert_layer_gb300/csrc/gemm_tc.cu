// Grouped SwiGLU FFN, tensor-core path for loaded experts (the GEMM side of the
// GEMV/GEMM switch in the Pangu Pro MoE disclosure, section SwiftGMM).
//
// Swap-AB tiles: the 128 weight rows of a channel tile are the MMA's M side and
// the task's <= 128 token rows its N side (N rounded up to 16), so a task with
// few tokens wastes no tensor work on padding rows of M.
//   D_gate[ch, tok] = W_gate[e][ch, :] . X[tok, :]     (and D_up likewise)
//   h[tok, ch]      = silu(D_gate) * D_up              (epilogue, bf16)
//   D[ch, tok]      = W_down[e][ch, :] . h[tok, :]     -> y[tok, ch] (fp32)
//
// Persistent CTAs, one per SM, dynamic tile scheduling, warp-specialised:
//   warp 6    : claims tiles from a global counter, decodes them and queues
//               them (up to four ahead) for the other roles.
//   warp 0    : TMA producer -- 128x64 weight tiles (3-D map over the expert
//               stack) and 64-row activation boxes, 128-byte swizzle, into a
//               multi-stage shared-memory ring.
//   warp 1    : allocates TMEM; one lane issues tcgen05.mma (kind::f16, bf16 in,
//               fp32 accumulate) and commits stage releases / tile completion.
//   warps 2-5 : epilogue -- tcgen05.ld of the accumulators (each warp owns one
//               32-lane quadrant of TMEM), SwiGLU, coalesced stores.
// Accumulators are double-buffered in TMEM so the epilogue of one tile overlaps
// the MMAs of the next.  Every wait is bounded.  In the single-launch FFN a down
// tile may span 2 x 128 channels (two weight boxes and two accumulators per K
// step sharing one activation box, as gate and up do), so loaded experts' h
// rows are read half as often.
#include <cudaTypedefs.h>

#include <cstring>
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace moe {

namespace {

constexpr int kThreads = 224;
constexpr int kSchedWarp = 6;
constexpr int kBK = 64;                          // K elements per stage: one 128-byte row
constexpr int kATileBytes = kTcM * kBK * 2;      // 16 KB
constexpr int kBTileBytes = kTcMaxN * kBK * 2;   // 16 KB
constexpr int kBoxRows = 64;
constexpr int kBoxBytes = kBoxRows * kBK * 2;    // 8 KB
constexpr int kTaskCache = 1024;                 // work-list tasks kept in shared memory

// Pass of a launch: the down projection, the gate/up projection with SwiGLU,
// or both in one launch (every gate/up tile, then every down tile; a down tile
// starts once its task's gate/up tiles have stored their h rows).
// kTcRouter: the large-batch router's logits, x . (W3 + W2 + W1)^T over the
// exact three-term bf16 split of W_r (rows [W3 | W2 | W1], written by
// router_split_kernel): a stage holds one x box and the three terms' weight
// tiles of the same 64 columns, the W3 and W2 products accumulate in one TMEM
// accumulator, the W1 products in another, and the logit is their sum (the
// small terms are never rounded against the large ones, as in the decode
// router).  x is read once per K step instead of once per term.
enum { kTcDown = 0, kTcGateUp = 1, kTcFfn = 2, kTcRouter = 3 };

template <int MODE>
struct Geom {
  static constexpr int kNA = MODE == kTcDown ? 1 : MODE == kTcRouter ? 3 : 2;  // weight tiles a stage holds
  static constexpr int kStageBytes = kNA * kATileBytes + kBTileBytes;
  static constexpr int kStages = MODE == kTcDown ? 6 : MODE == kTcRouter ? 3 : 4;
  static constexpr int kTmemCols = MODE == kTcDown ? 256 : 512;
  static constexpr int kAccStride = MODE == kTcDown ? 128 : 256;  // columns per accumulator buffer
  static constexpr int kBarBytes = 512;
  // the work list's tile starts and tasks, when it has at most kTaskCache tasks
  static constexpr int kCacheOff = kStages * kStageBytes + kBarBytes;
  static constexpr int kCacheBytes = kTaskCache * (2 * 4 + (int)sizeof(FfnTask));
  static constexpr int kSmemBytes = 1024 + kCacheOff + kCacheBytes;
};

struct TcMaps {
  CUtensorMap a0;   // routed weights: gate (gate/up pass) or down
  CUtensorMap a1;   // routed up weights (gate/up pass)
  CUtensorMap sa0;  // shared expert counterparts
  CUtensorMap sa1;
  CUtensorMap b;    // routed activation rows
  CUtensorMap sb;   // shared expert activation rows
  // single-launch FFN only: the down pass's weights and activation (h) rows
  CUtensorMap d0;
  CUtensorMap sd0;
  CUtensorMap h;
  CUtensorMap sh;
};

struct TcArgs {
  const FfnTask* tasks;
  const int32_t* tile_start;
  const int32_t* counts;
  int task_slot, tile_slot;
  uint16_t* out_h;
  float* out_y;
  uint16_t* sout_h;
  float* sout_y;
  int K, Ks, N, Ns;  // of the pass (single-launch FFN: of its gate/up pass)
  int b_kmod;  // > 0: routed activation K coordinate modulo b_kmod (router tiles)
  int* sched;  // dynamic tile counter, zero at launch
  DevStatus* status;
  ScatterAdd sc;  // down pass: add w * y into the tokens' accumulators
  // single-launch FFN: the down tiles (numbered after the gate/up tiles), and
  // the per-task count of gate/up epilogue warps done (4 per channel tile)
  const int32_t* tile_start_dn;
  int tile_slot_dn;
  int* gu_done;
  int gu_tiles, gu_tiles_shared;  // gate/up channel tiles of a routed / shared task
  SmallFinalize fin;
  int dn_wide;  // single-launch FFN: down tiles of 2 x kTcM channels (two weight boxes and
                // two accumulators per K step, one activation box)
  int task_prefetch;  // work-list entries (< the arrays' capacity, <= kThreads) loaded
                      // together with the counts
};

// Small layers: the last CTA of the down pass to finish rounds the tokens'
// accumulators to bf16.  Every thread fences its own adds before the CTA
// counts itself done, so the last CTA sees all of them.
__device__ __forceinline__ void finalize_if_last(const SmallFinalize& f) {
  __shared__ int last;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) last = atomicAdd(f.ctr, 1) == (int)gridDim.x - 1;
  __syncthreads();
  if (!last) return;
  __threadfence();
  for (int i = threadIdx.x; i < f.n8; i += blockDim.x) {
    const float4 a0 = __ldcg(reinterpret_cast<const float4*>(f.acc) + 2 * i);
    const float4 a1 = __ldcg(reinterpret_cast<const float4*>(f.acc) + 2 * i + 1);
    const float v[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
    uint32_t q[4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
      q[j] = (uint32_t)f_to_bf16(v[2 * j]) | ((uint32_t)f_to_bf16(v[2 * j + 1]) << 16);
    reinterpret_cast<uint4*>(f.out)[i] = make_uint4(q[0], q[1], q[2], q[3]);
  }
  if (threadIdx.x == 0) *f.ctr = 0;  // ready for the next call
}

// Single-launch FFN: a down tile of at most one 64-row activation box carries
// two K steps per stage, each [16 KB weight tile | 8 KB activation box] (narrow
// down tiles; wide ones hold two weight tiles per K step, as gate/up tiles do).
constexpr int kPackedStep = kATileBytes + kBoxBytes;
template <int MODE>
__device__ __forceinline__ bool packed_down(bool gu, int n, int wide) {
  return MODE == kTcFfn && !gu && !wide && n <= kBoxRows;
}
// Whether a tile carries two weight tiles per K step: gate and up, or the two
// channel halves of a wide down tile.
template <int MODE>
__device__ __forceinline__ bool two_weight_tiles(bool gu, int wide) {
  return MODE == kTcGateUp || (MODE == kTcFfn && (gu || wide));
}
static_assert(2 * kPackedStep <= Geom<kTcFfn>::kStageBytes, "two packed K steps fill a stage");

// Order in which the gate/up tiles are handed out: the shared expert's S tiles
// (tiles 0 .. S-1, in groups of g: the g row chunks of one channel tile, which
// read the same weights, once from HBM and otherwise from L2) are spread over
// the first `span` of the R routed tiles, one group after every span / (S / g)
// routed tiles, instead of all coming first.  A bijection of 0 .. S+R-1 that
// keeps the routed tiles in order.
__device__ __forceinline__ int interleave_tile(int c, int S, int g, int R, int span) {
  if (S <= 0 || g <= 0 || R <= 0) return c;
  const int G = S / g;
  const int q = span / G;
  if (q <= 0) return c;
  const int b = c / (g + q), pos = c % (g + q);
  if (b < G) return pos < g ? b * g + pos : S + b * q + (pos - g);
  return S + G * q + (c - G * (g + q));
}

// Single-launch FFN producer: waits (bounded) until a down tile's task has
// target gate/up epilogue warps done; on a timeout it reports the status and
// sets the CTA's abort flag.
__device__ __forceinline__ bool wait_h_rows(const TcArgs& a, int task, int target, int kind,
                                            volatile int* abort_flag) {
  if (wait_rows_done(a.gu_done + task, target)) return true;
  raise_status(a.status, kStTimeout, kind);
  *abort_flag = 1;
  return false;
}

// tasks and start: the work list in shared memory when it fits, else in global
// memory (a binary search of dependent loads).
__device__ __forceinline__ QTile decode_tile(const FfnTask* tasks, int tile, int ntasks, int gu,
                                             const int32_t* start) {
  QTile t;
  int task;
  tc_tile_of(tasks, start, ntasks, tile, &task, &t.ct);
  const FfnTask tk = tasks[task];
  t.tile = tile;
  t.row0 = tk.row0;
  t.n = tk.nrows;
  t.shared = tk.expert < 0;
  t.e = t.shared ? 0 : tk.expert;
  t.task = task;
  t.gu = gu;
  return t;
}

template <int MODE>
__global__ void __launch_bounds__(kThreads, 1)
    tc_kernel(const __grid_constant__ TcMaps maps, const TcArgs a) {
  using G = Geom<MODE>;
  constexpr bool FFN = MODE == kTcFfn;
  extern __shared__ uint8_t smem_raw[];
  const int kind = MODE == kTcDown ? MOE_K_TC_DOWN
                   : MODE == kTcRouter ? MOE_K_ROUTER
                                       : MOE_K_TC_GATE_UP;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  // 1024-byte aligned ring (128-byte swizzle atoms), barriers after it
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + G::kStages * G::kStageBytes);
  uint64_t* empty = full + G::kStages;
  uint64_t* acc_full = empty + G::kStages;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* drain = acc_empty + 2;
  uint64_t* tq_full = drain + 1;
  uint64_t* tq_empty = tq_full + kTileQueue;
  QTile* tq = reinterpret_cast<QTile*>(tq_empty + kTileQueue);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tq + kTileQueue);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  // barriers and tensor maps first: they touch no global memory, so they run
  // before the wait for the previous kernel of the stream
  if (threadIdx.x == 0) {
    for (int s = 0; s < G::kStages; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&acc_full[b]), 1);
      mbar_init(smem_u32(&acc_empty[b]), 4);
    }
    mbar_init(smem_u32(drain), 1);
    for (int s = 0; s < kTileQueue; ++s) {
      mbar_init(smem_u32(&tq_full[s]), 1);
      mbar_init(smem_u32(&tq_empty[s]), 6);  // producer, MMA thread, 4 epilogue warps
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tensormap(&maps.a0);
    prefetch_tensormap(&maps.b);
    if (MODE == kTcGateUp || MODE == kTcFfn) prefetch_tensormap(&maps.a1);
  }
  // TMEM touches no global memory either (no kernel of this library that can
  // share an SM with this one holds TMEM)
  if (warp == 1) tmem_alloc(smem_u32(tmem_slot), G::kTmemCols);
  pdl_wait();
  // the work list's first entries load in the same round as its counts (any
  // index below the arrays' capacity may be read; those past the count go unused)
  const bool pf = (int)threadIdx.x < a.task_prefetch;
  int32_t pf_start = 0, pf_start_dn = 0;
  FfnTask pf_task{};
  if (pf) {
    pf_start = a.tile_start[threadIdx.x];
    if (FFN) pf_start_dn = a.tile_start_dn[threadIdx.x];
    pf_task = a.tasks[threadIdx.x];
  }
  const int ntasks = a.counts[a.task_slot];
  const int ntiles_first = a.counts[a.tile_slot];
  const int ntiles = ntiles_first + (FFN ? a.counts[a.tile_slot_dn] : 0);
  if (ntiles <= 0 || (int)blockIdx.x >= ntiles) {  // uniform across the CTA
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(*tmem_slot, G::kTmemCols);
    if (MODE != kTcGateUp && a.fin.ctr) finalize_if_last(a.fin);
    return;
  }
  // the work list's starts and tasks, in one round of parallel loads, so the
  // scheduler's decodes read shared memory
  int32_t* s_start = reinterpret_cast<int32_t*>(smem + G::kCacheOff);
  int32_t* s_start_dn = s_start + kTaskCache;
  FfnTask* s_tasks = reinterpret_cast<FfnTask*>(s_start_dn + kTaskCache);
  const bool cached = ntasks <= kTaskCache;
  if (cached)
    for (int i = threadIdx.x; i < ntasks; i += blockDim.x) {
      if (i < a.task_prefetch) {  // i == threadIdx.x: this thread's prefetched entry
        s_start[i] = pf_start;
        if (FFN) s_start_dn[i] = pf_start_dn;
        s_tasks[i] = pf_task;
      } else {
        s_start[i] = a.tile_start[i];
        if (FFN) s_start_dn[i] = a.tile_start_dn[i];
        s_tasks[i] = a.tasks[i];
      }
    }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const FfnTask* d_tasks = cached ? s_tasks : a.tasks;
  const int32_t* d_start = cached ? s_start : a.tile_start;
  const int32_t* d_start_dn = cached ? s_start_dn : a.tile_start_dn;
  // the shared expert's tasks come first in the work list: its row chunks and
  // its gate/up tiles (single-launch FFN)
  int sh_chunks = 0, sh_gu = 0;
  if (FFN && ntasks > 0 && d_tasks[0].expert < 0) {
    sh_chunks = d_tasks[0].chunk & 0xffff;
    sh_gu = sh_chunks * a.gu_tiles_shared;
  }

  if (warp == kSchedWarp && lane == 0) {
    // ---------------------------------------------------------- scheduler --
    // Claims and decodes tiles up to kTileQueue ahead of the producer, so the
    // claim's atomic and the decode's dependent loads never stall the rings.
    for (uint32_t n = 0;; ++n) {
      QTile t;
      t.tile = -1;
      if (!*abort_flag) {
        const int tile = atomicAdd(a.sched, 1);
        if (tile < ntiles_first)
          t = decode_tile(d_tasks,
                          interleave_tile(tile, sh_gu, sh_chunks, ntiles_first - sh_gu,
                                          (ntiles_first - sh_gu) / 2),
                          ntasks, MODE == kTcGateUp || MODE == kTcFfn, d_start);
        else if (tile < ntiles)
          t = decode_tile(d_tasks, tile - ntiles_first, ntasks, 0, d_start_dn);
      }
      if (!tq_push(tq, tq_full, tq_empty, n, t)) {
        raise_status(a.status, kStTimeout, kind);
        *abort_flag = 1;
        break;
      }
      if (t.tile < 0) {
        pdl_trigger();  // no tiles left: the next kernel may launch
        break;
      }
    }
  } else if (warp == 0 && lane == 0) {
    // ---------------------------------------------------------- producer --
    const uint64_t pol_w = policy_evict_first(), pol_x = policy_evict_last();
    uint32_t iter = 0;
    bool ok = true;
    for (uint32_t n = 0; ok; ++n) {
      QTile t;
      if (!tq_pop(tq, tq_full, tq_empty, n, &t, false)) {
        raise_status(a.status, kStTimeout, kind);
        *abort_flag = 1;
        break;
      }
      if (t.tile < 0) break;
      const bool gu = MODE == kTcGateUp || (FFN && t.gu != 0);
      const bool two = two_weight_tiles<MODE>(gu, a.dn_wide);
      const CUtensorMap* A0;
      const CUtensorMap* A1 = t.shared ? &maps.sa1 : &maps.a1;
      const CUtensorMap* B;
      int K;
      // weight rows of the tile's first box; the second box (up weights, or a
      // wide down tile's second channel half) starts at a1_row of A1
      int a0_row = t.ct * kTcM, a1_row = t.ct * kTcM;
      // a down tile's h rows are complete once all its task's gate/up tiles are
      // stored; its first stage's weight boxes are issued before that wait
      bool h_wait = false;
      int h_target = 0;
      if (FFN && !gu) {
        h_wait = true;
        h_target = 4 * (t.shared ? a.gu_tiles_shared : a.gu_tiles);
        A0 = t.shared ? &maps.sd0 : &maps.d0;
        B = t.shared ? &maps.sh : &maps.h;
        K = t.shared ? a.Ns : a.N;  // the down pass reduces over the intermediate size
        if (a.dn_wide) {
          A1 = A0;
          a0_row = t.ct * 2 * kTcM;
          a1_row = a0_row + kTcM;
        }
      } else {
        A0 = t.shared ? &maps.sa0 : &maps.a0;
        B = t.shared ? &maps.sb : &maps.b;
        K = t.shared ? a.Ks : a.K;
      }
      const int nb = (t.n + kBoxRows - 1) / kBoxRows;
      const int nks = (K + kBK - 1) / kBK;
      // single-launch FFN, down tile of <= 64 rows: two K steps per stage (each a
      // 16 KB weight tile and an 8 KB activation box), so the down tiles keep as
      // many weight bytes in flight as the gate/up tiles
      const int sub = packed_down<MODE>(gu, t.n, a.dn_wide) ? 2 : 1;
      for (int ks = 0; ks < nks; ks += sub) {
        if (*abort_flag) {
          ok = false;
          break;
        }
        const int stage = iter % G::kStages;
        const uint32_t par = (iter / G::kStages) & 1u;
        if (!mbar_wait(smem_u32(&empty[stage]), par ^ 1u)) {
          raise_status(a.status, kStTimeout, kind);
          *abort_flag = 1;
          ok = false;
          break;
        }
        const uint32_t bar = smem_u32(&full[stage]);
        uint8_t* st = smem + (size_t)stage * G::kStageBytes;
        if (sub == 2) {
          const int nsub = min(2, nks - ks);
          mbar_arrive_expect_tx(bar, (uint32_t)(nsub * (kATileBytes + kBoxBytes)));
          for (int u = 0; u < nsub; ++u)
            tma_load_3d(smem_u32(st + u * kPackedStep), A0, (ks + u) * kBK, a0_row, t.e, bar,
                        pol_w);
          if (h_wait && !wait_h_rows(a, t.task, h_target, kind, abort_flag)) ok = false;
          h_wait = false;
          // (after a failed wait the boxes still load, so the stage completes)
          for (int u = 0; u < nsub; ++u)
            tma_load_3d(smem_u32(st + u * kPackedStep + kATileBytes), B, (ks + u) * kBK, t.row0,
                        0, bar, pol_x);
          ++iter;
          if (!ok) break;
          continue;
        }
        if (MODE == kTcRouter) {
          // the three split terms' tiles of these 64 columns: K offsets 0, H, 2H
          mbar_arrive_expect_tx(bar, (uint32_t)(3 * kATileBytes + nb * kBoxBytes));
          for (int j = 0; j < 3; ++j)
            tma_load_3d(smem_u32(st + j * kATileBytes), A0, j * K + ks * kBK, t.ct * kTcM, t.e,
                        bar, pol_w);
        } else {
          mbar_arrive_expect_tx(bar, (uint32_t)((two ? 2 : 1) * kATileBytes + nb * kBoxBytes));
          tma_load_3d(smem_u32(st), A0, ks * kBK, a0_row, t.e, bar, pol_w);
          if (two)
            tma_load_3d(smem_u32(st + kATileBytes), A1, ks * kBK, a1_row, t.e, bar, pol_w);
        }
        if (h_wait && !wait_h_rows(a, t.task, h_target, kind, abort_flag)) ok = false;
        h_wait = false;
        uint8_t* sb = st + G::kNA * kATileBytes;
        const int bk = (!t.shared && a.b_kmod > 0) ? (ks * kBK) % a.b_kmod : ks * kBK;
        for (int j = 0; j < nb; ++j)
          tma_load_3d(smem_u32(sb + j * kBoxBytes), B, bk, t.row0 + j * kBoxRows, 0, bar, pol_x);
        ++iter;
        if (!ok) break;
      }
    }
    const uint32_t first = iter > (uint32_t)G::kStages ? iter - G::kStages : 0u;
    for (uint32_t j = first; j < iter; ++j)
      mbar_wait(smem_u32(&full[j % G::kStages]), (j / G::kStages) & 1u);
  } else if (warp == 1 && lane == 0) {
    // --------------------------------------------------------- MMA issuer --
    uint32_t iter = 0, local = 0;
    bool ok = true;
    for (uint32_t n = 0; ok; ++n, ++local) {
      QTile t;
      if (!tq_pop(tq, tq_full, tq_empty, n, &t, false)) {
        raise_status(a.status, kStTimeout, kind);
        *abort_flag = 1;
        break;
      }
      if (t.tile < 0) break;
      const bool gu = MODE == kTcGateUp || (FFN && t.gu != 0);
      const uint32_t buf = local & 1u, use = local >> 1;
      if (!mbar_wait(smem_u32(&acc_empty[buf]), (use & 1u) ^ 1u)) {
        raise_status(a.status, kStTimeout, kind);
        *abort_flag = 1;
        break;
      }
      tc_fence_after();
      const uint32_t nmma = (uint32_t)((t.n + 15) / 16 * 16);
      const uint32_t idesc = idesc_bf16_f32(kTcM, nmma);
      const uint32_t d0 = tmem + buf * G::kAccStride;
      const uint32_t d1 = d0 + kTcMaxN;
      const bool two = two_weight_tiles<MODE>(gu, a.dn_wide);
      const int K = (FFN && !gu) ? (t.shared ? a.Ns : a.N) : (t.shared ? a.Ks : a.K);
      const int nks = (K + kBK - 1) / kBK;
      const int sub = packed_down<MODE>(gu, t.n, a.dn_wide) ? 2 : 1;
      for (int ks = 0; ks < nks; ks += sub) {
        if (*abort_flag) {
          ok = false;
          break;
        }
        const int stage = iter % G::kStages;
        const uint32_t par = (iter / G::kStages) & 1u;
        if (!mbar_wait(smem_u32(&full[stage]), par)) {
          raise_status(a.status, kStTimeout, kind);
          *abort_flag = 1;
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t sa = smem_u32(smem + (size_t)stage * G::kStageBytes);
        if (sub == 2) {
          const int nsub = min(2, nks - ks);
          for (int u = 0; u < nsub; ++u) {
            const uint32_t su = sa + u * kPackedStep;
#pragma unroll
            for (int k = 0; k < kBK / 16; ++k) {
              const uint32_t acc = (ks + u > 0 || k > 0) ? 1u : 0u;
              tc_mma_bf16(d0, sdesc_sw128(su + k * 32), sdesc_sw128(su + kATileBytes + k * 32),
                          idesc, acc);
            }
          }
          tc_commit(smem_u32(&empty[stage]));
          ++iter;
          continue;
        }
        const uint32_t sb = sa + G::kNA * kATileBytes;
#pragma unroll
        for (int k = 0; k < kBK / 16; ++k) {
          const uint64_t bdesc = sdesc_sw128(sb + k * 32);
          const uint32_t acc = (ks > 0 || k > 0) ? 1u : 0u;
          if (MODE == kTcRouter) {
            tc_mma_bf16(d0, sdesc_sw128(sa + k * 32), bdesc, idesc, acc);                    // W3
            tc_mma_bf16(d0, sdesc_sw128(sa + kATileBytes + k * 32), bdesc, idesc, 1u);      // W2
            tc_mma_bf16(d1, sdesc_sw128(sa + 2 * kATileBytes + k * 32), bdesc, idesc, acc);  // W1
          } else {
            tc_mma_bf16(d0, sdesc_sw128(sa + k * 32), bdesc, idesc, acc);
            if (two) tc_mma_bf16(d1, sdesc_sw128(sa + kATileBytes + k * 32), bdesc, idesc, acc);
          }
        }
        tc_commit(smem_u32(&empty[stage]));
        ++iter;
      }
      if (!ok) break;
      tc_commit(smem_u32(&acc_full[buf]));
    }
    if (*abort_flag) {  // let issued MMAs finish before TMEM is released
      tc_commit(smem_u32(drain));
      mbar_wait(smem_u32(drain), 0u);
    }
  } else if (warp >= 2 && warp < kSchedWarp) {  // warps 2-5
    // ----------------------------------------------------------- epilogue --
    const int q = warp % 4;  // TMEM lane quadrant this warp may access
    uint32_t local = 0;
    for (uint32_t n = 0;; ++n, ++local) {
      QTile t;
      if (!tq_pop(tq, tq_full, tq_empty, n, &t, true)) {
        if (lane == 0) raise_status(a.status, kStTimeout, kind);
        *abort_flag = 1;
        break;
      }
      if (t.tile < 0 || warp_flag(abort_flag)) break;
      const bool gu = MODE == kTcGateUp || (FFN && t.gu != 0);
      // output channels of this tile's pass: gate/up -> N (I or I_s); down -> H
      const int tN = (FFN && !gu) ? a.K : (t.shared ? a.Ns : a.N);
      // a wide down tile's second accumulator holds channels ch + kTcM
      const bool wide = FFN && !gu && a.dn_wide;
      const uint32_t buf = local & 1u, use = local >> 1;
      if (!warp_wait(smem_u32(&acc_full[buf]), use & 1u)) {
        if (lane == 0) raise_status(a.status, kStTimeout, kind);
        *abort_flag = 1;
        break;
      }
      tc_fence_after();
      const int ch = t.ct * (wide ? 2 * kTcM : kTcM) + q * 32 + lane;
      const uint32_t trow = tmem + ((uint32_t)(q * 32) << 16) + buf * G::kAccStride;
      const bool fused = !gu && a.sc.acc != nullptr;
      for (int j0 = 0; j0 < t.n; j0 += 16) {
        // fused combine: lane i < 16 looks up token j0 + i's target row and
        // routing weight while the accumulators are loaded
        int tk_l = 0;
        float wt_l = 0.f;
        if (fused && lane < 16 && j0 + lane < t.n)
          scatter_target(a.sc, t.row0 + j0 + lane, t.shared, &tk_l, &wt_l);
        uint32_t g[16], u[16];
        tmem_ld16(trow + j0, g);
        if (gu || MODE == kTcRouter || wide) tmem_ld16(trow + kTcMaxN + j0, u);
        tmem_ld_wait();
        if (fused) {
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int tk = __shfl_sync(0xffffffffu, tk_l, i);
            const float wt = __shfl_sync(0xffffffffu, wt_l, i);
            if (j0 + i < t.n) {
              float* arow = a.sc.acc + (size_t)tk * tN;
              if (ch < tN) atomicAdd(arow + ch, wt * __uint_as_float(g[i]));
              if (wide && ch + kTcM < tN) atomicAdd(arow + ch + kTcM, wt * __uint_as_float(u[i]));
            }
          }
        } else if (wide) {
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int tok = j0 + i;
            if (tok < t.n) {
              float* yrow = (t.shared ? a.sout_y : a.out_y) + (size_t)(t.row0 + tok) * tN;
              if (ch < tN) yrow[ch] = __uint_as_float(g[i]);
              if (ch + kTcM < tN) yrow[ch + kTcM] = __uint_as_float(u[i]);
            }
          }
        } else if (ch < tN) {
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int tok = j0 + i;
            if (tok < t.n) {
              const size_t o = (size_t)(t.row0 + tok) * tN + ch;
              const float gv = __uint_as_float(g[i]);
              if (gu) {
                const float h = gv * __frcp_rn(1.f + __expf(-gv)) * __uint_as_float(u[i]);
                (t.shared ? a.sout_h : a.out_h)[o] = f_to_bf16(h);
              } else if (MODE == kTcRouter) {
                a.out_y[o] = gv + __uint_as_float(u[i]);  // small terms + W1 terms
              } else {
                (t.shared ? a.sout_y : a.out_y)[o] = gv;
              }
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(smem_u32(&acc_empty[buf]));
        // single-launch FFN: this warp's h rows of the tile are stored
        if (FFN && gu) signal_rows_done(a.gu_done + t.task);
      }
    }
  }

  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, G::kTmemCols);
  }
  if (MODE != kTcGateUp && a.fin.ctr) finalize_if_last(a.fin);
}

// ------------------------------------------------------------ host side --
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// bf16 [outer][rows][K] tensor, box = 64 (K) x box_rows x 1, 128-byte swizzle,
// out-of-range elements read as zero.
bool make_map(CUtensorMap* m, const void* base, uint64_t K, uint64_t rows, uint64_t outer,
              uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn || !base) return false;
  const cuuint64_t dims[3] = {K, rows, outer};
  const cuuint64_t strides[2] = {K * 2, rows * K * 2};
  const cuuint32_t box[3] = {(cuuint32_t)kBK, box_rows, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Router work list: token chunks of <= 128 rows, all expert tiles of each.
__global__ void router_tasks_kernel(FfnTask* tasks, int32_t* start, int32_t* counts, int T,
                                    int ctiles) {
  pdl_enter();
  const int nt = (T + kTcMaxN - 1) / kTcMaxN;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < nt; i += gridDim.x * blockDim.x) {
    FfnTask tk;
    tk.expert = 0;
    tk.row0 = i * kTcMaxN;
    tk.nrows = min(kTcMaxN, T - i * kTcMaxN);
    tk.chunk = (i << 16) | nt;
    tasks[i] = tk;
    start[i] = i * ctiles;
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    counts[kWlTcTasks] = nt;
    counts[kWlTcTilesDN] = nt * ctiles;
    counts[kWlSchedDN] = 0;
  }
}

TcArgs make_args(const Launch& L, const TcPass& p) {
  TcArgs a{};
  a.tasks = p.tasks;
  a.tile_start = p.tile_start;
  a.counts = p.counts;
  a.task_slot = p.task_slot;
  a.tile_slot = p.tile_slot;
  a.out_h = p.out_h;
  a.out_y = p.out_y;
  a.sout_h = p.sout_h;
  a.sout_y = p.sout_y;
  a.K = p.K;
  a.Ks = p.Ks;
  a.N = p.N;
  a.Ns = p.Ns;
  a.b_kmod = p.b_kmod;
  a.sched = const_cast<int32_t*>(p.counts) + p.sched_slot;
  a.status = L.status;
  a.sc = p.sc;
  a.fin = p.fin;
  a.task_prefetch = p.task_cap < kThreads ? p.task_cap : kThreads;
  return a;
}

// Tensor maps of one pass's weights and activation rows (routed, then shared).
bool pass_maps(const TcPass& p, bool gu, CUtensorMap* w0, CUtensorMap* w1, CUtensorMap* act,
               CUtensorMap* sw0, CUtensorMap* sw1, CUtensorMap* sact) {
  const uint64_t Kr = p.K, Nr = p.N;
  const uint64_t Kb = p.b_kmod > 0 ? (uint64_t)p.b_kmod : Kr;  // activation row length
  bool ok = make_map(w0, p.w0, Kr, Nr, p.n_experts, kTcM) &&
            make_map(act, p.act, Kb, p.act_rows, 1, kBoxRows);
  if (gu) ok = ok && make_map(w1, p.w1, Kr, Nr, p.n_experts, kTcM);
  if (p.sw0) {
    ok = ok && make_map(sw0, p.sw0, p.Ks, p.Ns, 1, kTcM) &&
         make_map(sact, p.sact, p.Ks, p.sact_rows, 1, kBoxRows);
    if (gu) ok = ok && make_map(sw1, p.sw1, p.Ks, p.Ns, 1, kTcM);
  }
  return ok;
}

template <int MODE>
bool launch_tc(const Launch& L, const TcPass& p, int kind) {
  using G = Geom<MODE>;
  TcMaps maps;
  memset(&maps, 0, sizeof maps);
  if (!pass_maps(p, MODE == kTcGateUp, &maps.a0, &maps.a1, &maps.b, &maps.sa0, &maps.sa1,
                 &maps.sb))
    return false;
  const TcArgs a = make_args(L, p);
  set_smem_attr_once(reinterpret_cast<const void*>(tc_kernel<MODE>), G::kSmemBytes,
                     MODE == kTcGateUp ? kAttrTcGU : kAttrTcDN);
  launch_begin(L, kind);
  launch_kernel(tc_kernel<MODE>, L.num_sms, kThreads, G::kSmemBytes, L.stream, maps, a);
  launch_end(L, kind);
  return true;
}

}  // namespace

bool launch_tc_gate_up(const Launch& L, const TcPass& p) {
  return launch_tc<kTcGateUp>(L, p, MOE_K_TC_GATE_UP);
}
bool launch_tc_down(const Launch& L, const TcPass& p) {
  return launch_tc<kTcDown>(L, p, MOE_K_TC_DOWN);
}

bool launch_tc_ffn(const Launch& L, const TcPass& gu, const TcPass& dn, int32_t* gu_done) {
  using G = Geom<kTcFfn>;
  TcMaps maps;
  memset(&maps, 0, sizeof maps);
  CUtensorMap unused;
  if (!pass_maps(gu, true, &maps.a0, &maps.a1, &maps.b, &maps.sa0, &maps.sa1, &maps.sb) ||
      !pass_maps(dn, false, &maps.d0, &unused, &maps.h, &maps.sd0, &unused, &maps.sh))
    return false;
  TcArgs a = make_args(L, gu);
  a.out_y = dn.out_y;
  a.sout_y = dn.sout_y;
  a.sc = dn.sc;
  a.fin = dn.fin;
  a.tile_start_dn = dn.tile_start;
  a.tile_slot_dn = dn.tile_slot;
  a.gu_done = gu_done;
  a.gu_tiles = (gu.N + kTcM - 1) / kTcM;
  a.gu_tiles_shared = (gu.Ns + kTcM - 1) / kTcM;
  a.dn_wide = dn.dn_wide;
  set_smem_attr_once(reinterpret_cast<const void*>(tc_kernel<kTcFfn>), G::kSmemBytes, kAttrTcFfn);
  launch_begin(L, MOE_K_TC_GATE_UP);
  launch_kernel(tc_kernel<kTcFfn>, L.num_sms, kThreads, G::kSmemBytes, L.stream, maps, a);
  launch_end(L, MOE_K_TC_GATE_UP);
  return true;
}

bool launch_tc_router(const Launch& L, const moe_config& c, int T, const void* x,
                      const uint16_t* w_split, FfnTask* tasks, int32_t* start, int32_t* counts,
                      float* logits) {
  const int E = c.n_routed + c.n_zero;
  const int ctiles = (E + kTcM - 1) / kTcM;
  const int nt = (T + kTcMaxN - 1) / kTcMaxN;
  launch_begin(L, MOE_K_ROUTER);
  launch_kernel(router_tasks_kernel, (nt + 255) / 256, 256, 0, L.stream, tasks, start, counts, T,
                ctiles);
  launch_end(L, MOE_K_ROUTER);
  TcPass p{};
  p.tasks = tasks;
  p.tile_start = start;
  p.counts = counts;
  p.task_slot = kWlTcTasks;
  p.tile_slot = kWlTcTilesDN;
  p.sched_slot = kWlSchedDN;
  p.w0 = w_split;
  p.n_experts = 1;
  p.act = x;
  p.act_rows = T;
  p.out_y = logits;
  p.K = c.hidden;  // K steps over H; each loads the three terms' tiles
  p.N = E;
  using G = Geom<kTcRouter>;
  TcMaps maps;
  memset(&maps, 0, sizeof maps);
  if (!make_map(&maps.a0, w_split, 3 * (uint64_t)c.hidden, E, 1, kTcM) ||
      !make_map(&maps.b, x, c.hidden, T, 1, kBoxRows))
    return false;
  const TcArgs a = make_args(L, p);
  set_smem_attr_once(reinterpret_cast<const void*>(tc_kernel<kTcRouter>), G::kSmemBytes,
                     kAttrTcRouter);
  launch_begin(L, MOE_K_ROUTER);
  launch_kernel(tc_kernel<kTcRouter>, L.num_sms, kThreads, G::kSmemBytes, L.stream, maps, a);
  launch_end(L, MOE_K_ROUTER);
  return true;
}

}  // namespace moe
