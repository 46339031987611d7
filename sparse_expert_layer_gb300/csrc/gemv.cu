// Grouped SwiGLU FFN, streaming path for lightly loaded experts.
//
// The Pangu Pro MoE disclosure (section SwiftGMM) names moving routed-expert
// weights as the decode bottleneck and switches between GEMV and GEMM by load.
// This is the GEMV side: each expert's weights are read from HBM exactly once
// and dotted with its few activation rows on CUDA cores.
//
// Work item = (task, block of output channels); a task is <= NR (1, 2, 4 or 8)
// rows of one expert.  Persistent CTAs (one per SM) walk the items round-robin.
//   warp 0     : producer.  Streams 1024-element slices of 16 weight rows and
//                of the task's activation rows into a shared-memory ring (as many
//                stages as fit in 200 KB: 5 to 6 at NR <= 4, 4 at NR = 8)
//                with cp.async.bulk (weights marked evict-first in L2).
//   warps 1..8 : consumers.  Warp w owns two weight rows -- (gate c, up c) in
//                the gate/up pass, (c, c+1) in the down pass -- and its lanes
//                split the slice; packed fp32x2 FMAs accumulate over all
//                slices, a butterfly reduces at the end of the item.
//   gate/up epilogue: h = silu(g) * u, stored bf16.  down epilogue: y fp32.
#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace moe {

namespace {

constexpr int kConsumerWarps = 8;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kKS = 1024;                      // elements per row slice
constexpr int kSliceBytes = kKS * 2;           // bytes per row slice
constexpr int kWRows = 2 * kConsumerWarps;     // weight row slices per stage
constexpr int kRingBudget = 200 * 1024;        // shared memory for the ring
constexpr int kStartsCache = 2048;             // item starts kept in shared memory

// A stage holds the 16 weight row slices plus room for NR activation slices, so
// a smaller row cap leaves room for more stages (more bytes in flight).
template <int NR>
struct Ring {
  static constexpr int kStageBytes = (kWRows + NR) * kSliceBytes;
  static constexpr int kStages = kRingBudget / kStageBytes < 8 ? kRingBudget / kStageBytes : 8;
  static constexpr int kBarOffset = kStages * kStageBytes;
  static constexpr int kStartsOffset = kBarOffset + 256;  // cached item starts
  static constexpr int kSmemBytes = kStartsOffset + kStartsCache * 4;
};

union F2 {
  float2 f;
  unsigned long long u;
};
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
  F2 A, B, C, D;
  A.f = a;
  B.f = b;
  C.f = c;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(D.u) : "l"(A.u), "l"(B.u), "l"(C.u));
  return D.f;
}
__device__ __forceinline__ float2 unpack2(uint32_t v) { return make_float2(bf16lo(v), bf16hi(v)); }

struct Item {
  const uint16_t* w0;   // first weight row of the block's matrix (gate or down)
  const uint16_t* w1;   // up rows (gate/up pass)
  const uint16_t* act;  // first activation row of the task
  uint16_t* out_h;
  float* out_y;
  int n, row0, N, c0, K;
  bool shared;
};

template <bool GU>
__device__ __forceinline__ void decode_item(const GemvPass& p, const int32_t* starts, int item,
                                            int ntasks, Item& it) {
  int lo = 0, hi = ntasks - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (starts[mid] <= item)
      lo = mid;
    else
      hi = mid - 1;
  }
  const FfnTask tk = p.tasks[lo];
  const int block = item - starts[lo];
  const bool shared = tk.expert < 0;
  it.n = tk.nrows;
  it.row0 = tk.row0;
  it.shared = shared;
  it.N = shared ? p.Ns : p.N;
  it.K = shared ? p.Ks : p.K;
  it.c0 = block * (GU ? kGemvChGU : kGemvChDN);
  const size_t mat = (size_t)p.N * p.K;
  it.w0 = shared ? p.sw0 : p.w0 + (size_t)tk.expert * mat;
  it.w1 = GU ? (shared ? p.sw1 : p.w1 + (size_t)tk.expert * mat) : nullptr;
  it.act = (shared ? p.sact : p.act) + (size_t)tk.row0 * it.K;
  it.out_h = shared ? p.sout_h : p.out_h;
  it.out_y = shared ? p.sout_y : p.out_y;
}

// Row of the block that weight slice j (0..15) of a stage holds; -1 if past N.
template <bool GU>
__device__ __forceinline__ const uint16_t* weight_row(const Item& it, int j) {
  if (GU) {
    const int c = it.c0 + (j % kGemvChGU);
    if (c >= it.N) return nullptr;
    return (j < kGemvChGU ? it.w0 : it.w1) + (size_t)c * it.K;
  }
  const int c = it.c0 + j;
  if (c >= it.N) return nullptr;
  return it.w0 + (size_t)c * it.K;
}

template <bool GU, int NR, int RING>
__device__ bool consume_item(const GemvPass& p, const Item& it, uint8_t* smem, uint64_t* full,
                             uint64_t* empty, volatile int* abort_flag, uint32_t& iter, int cw,
                             int lane, DevStatus* st) {
  using G = Ring<RING>;
  float2 acc0[NR], acc1[NR];
#pragma unroll
  for (int r = 0; r < NR; ++r) acc0[r] = acc1[r] = make_float2(0.f, 0.f);
  const int n = it.n;
  const int sa = GU ? cw : 2 * cw;                 // weight slices this warp reads
  const int sb = GU ? kGemvChGU + cw : 2 * cw + 1;
  const int nsl = (it.K + kKS - 1) / kKS;
  for (int s = 0; s < nsl; ++s, ++iter) {
    if (*abort_flag) return false;
    const int stage = iter % G::kStages;
    const uint32_t par = (iter / G::kStages) & 1u;
    if (!mbar_wait(smem_u32(&full[stage]), par)) {
      if (lane == 0) raise_status(st, kStTimeout, GU ? MOE_K_GEMV_GATE_UP : MOE_K_GEMV_DOWN);
      *abort_flag = 1;
      return false;
    }
    const uint8_t* sbase = smem + (size_t)stage * G::kStageBytes;
    const uint4* wa = reinterpret_cast<const uint4*>(sbase + sa * kSliceBytes);
    const uint4* wb = reinterpret_cast<const uint4*>(sbase + sb * kSliceBytes);
    const uint4* xs = reinterpret_cast<const uint4*>(sbase + kWRows * kSliceBytes);
    const int nchunks = min(kKS, it.K - s * kKS) / 8;
    for (int c = lane; c < nchunks; c += 32) {
      const uint4 A = wa[c], B = wb[c];
      const float2 a0 = unpack2(A.x), a1 = unpack2(A.y), a2 = unpack2(A.z), a3 = unpack2(A.w);
      const float2 b0 = unpack2(B.x), b1 = unpack2(B.y), b2 = unpack2(B.z), b3 = unpack2(B.w);
#pragma unroll
      for (int r = 0; r < NR; ++r) {
        if (r < n) {
          const uint4 X = xs[r * (kSliceBytes / 16) + c];
          const float2 x0 = unpack2(X.x), x1 = unpack2(X.y), x2 = unpack2(X.z),
                       x3 = unpack2(X.w);
          acc0[r] = ffma2(a0, x0, acc0[r]);
          acc1[r] = ffma2(b0, x0, acc1[r]);
          acc0[r] = ffma2(a1, x1, acc0[r]);
          acc1[r] = ffma2(b1, x1, acc1[r]);
          acc0[r] = ffma2(a2, x2, acc0[r]);
          acc1[r] = ffma2(b2, x2, acc1[r]);
          acc0[r] = ffma2(a3, x3, acc0[r]);
          acc1[r] = ffma2(b3, x3, acc1[r]);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&empty[stage]));
  }
  // epilogue
#pragma unroll
  for (int r = 0; r < NR; ++r) {
    if (r < n) {
      const float g = warp_sum(acc0[r].x + acc0[r].y);
      const float u = warp_sum(acc1[r].x + acc1[r].y);
      if (lane == r) {
        const size_t row = (size_t)(it.row0 + r) * it.N;
        if (GU) {
          const int c = it.c0 + cw;
          if (c < it.N) it.out_h[row + c] = f_to_bf16(g / (1.f + expf(-g)) * u);
        } else if (p.sc.acc) {  // fused combine: add w * y into the token's row
          int tk;
          float wt;
          scatter_target(p.sc, it.row0 + r, it.shared, &tk, &wt);
          float* dst = p.sc.acc + (size_t)tk * it.N;
          const int c = it.c0 + 2 * cw;
          if (c < it.N) atomicAdd(dst + c, wt * g);
          if (c + 1 < it.N) atomicAdd(dst + c + 1, wt * u);
        } else {
          const int c = it.c0 + 2 * cw;
          if (c < it.N) it.out_y[row + c] = g;
          if (c + 1 < it.N) it.out_y[row + c + 1] = u;
        }
      }
    }
  }
  return true;
}

template <bool GU, int NR>
__global__ void __launch_bounds__(kThreads, 1) gemv_kernel(GemvPass p, DevStatus* st) {
  pdl_wait();
  using G = Ring<NR>;
  extern __shared__ __align__(16) uint8_t smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + G::kBarOffset);
  uint64_t* empty = full + G::kStages;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + G::kStages);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (threadIdx.x == 0) {
    for (int s = 0; s < G::kStages; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), kConsumerWarps);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  const int ntasks = p.counts[p.task_slot];
  const int nitems = p.counts[p.item_slot];
  // The tasks' first items, for the per-item binary search: in shared memory
  // when they fit, so a search costs a few shared loads instead of a chain of
  // dependent global loads.
  int32_t* cache = reinterpret_cast<int32_t*>(smem + G::kStartsOffset);
  const bool cached = ntasks <= kStartsCache;
  if (cached)
    for (int i = threadIdx.x; i < ntasks; i += blockDim.x) cache[i] = p.item_start[i];
  const int32_t* starts = cached ? cache : p.item_start;
  __syncthreads();
  uint32_t iter = 0;

  if (warp == 0) {
    const uint64_t pol_w = policy_evict_first(), pol_x = policy_evict_last();
    bool ok = true;
    // the next item is decoded one item ahead, so its task load is in flight
    // while the current item's copies are issued
    Item nit;
    if ((int)blockIdx.x < nitems) decode_item<GU>(p, starts, blockIdx.x, ntasks, nit);
    for (int item = blockIdx.x; ok && item < nitems; item += gridDim.x) {
      const Item it = nit;
      if (item + (int)gridDim.x < nitems) decode_item<GU>(p, starts, item + gridDim.x, ntasks, nit);
      const int chans = GU ? kGemvChGU : kGemvChDN;
      const int vrows = min(chans, it.N - it.c0);
      const int wrows = GU ? 2 * vrows : vrows;
      const uint16_t* wrow = weight_row<GU>(it, lane % kWRows);
      const int nsl = (it.K + kKS - 1) / kKS;
      for (int s = 0; s < nsl; ++s) {
        if (*abort_flag) {
          ok = false;
          break;
        }
        const int stage = iter % G::kStages;
        const uint32_t par = (iter / G::kStages) & 1u;
        if (!mbar_wait(smem_u32(&empty[stage]), par ^ 1u)) {
          if (lane == 0) raise_status(st, kStTimeout, GU ? MOE_K_GEMV_GATE_UP : MOE_K_GEMV_DOWN);
          *abort_flag = 1;
          ok = false;
          break;
        }
        const int len = min(kKS, it.K - s * kKS);
        const uint32_t bytes = (uint32_t)len * 2u;
        const uint32_t bar = smem_u32(&full[stage]);
        if (lane == 0) mbar_arrive_expect_tx(bar, (uint32_t)(wrows + it.n) * bytes);
        __syncwarp();
        const uint32_t sbase = smem_u32(smem + (size_t)stage * G::kStageBytes);
        if (lane < kWRows) {
          if (wrow) bulk_g2s(sbase + lane * kSliceBytes, wrow + (size_t)s * kKS, bytes, bar, pol_w);
        } else if (lane - kWRows < it.n) {
          const int a = lane - kWRows;
          bulk_g2s(sbase + (kWRows + a) * kSliceBytes, it.act + (size_t)a * it.K + (size_t)s * kKS,
                   bytes, bar, pol_x);
        }
        ++iter;
      }
    }
    // Drain: every issued copy lands before the CTA may exit.
    if (lane == 0) {
      const uint32_t first = iter > (uint32_t)G::kStages ? iter - G::kStages : 0u;
      for (uint32_t j = first; j < iter; ++j)
        mbar_wait(smem_u32(&full[j % G::kStages]), (j / G::kStages) & 1u);
    }
    return;
  }

  const int cw = warp - 1;
  Item nit;
  if ((int)blockIdx.x < nitems) decode_item<GU>(p, starts, blockIdx.x, ntasks, nit);
  for (int item = blockIdx.x; item < nitems; item += gridDim.x) {
    const Item it = nit;  // decoded one item ahead, like the producer's
    if (item + (int)gridDim.x < nitems) decode_item<GU>(p, starts, item + gridDim.x, ntasks, nit);
    bool ok;
    if (NR == 1 || it.n <= 1)
      ok = consume_item<GU, 1, NR>(p, it, smem, full, empty, abort_flag, iter, cw, lane, st);
    else if (NR == 2 || it.n <= 2)
      ok = consume_item<GU, (NR < 2 ? NR : 2), NR>(p, it, smem, full, empty, abort_flag, iter, cw,
                                                   lane, st);
    else if (NR == 4 || it.n <= 4)
      ok = consume_item<GU, (NR < 4 ? NR : 4), NR>(p, it, smem, full, empty, abort_flag, iter, cw,
                                                   lane, st);
    else
      ok = consume_item<GU, NR, NR>(p, it, smem, full, empty, abort_flag, iter, cw, lane, st);
    if (!ok) break;
  }
}

template <bool GU, int NR>
void launch_nr(const Launch& L, const GemvPass& p) {
  using G = Ring<NR>;
  const int kind = GU ? MOE_K_GEMV_GATE_UP : MOE_K_GEMV_DOWN;
  const int nr_slot = NR == 1 ? 0 : NR == 2 ? 1 : NR == 4 ? 2 : 3;
  set_smem_attr_once(reinterpret_cast<const void*>(gemv_kernel<GU, NR>), G::kSmemBytes,
                     kAttrGemvBase + (GU ? 0 : 1) + 2 * nr_slot);
  launch_begin(L, kind);
  launch_kernel(gemv_kernel<GU, NR>, L.num_sms, kThreads, G::kSmemBytes, L.stream, p, L.status);
  launch_end(L, kind);
}

template <bool GU>
void launch_gemv(const Launch& L, const GemvPass& p) {
  switch (p.max_rows) {
    case 1: launch_nr<GU, 1>(L, p); break;
    case 2: launch_nr<GU, 2>(L, p); break;
    case 4: launch_nr<GU, 4>(L, p); break;
    default: launch_nr<GU, 8>(L, p); break;
  }
}

}  // namespace

void launch_gemv_gate_up(const Launch& L, const GemvPass& p) { launch_gemv<true>(L, p); }
void launch_gemv_down(const Launch& L, const GemvPass& p) { launch_gemv<false>(L, p); }

}  // namespace moe
