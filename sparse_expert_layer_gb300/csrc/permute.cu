// Stable re-sort of the token picks by expert (InitialRouting in the DeepSeek-V3/R1
// on Ascend article, section "2. MOE 算子优化"), the row gather, and the grouped-FFN
// work list.
//
//  count   : one CTA per block of 256 tokens counts its picks per expert (smem
//            atomics) -> block_counts[b][e].
//  scan    : one CTA turns block counts into counts[e], offsets[e] and the first
//            sorted position of block b within expert e.
//  scatter : one CTA per token block; a [expert][token] bitmap in smem gives each
//            pick its rank among the block's earlier tokens of the same expert,
//            so the order inside an expert is by token (stable).
//  gather  : one warp per pick copies the token row to its sorted position with
//            128-bit loads/stores (W8A8: quantises the row on the way).
#include <math.h>

#include "common.cuh"
#include "internal.h"
#include "topk.cuh"

namespace moe {

namespace {

constexpr int kPermThreads = 256;
constexpr int kWords = kPermTokens / 32;

__global__ void __launch_bounds__(kPermThreads)
    perm_count_kernel(const int32_t* ids, int32_t* bc, int T, int k, int E, DevStatus* st) {
  pdl_enter();
  extern __shared__ int32_t cnt[];
  const int b = blockIdx.x;
  for (int e = threadIdx.x; e < E; e += kPermThreads) cnt[e] = 0;
  __syncthreads();
  const int r0 = b * kPermTokens * k, r1 = min(T, (b + 1) * kPermTokens) * k;
  for (int r = r0 + threadIdx.x; r < r1; r += kPermThreads) {
    const int e = ids[r];
    if ((unsigned)e >= (unsigned)E) {
      raise_status(st, kStBadId, MOE_K_PERM_COUNT);
      continue;
    }
    atomicAdd(&cnt[e], 1);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += kPermThreads) bc[(size_t)b * E + e] = cnt[e];
}

__global__ void __launch_bounds__(1024)
    perm_scan_kernel(int32_t* bc, int32_t* counts, int32_t* offsets, int nblk, int E) {
  pdl_enter();
  __shared__ int32_t warp_tot[32];
  __shared__ int32_t carry;
  const int tid = threadIdx.x, lane = tid % 32, warp = tid / 32;
  // per expert: exclusive prefix over blocks (in place) and the total
  for (int e = tid; e < E; e += 1024) {
    int run = 0;
    for (int b = 0; b < nblk; ++b) {
      const int v = bc[(size_t)b * E + e];
      bc[(size_t)b * E + e] = run;
      run += v;
    }
    counts[e] = run;
  }
  if (tid == 0) carry = 0;
  __syncthreads();
  // exclusive scan of counts -> offsets, 1024 experts per round
  for (int base = 0; base < E; base += 1024) {
    const int e = base + tid;
    const int v = e < E ? counts[e] : 0;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += n;
    }
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    if (warp == 0) {
      int w = warp_tot[lane];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, w, o);
        if (lane >= o) w += n;
      }
      warp_tot[lane] = w;  // inclusive over warps
    }
    __syncthreads();
    const int excl = carry + (warp > 0 ? warp_tot[warp - 1] : 0) + incl - v;
    if (e < E) offsets[e] = excl;
    __syncthreads();
    if (tid == 1023) carry = excl + v;
    __syncthreads();
  }
  if (tid == 0) offsets[E] = carry;
  __syncthreads();
  for (int e = tid; e < E; e += 1024) {
    const int off = offsets[e];
    for (int b = 0; b < nblk; ++b) bc[(size_t)b * E + e] += off;
  }
}

__global__ void __launch_bounds__(kPermThreads)
    perm_scatter_kernel(const int32_t* ids, const int32_t* base, int32_t* s2e, int32_t* e2s, int T,
                        int k, int E) {
  pdl_enter();
  extern __shared__ uint32_t bm[];  // [E][kWords]
  const int b = blockIdx.x;
  for (int i = threadIdx.x; i < E * kWords; i += kPermThreads) bm[i] = 0u;
  __syncthreads();
  const int t0 = b * kPermTokens;
  const int r0 = t0 * k, r1 = min(T, t0 + kPermTokens) * k;
  for (int r = r0 + threadIdx.x; r < r1; r += kPermThreads) {
    const int e = ids[r];
    if ((unsigned)e >= (unsigned)E) continue;
    const int tl = r / k - t0;
    atomicOr(&bm[e * kWords + tl / 32], 1u << (tl % 32));
  }
  __syncthreads();
  for (int r = r0 + threadIdx.x; r < r1; r += kPermThreads) {
    const int e = ids[r];
    if ((unsigned)e >= (unsigned)E) {
      e2s[r] = -1;
      continue;
    }
    const int tl = r / k - t0;
    int rank = 0;
    for (int w = 0; w < tl / 32; ++w) rank += __popc(bm[e * kWords + w]);
    rank += __popc(bm[e * kWords + tl / 32] & ((1u << (tl % 32)) - 1u));
    const int p = base[(size_t)b * E + e] + rank;
    s2e[p] = r;
    e2s[r] = p;
  }
}

struct GatherArgs {
  const int32_t* ids;
  const int32_t* e2s;
  const uint16_t* x;
  void* x_perm;
  float* scale;
  const float* w;  // fused combine: routing weights and the tokens' accumulators
  float* acc;      // (nullptr: no accumulator rows to start)
  int R, k, H, E_r, E, w8a8, gather_blocks;
};

__global__ void __launch_bounds__(256) perm_gather_kernel(GatherArgs a) {
  pdl_enter();
  const int lane = threadIdx.x % 32;
  if ((int)blockIdx.x >= a.gather_blocks) {
    // fused combine: the tokens' accumulator rows start with their
    // zero-computation picks' w * x (the down pass adds the expert outputs);
    // one thread per 8 elements
    const int per_row = a.H / 8;
    const long long idx = (long long)(blockIdx.x - a.gather_blocks) * blockDim.x + threadIdx.x;
    const int t = (int)(idx / per_row);
    if (t < a.R / a.k)
      zero_pick_init(a.ids, a.w, t, a.k, a.E_r, a.E, a.x + (size_t)t * a.H,
                     a.acc + (size_t)t * a.H, a.H, (int)(idx % per_row), per_row);
    return;
  }
  const int r = blockIdx.x * 8 + threadIdx.x / 32;
  if (r >= a.R) return;
  const int e = a.ids[r];
  if ((unsigned)e >= (unsigned)a.E_r) return;  // zero-computation expert or bad id
  const int p = a.e2s[r];
  if (p < 0) return;
  const int t = r / a.k;
  const uint4* src = reinterpret_cast<const uint4*>(a.x + (size_t)t * a.H);
  const int nv = a.H / 8;
  if (!a.w8a8) {
    uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(a.x_perm) + (size_t)p * a.H);
    for (int i = lane; i < nv; i += 32) dst[i] = __ldg(src + i);
    return;
  }
  // W8A8: symmetric per-row int8, scale = amax / 127, round half to even.
  float amax = 0.f;
  for (int i = lane; i < nv; i += 32) {
    const uint4 v = __ldg(src + i);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) amax = fmaxf(amax, fmaxf(fabsf(bf16lo(w[j])), fabsf(bf16hi(w[j]))));
  }
  amax = warp_max(amax);
  const float s = amax / 127.0f;
  if (lane == 0) a.scale[p] = s;
  uint2* dst = reinterpret_cast<uint2*>(static_cast<int8_t*>(a.x_perm) + (size_t)p * a.H);
  for (int i = lane; i < nv; i += 32) {
    const uint4 v = __ldg(src + i);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t q[2] = {0u, 0u};
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float f = (j & 1) ? bf16hi(w[j / 2]) : bf16lo(w[j / 2]);
      int qi = 0;
      if (amax > 0.f) qi = (int)fminf(127.f, fmaxf(-127.f, rintf(f / s)));
      q[j / 4] |= (uint32_t)(qi & 0xff) << (8 * (j % 4));
    }
    dst[i] = make_uint2(q[0], q[1]);
  }
}

// Work list of the grouped FFN.  Units are the shared expert first (its tiles,
// the heaviest, start early instead of running at the pass's tail), then the
// routed experts in index order.  A unit with n rows becomes GEMV tasks of <= gemv_chunk
// rows when n <= gemv_max, else tensor-core tasks of <= tc_chunk rows.
struct WlArgs {
  const int32_t* offsets;
  WorkList wl;
  int E_r, T, has_shared, gemv_max, gemv_chunk, tc_chunk;
  int items_gu, items_gu_shared, items_dn;        // GEMV items per task
  int tiles_gu, tiles_gu_shared, tiles_dn;        // tensor-core tiles per task
  DevStatus* status;
};

__device__ int block_exclusive_scan(int v, int* tot, int* sh) {
  const int lane = threadIdx.x % 32, warp = threadIdx.x / 32;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += n;
  }
  if (lane == 31) sh[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = lane < (int)(blockDim.x / 32) ? sh[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += n;
    }
    sh[lane] = w;
  }
  __syncthreads();
  const int excl = (warp > 0 ? sh[warp - 1] : 0) + incl - v;
  *tot = sh[blockDim.x / 32 - 1];
  __syncthreads();
  return excl;
}

// Exclusive scans of N values per thread across the block at once (three block
// barriers for all N); sh holds 32 * N ints.
template <int N>
__device__ void block_exclusive_scan_n(const int (&v)[N], int (&excl)[N], int (&tot)[N], int* sh) {
  const int lane = threadIdx.x % 32, warp = threadIdx.x / 32, nw = blockDim.x / 32;
  int incl[N];
#pragma unroll
  for (int i = 0; i < N; ++i) incl[i] = v[i];
#pragma unroll
  for (int o = 1; o < 32; o <<= 1)
#pragma unroll
    for (int i = 0; i < N; ++i) {
      const int n = __shfl_up_sync(0xffffffffu, incl[i], o);
      if (lane >= o) incl[i] += n;
    }
  if (lane == 31)
#pragma unroll
    for (int i = 0; i < N; ++i) sh[i * 32 + warp] = incl[i];
  __syncthreads();
  if (warp == 0)
#pragma unroll
    for (int i = 0; i < N; ++i) {
      int w = lane < nw ? sh[i * 32 + lane] : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, w, o);
        if (lane >= o) w += n;
      }
      sh[i * 32 + lane] = w;
    }
  __syncthreads();
#pragma unroll
  for (int i = 0; i < N; ++i) {
    excl[i] = (warp > 0 ? sh[i * 32 + warp - 1] : 0) + incl[i] - v[i];
    tot[i] = sh[i * 32 + nw - 1];
  }
  __syncthreads();
}

constexpr int kWlScanInts = 32 * 6;  // shared scratch of build_worklist

// Builds the work list from the experts' offsets; called by all threads of a
// 1024-thread CTA (block-wide scans inside; sh holds kWlScanInts ints).  With
// at most 32 units, warp 0 builds it alone with warp scans (no block barrier).
__device__ void build_worklist(const WlArgs& a, const int32_t* offsets, int* sh) {
  int carry[6] = {0, 0, 0, 0, 0, 0};
  const int units = a.E_r + (a.has_shared ? 1 : 0);
  const bool one_warp = units <= 32;
  if (one_warp && threadIdx.x >= 32) return;
  for (int base = 0; base < units; base += blockDim.x) {
    const int u = base + threadIdx.x;
    const int e = a.has_shared ? u - 1 : u;  // routed expert of this unit; -1: shared
    int n = 0, row0 = 0, shared = 0;
    if (u < units) {
      if (e < 0) {
        n = a.T;
        shared = 1;
      } else {
        row0 = offsets[e];
        n = offsets[e + 1] - row0;
      }
    }
    const bool gemv = n > 0 && n <= a.gemv_max;
    const int n_gemv = gemv ? (n + a.gemv_chunk - 1) / a.gemv_chunk : 0;
    const int n_tc = (!gemv && n > 0) ? (n + a.tc_chunk - 1) / a.tc_chunk : 0;
    const int gi_gu = shared ? a.items_gu_shared : a.items_gu;
    const int ti_gu = shared ? a.tiles_gu_shared : a.tiles_gu;
    const int v[6] = {n_gemv, n_gemv * gi_gu, n_gemv * a.items_dn, n_tc, n_tc * ti_gu,
                      n_tc * a.tiles_dn};
    int pos[6], tot[6];
    if (one_warp) {
      const int lane = threadIdx.x;
#pragma unroll
      for (int i = 0; i < 6; ++i) {
        int incl = v[i];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int nb = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += nb;
        }
        pos[i] = incl - v[i];
        tot[i] = __shfl_sync(0xffffffffu, incl, 31);
      }
    } else {
      block_exclusive_scan_n<6>(v, pos, tot, sh);
    }
#pragma unroll
    for (int i = 0; i < 6; ++i) {
      pos[i] += carry[i];
      carry[i] += tot[i];
    }
    for (int j = 0; j < n_gemv; ++j) {
      const int ti = pos[0] + j;
      if (ti >= a.wl.capacity) {
        raise_status(a.status, kStInternal, MOE_K_WORKLIST);
        break;
      }
      FfnTask tk;
      tk.expert = shared ? -1 : e;
      tk.row0 = row0 + j * a.gemv_chunk;
      tk.nrows = min(a.gemv_chunk, n - j * a.gemv_chunk);
      tk.chunk = 0;
      a.wl.gemv_tasks[ti] = tk;
      a.wl.gemv_start_gu[ti] = pos[1] + j * gi_gu;
      a.wl.gemv_start_dn[ti] = pos[2] + j * a.items_dn;
    }
    for (int j = 0; j < n_tc; ++j) {
      const int ti = pos[3] + j;
      if (ti >= a.wl.capacity) {
        raise_status(a.status, kStInternal, MOE_K_WORKLIST);
        break;
      }
      FfnTask tk;
      tk.expert = shared ? -1 : e;
      tk.row0 = row0 + j * a.tc_chunk;
      tk.nrows = min(a.tc_chunk, n - j * a.tc_chunk);
      tk.chunk = (j << 16) | n_tc;  // chunk index, chunks of this unit (tile interleaving)
      a.wl.tc_tasks[ti] = tk;
      a.wl.tc_start_gu[ti] = pos[4] + j * ti_gu;
      a.wl.tc_start_dn[ti] = pos[5] + j * a.tiles_dn;
      if (a.wl.gu_done) a.wl.gu_done[ti] = 0;
    }
  }
  if (threadIdx.x == 0) {
    if (a.wl.redo_gu) a.wl.redo_gu[0] = 0;
    if (a.wl.redo_dn) a.wl.redo_dn[0] = 0;
    a.wl.counts[kWlSchedGU] = 0;
    a.wl.counts[kWlSchedDN] = 0;
    a.wl.counts[kWlGemvTasks] = min(carry[0], a.wl.capacity);
    a.wl.counts[kWlGemvItemsGU] = carry[0] <= a.wl.capacity ? carry[1] : 0;
    a.wl.counts[kWlGemvItemsDN] = carry[0] <= a.wl.capacity ? carry[2] : 0;
    a.wl.counts[kWlTcTasks] = min(carry[3], a.wl.capacity);
    a.wl.counts[kWlTcTilesGU] = carry[3] <= a.wl.capacity ? carry[4] : 0;
    a.wl.counts[kWlTcTilesDN] = carry[3] <= a.wl.capacity ? carry[5] : 0;
  }
}

__global__ void __launch_bounds__(1024) worklist_kernel(WlArgs a) {
  pdl_enter();
  __shared__ int sh[kWlScanInts];
  build_worklist(a, a.offsets, sh);
}

// Small batches: the whole re-sort in one CTA, and (with build_wl) the work list
// after it, in place of the count / scan / scatter / work-list launches.  An
// [expert][token] bitmap of all T tokens sits in shared memory: popcounts give
// each expert's count and each pick's rank among the earlier tokens of its
// expert, so the order inside an expert is by token, as in the multi-CTA path.
static_assert(kSmallRouteWarps * 32 == 1024, "the one-CTA re-sort routes with all its warps");
__global__ void __launch_bounds__(1024)
    sort_small_kernel(const int32_t* ids, int32_t* counts, int32_t* offsets, int32_t* s2e,
                      int32_t* e2s, int T, int k, int E, WlArgs wla, int build_wl,
                      DevStatus* st, SmallGather g, SmallRoute rt, TopkArgs tk) {
  // bitmap [E][W], offsets [E + 1], then (rt.x set) the router's region
  extern __shared__ __align__(16) uint32_t sm[];
  __shared__ int sh[kWlScanInts];
  const int tid = threadIdx.x;
  const int W = (T + 31) / 32, R = T * k;
  uint32_t* bm = sm;
  int32_t* off = reinterpret_cast<int32_t*>(sm + (size_t)E * W);
  for (int i = tid; i < E * W; i += blockDim.x) bm[i] = 0u;  // shared only: before the wait
  pdl_enter();
  // small layers: route the tokens here (ids and weights written to global
  // memory, visible to the block after the routine's closing barrier)
  if (rt.x)
    route_small_block(rt, tk, reinterpret_cast<unsigned char*>(sm) +
                                  align16(((size_t)E * W + E + 1) * 4));
  __syncthreads();
  for (int r = tid; r < R; r += blockDim.x) {
    const int e = ids[r];
    if ((unsigned)e >= (unsigned)E) {
      raise_status(st, kStBadId, MOE_K_SORT);
      continue;
    }
    const int t = r / k;
    atomicOr(&bm[e * W + t / 32], 1u << (t % 32));
  }
  __syncthreads();
  // counts, and their exclusive scan: by warp 0 alone for at most 32 experts,
  // else 1024 experts per round
  if (E <= 32) {
    if (tid < 32) {
      int c = 0;
      if (tid < E) {
        for (int w = 0; w < W; ++w) c += __popc(bm[tid * W + w]);
        counts[tid] = c;
      }
      int incl = c;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int nb = __shfl_up_sync(0xffffffffu, incl, o);
        if (tid >= o) incl += nb;
      }
      if (tid < E) off[tid] = incl - c;
      if (tid == 31) off[E] = incl;
    }
  } else {
    int carry = 0;
    for (int base = 0; base < E; base += blockDim.x) {
      const int e = base + tid;
      int c = 0;
      if (e < E) {
        for (int w = 0; w < W; ++w) c += __popc(bm[e * W + w]);
        counts[e] = c;
      }
      int tot;
      const int excl = block_exclusive_scan(c, &tot, sh);
      if (e < E) off[e] = carry + excl;
      carry += tot;
    }
    if (tid == 0) off[E] = carry;
  }
  __syncthreads();
  for (int e = tid; e <= E; e += blockDim.x) offsets[e] = off[e];
  for (int r = tid; r < R; r += blockDim.x) {
    const int e = ids[r];
    if ((unsigned)e >= (unsigned)E) {
      e2s[r] = -1;
      continue;
    }
    const int t = r / k;
    int rank = 0;
    for (int w = 0; w < t / 32; ++w) rank += __popc(bm[e * W + w]);
    rank += __popc(bm[e * W + t / 32] & ((1u << (t % 32)) - 1u));
    const int p = off[e] + rank;
    s2e[p] = r;
    e2s[r] = p;
  }
  if (build_wl) {
    __syncthreads();
    build_worklist(wla, off, sh);
  }
  if (g.x_perm) {
    // small layers: the row gather (and the fused combine's accumulator rows)
    // in the same CTA, in place of the gather launch
    __syncthreads();
    const int per_row = g.H / 8;
    for (int idx = tid; idx < R * per_row; idx += blockDim.x) {
      const int r = idx / per_row, i = idx % per_row;
      const int e = ids[r];
      const int p = e2s[r];
      if ((unsigned)e >= (unsigned)g.E_r || p < 0) continue;
      reinterpret_cast<uint4*>(g.x_perm + (size_t)p * g.H)[i] =
          reinterpret_cast<const uint4*>(g.x + (size_t)(r / k) * g.H)[i];
    }
    if (g.acc)
      for (int idx = tid; idx < T * per_row; idx += blockDim.x) {
        const int t = idx / per_row;
        zero_pick_init(ids, g.w, t, k, g.E_r, E, g.x + (size_t)t * g.H, g.acc + (size_t)t * g.H,
                       g.H, idx % per_row, per_row);
      }
  }
}

WlArgs make_wl_args(const Launch& L, const moe_config& c, int T, const int32_t* offsets,
                    const WorkList& wl, int gemv_max_rows, int gemv_chunk, int tc_chunk,
                    int dn_ch) {
  WlArgs a;
  a.offsets = offsets;
  a.wl = wl;
  a.E_r = c.n_routed;
  a.T = T;
  a.has_shared = c.shared_inter > 0;
  a.gemv_max = gemv_max_rows;
  a.gemv_chunk = gemv_chunk;
  a.tc_chunk = tc_chunk;
  // W8A8 streaming items are 128-channel tiles; bf16 ones 8 gate/up pairs or 16
  // down channels
  const int ch_gu = c.wdtype == MOE_W8A8 ? kGemvI8Ch : kGemvChGU;
  const int ch_dn = c.wdtype == MOE_W8A8 ? kGemvI8Ch : kGemvChDN;
  a.items_gu = (c.inter + ch_gu - 1) / ch_gu;
  a.items_gu_shared = (c.shared_inter + ch_gu - 1) / ch_gu;
  a.items_dn = (c.hidden + ch_dn - 1) / ch_dn;
  // W8A8 tensor-core tiles span 256 channels (two-SM tiles), bf16 ones 128
  const int tch = c.wdtype == MOE_W8A8 ? 2 * kTcM : kTcM;
  a.tiles_gu = (c.inter + tch - 1) / tch;
  a.tiles_gu_shared = (c.shared_inter + tch - 1) / tch;
  const int dch = dn_ch > 0 ? dn_ch : tch;
  a.tiles_dn = (c.hidden + dch - 1) / dch;
  a.status = L.status;
  return a;
}

size_t sort_small_smem(int T, int E) {
  return ((size_t)E * ((T + 31) / 32) + E + 1) * 4;
}

}  // namespace

bool sort_small_fits(int T, int E) {
  return T <= kSortSmallMaxT && sort_small_smem(T, E) <= (size_t)kSortSmallSmem;
}

bool route_small_fits(const moe_config& c, int T) {
  const int E = c.n_routed + c.n_zero, H = c.hidden;
  if (T < 1 || E < 1 || H % 8 != 0 || c.top_k > 32 || (long long)T * E * H > kSmallRouteWork ||
      !sort_small_fits(T, E))
    return false;
  // the re-sort's bitmap and the router's region fit one CTA together
  return align16(sort_small_smem(T, E)) + small_route_plan(T, E, H).total <=
         (size_t)kSortSmallSmem;
}

size_t route_small_smem(const moe_config& c, int T) {
  return small_route_plan(T, c.n_routed + c.n_zero, c.hidden).total;
}

void launch_sort_small(const Launch& L, const moe_config& c, int T, const int32_t* ids,
                       int32_t* counts, int32_t* offsets, int32_t* s2e, int32_t* e2s,
                       const WorkList* wl, int gemv_max_rows, int gemv_chunk, int tc_chunk,
                       const SmallGather* gather, const SmallRoute* route, const TopkArgs* tk,
                       int dn_ch) {
  const int E = c.n_routed + c.n_zero;
  WlArgs a{};
  if (wl) a = make_wl_args(L, c, T, offsets, *wl, gemv_max_rows, gemv_chunk, tc_chunk, dn_ch);
  set_smem_attr_once(reinterpret_cast<const void*>(sort_small_kernel), kSortSmallSmem,
                     kAttrSortSmall);
  launch_begin(L, MOE_K_SORT);
  SmallGather g{};
  if (gather) g = *gather;
  SmallRoute rt{};
  TopkArgs tka{};
  size_t smem = sort_small_smem(T, E);
  if (route && tk) {
    rt = *route;
    tka = *tk;
    smem = align16(smem) + route_small_smem(c, T);
  }
  launch_kernel(sort_small_kernel, 1, 1024, smem, L.stream, ids, counts, offsets, s2e, e2s, T,
                c.top_k, E, a, wl ? 1 : 0, L.status, g, rt, tka);
  launch_end(L, MOE_K_SORT);
}

void launch_perm_count(const Launch& L, int T, int k, int E, const int32_t* ids, int32_t* bc) {
  const int nblk = (T + kPermTokens - 1) / kPermTokens;
  launch_begin(L, MOE_K_PERM_COUNT);
  launch_kernel(perm_count_kernel, nblk, kPermThreads, E * sizeof(int32_t), L.stream, ids, bc, T,
                k, E, L.status);
  launch_end(L, MOE_K_PERM_COUNT);
}

void launch_perm_scan(const Launch& L, int T, int E, int32_t* bc, int32_t* counts,
                      int32_t* offsets) {
  const int nblk = (T + kPermTokens - 1) / kPermTokens;
  launch_begin(L, MOE_K_PERM_SCAN);
  launch_kernel(perm_scan_kernel, 1, 1024, 0, L.stream, bc, counts, offsets, nblk, E);
  launch_end(L, MOE_K_PERM_SCAN);
}

void launch_perm_scatter(const Launch& L, int T, int k, int E, const int32_t* ids,
                         const int32_t* bc, int32_t* s2e, int32_t* e2s) {
  const int nblk = (T + kPermTokens - 1) / kPermTokens;
  const size_t smem = (size_t)E * kWords * sizeof(uint32_t);
  set_smem_attr_once(reinterpret_cast<const void*>(perm_scatter_kernel), 200 * 1024,
                     kAttrPermScatter);
  launch_begin(L, MOE_K_PERM_SCATTER);
  launch_kernel(perm_scatter_kernel, nblk, kPermThreads, smem, L.stream, ids, bc, s2e, e2s, T, k,
                E);
  launch_end(L, MOE_K_PERM_SCATTER);
}

void launch_perm_gather(const Launch& L, const moe_config& c, int T, const int32_t* ids,
                        const int32_t* e2s, const void* x, void* x_perm, float* x_perm_scale,
                        const float* w, float* acc) {
  GatherArgs a;
  a.ids = ids;
  a.e2s = e2s;
  a.x = static_cast<const uint16_t*>(x);
  a.x_perm = x_perm;
  a.scale = x_perm_scale;
  a.R = T * c.top_k;
  a.k = c.top_k;
  a.H = c.hidden;
  a.E_r = c.n_routed;
  a.E = c.n_routed + c.n_zero;
  a.w8a8 = c.wdtype == MOE_W8A8;
  a.w = w;
  a.acc = acc;
  a.gather_blocks = (a.R + 7) / 8;
  const int init_blocks = acc ? (int)(((long long)T * (c.hidden / 8) + 255) / 256) : 0;
  launch_begin(L, MOE_K_PERM_GATHER);
  launch_kernel(perm_gather_kernel, a.gather_blocks + init_blocks, 256, 0, L.stream, a);
  launch_end(L, MOE_K_PERM_GATHER);
}

void launch_worklist(const Launch& L, const moe_config& c, int T, const int32_t* offsets,
                     const WorkList& wl, int gemv_max_rows, int gemv_chunk, int tc_chunk,
                     int dn_ch) {
  const WlArgs a =
      make_wl_args(L, c, T, offsets, wl, gemv_max_rows, gemv_chunk, tc_chunk, dn_ch);
  launch_begin(L, MOE_K_WORKLIST);
  launch_kernel(worklist_kernel, 1, 1024, 0, L.stream, a);
  launch_end(L, MOE_K_WORKLIST);
}

}  // namespace moe
