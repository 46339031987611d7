// C ABI of the layer: argument checks, workspace layout, launch sequencing and
// diagnostics.  No device memory is allocated here; every buffer comes from the
// caller (tensors) or from the caller's workspace.
#include <math.h>

#include <atomic>
#include <climits>
#include <cstdlib>
#include <mutex>
#include <vector>

#include "common.cuh"
#include "internal.h"
#include "small_ffn.h"

namespace moe {

namespace {

constexpr int kMaxExperts = 4096;
constexpr int kMaxTopK = 32;
constexpr int kMaxGroups = 64;
constexpr int kMaxDevices = 64;

// ------------------------------------------------------------ bookkeeping --
std::atomic<long long> g_launches[MOE_K_COUNT];
std::atomic<int> g_attr_done[kAttrSlots][kMaxDevices];
std::atomic<int> g_sm_count[kMaxDevices];

struct TimedLaunch {
  int kind;
  cudaEvent_t a, b;
};
std::mutex g_tmu;
std::atomic<bool> g_timing{false};
std::vector<TimedLaunch> g_records;
std::vector<cudaEvent_t> g_event_pool;
thread_local cudaEvent_t t_open_event = nullptr;
thread_local cudaError_t t_launch_error = cudaSuccess;

cudaEvent_t take_event() {
  std::lock_guard<std::mutex> lk(g_tmu);
  if (!g_event_pool.empty()) {
    cudaEvent_t e = g_event_pool.back();
    g_event_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}

int current_device() {
  int d = 0;
  if (cudaGetDevice(&d) != cudaSuccess) return -1;
  return d;
}

int sm_count(int dev) {
  if (dev < 0 || dev >= kMaxDevices) return 148;
  int n = g_sm_count[dev].load();
  if (n <= 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 148;
    g_sm_count[dev].store(n);
  }
  return n;
}

size_t align256(size_t v) { return (v + 255) & ~(size_t)255; }

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// ---------------------------------------------------------- config checks --
moe_status check_cfg(const moe_config* c, int32_t T) {
  if (!c || T < 0) return MOE_ERR_INVALID_ARG;
  if (c->hidden < 8 || c->hidden % 8) return MOE_ERR_INVALID_ARG;
  if (c->n_routed < 0 || c->n_zero < 0) return MOE_ERR_INVALID_ARG;
  const int E = c->n_routed + c->n_zero;
  if (E < 1) return MOE_ERR_INVALID_ARG;
  if (E > kMaxExperts) return MOE_ERR_UNSUPPORTED;
  if (c->n_routed > 0 && (c->inter < 8 || c->inter % 8)) return MOE_ERR_INVALID_ARG;
  if (c->top_k < 1 || c->top_k > E) return MOE_ERR_INVALID_ARG;
  if (c->top_k > kMaxTopK) return MOE_ERR_UNSUPPORTED;
  if (c->n_group < 1 || E % c->n_group) return MOE_ERR_INVALID_ARG;
  if (c->n_group > kMaxGroups) return MOE_ERR_UNSUPPORTED;
  if (c->n_group > 1) {
    const int G = E / c->n_group;
    if (c->per_group_k < 0) return MOE_ERR_INVALID_ARG;
    if (c->per_group_k > 0) {
      if (c->per_group_k > G || c->per_group_k * c->n_group != c->top_k) return MOE_ERR_INVALID_ARG;
    } else {
      if (c->topk_group < 1 || c->topk_group > c->n_group) return MOE_ERR_INVALID_ARG;
      if (c->top_k > c->topk_group * G) return MOE_ERR_INVALID_ARG;
    }
  }
  if (c->score != MOE_SCORE_SOFTMAX && c->score != MOE_SCORE_SIGMOID) return MOE_ERR_INVALID_ARG;
  if (c->renormalize != 0 && c->renormalize != 1) return MOE_ERR_INVALID_ARG;
  if (!isfinite(c->routed_scale)) return MOE_ERR_INVALID_ARG;
  if (c->bias_mode < MOE_BIAS_NONE || c->bias_mode > MOE_BIAS_SELECT) return MOE_ERR_INVALID_ARG;
  if (c->shared_inter < 0 || c->shared_inter % 8) return MOE_ERR_INVALID_ARG;
  if (c->wdtype != MOE_W_BF16 && c->wdtype != MOE_W8A8) return MOE_ERR_INVALID_ARG;
  if (c->wdtype == MOE_W8A8) {
    // int8 rows must be whole 16-byte vectors; per-row sums of squared codes must
    // fit int32 (K <= 131071); no shared expert in this mode.
    if (c->hidden % 16 || (c->n_routed > 0 && c->inter % 16)) return MOE_ERR_INVALID_ARG;
    if (c->hidden > 131071 || c->inter > 131071) return MOE_ERR_UNSUPPORTED;
    // the shared expert is int8 like the routed ones: its K (I_s) in 16-byte rows
    if (c->shared_inter % 16 || c->shared_inter > 131071) return MOE_ERR_INVALID_ARG;
    if (c->shared_inter > 0 && c->n_routed == 0) return MOE_ERR_UNSUPPORTED;
  }
  if (c->out_fp32 != 0 && c->out_fp32 != 1) return MOE_ERR_INVALID_ARG;
  if (c->combine < MOE_COMBINE_DEFAULT || c->combine > MOE_COMBINE_FUSED)
    return MOE_ERR_INVALID_ARG;
  if (c->ffn_launch < MOE_FFN_LAUNCH_DEFAULT || c->ffn_launch > MOE_FFN_LAUNCH_ONE_WIDE)
    return MOE_ERR_INVALID_ARG;
  // work-list chunk indices are 16-bit: at most 65535 chunks of 128 rows per unit
  if ((long long)T * c->top_k > (1LL << 30) || T > 65535 * kTcMaxN) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

// ------------------------------------------------------ tile parameters --
// The grouped FFN's tiling choices come from a table measured offline on GB300
// (tuning/tile_table.json, compiled in): the history-based tiling choice of the
// Pangu Pro MoE disclosure, section SwiftGMM.  It is keyed by weight type, H, I
// and the load bucket of the expected picks per expert, T * k / (E_r + E_z);
// the entry of the same weight type nearest in bucket, then in H * I, applies.
struct TileEntry {
  int wdtype, hidden, inter, bucket, gemv_max, one_launch, dn_wide;
};
#include "tile_table.inc"

int load_bucket(const moe_config& c, int T) {
  const double m = (double)T * c.top_k / (double)(c.n_routed + c.n_zero);
  int b = 0;
  for (int v : kTileBuckets) {
    if (m < v) return b;
    ++b;
  }
  return b;
}

const TileEntry* tile_entry(const moe_config& c, int T) {
  const int b = load_bucket(c, T);
  const double hi = (double)c.hidden * (c.inter > 0 ? c.inter : 1);
  const TileEntry* best = nullptr;
  double best_d = 0.0;
  for (const TileEntry& e : kTileTable) {
    if (e.wdtype != c.wdtype) continue;
    const double d = 1000.0 * abs(e.bucket - b) + fabs(log2(hi / ((double)e.hidden * e.inter)));
    if (!best || d < best_d) {
      best = &e;
      best_d = d;
    }
  }
  return best;
}

// Experts (and the shared expert) with at most this many rows stream through
// the GEMV path; the others run on tensor-core tiles.  gemv_max_rows > 0 sets
// the switch point, < 0 turns the GEMV path off, 0 takes the table's.
int effective_gemv_max(const moe_config& c, int T) {
  if (c.gemv_max_rows > 0) return c.gemv_max_rows;
  if (c.gemv_max_rows < 0) return 0;
  const TileEntry* e = tile_entry(c, T);
  if (e) return e->gemv_max;
  return c.wdtype == MOE_W8A8 ? kDefaultGemvMaxRowsW8 : kDefaultGemvMaxRows;
}
// Whether moe_layer_forward adds the expert outputs into the tokens' fp32
// accumulators in the down projection's epilogue (the library default) instead
// of writing per-pick rows for the ordered combine kernel.  A W8A8 layer without
// FFN experts has no quantising gather to start the accumulators, so it takes
// the ordered combine.
bool fused_combine(const moe_config& c) {
  if (c.combine == MOE_COMBINE_ORDERED) return false;
  if (c.wdtype == MOE_W8A8 && c.n_routed == 0) return false;
  return true;
}

// Whether the bf16 grouped FFN runs its tensor-core gate/up and down passes as
// one persistent launch (down tiles wait for their task's gate/up tiles, which
// fills the gate/up pass's last partial wave) instead of two: cfg.ffn_launch,
// or the table's choice when it is MOE_FFN_LAUNCH_DEFAULT.
bool ffn_one_launch(const moe_config& c, int T) {
  if (c.wdtype != MOE_W_BF16) return false;
  if (c.ffn_launch == MOE_FFN_LAUNCH_TWO) return false;
  if (c.ffn_launch == MOE_FFN_LAUNCH_ONE || c.ffn_launch == MOE_FFN_LAUNCH_ONE_WIDE) return true;
  const TileEntry* e = tile_entry(c, T);
  return e ? e->one_launch != 0 : true;
}

// Whether the one-launch FFN's down tiles span 2 x kTcM output channels: two
// weight boxes and two accumulators per K step share one activation box, so a
// task's h rows are read half as often (measured on GB300: a gain with tens of
// rows per expert, a small loss with a few): cfg.ffn_launch, or the table's
// choice when it is MOE_FFN_LAUNCH_DEFAULT.
bool ffn_dn_wide(const moe_config& c, int T) {
  if (!ffn_one_launch(c, T)) return false;
  if (c.ffn_launch != MOE_FFN_LAUNCH_DEFAULT) return c.ffn_launch == MOE_FFN_LAUNCH_ONE_WIDE;
  const TileEntry* e = tile_entry(c, T);
  return e && e->dn_wide != 0;
}

// Whether the bf16 grouped FFN runs as the small-layer kernel (library defaults
// only: an explicit GEMV switch point or launch form keeps the other paths).
bool small_ffn_chosen(const moe_config& c, int T) {
  return c.gemv_max_rows == 0 && c.ffn_launch == MOE_FFN_LAUNCH_DEFAULT && c.n_routed > 0 &&
         small_ffn_fits(c, T);
}

// The GEMV launches are skipped when no unit can take that path.
bool gemv_possible(int gemv_max) { return gemv_max > 0; }

// Rows per GEMV task: the smallest of 1, 2, 4, 8 that holds gemv_max rows (8 when
// gemv_max is larger: such units are split into 8-row tasks).
int gemv_chunk(int gemv_max) {
  int c = 1;
  while (c < gemv_max && c < kGemvMaxRows) c *= 2;
  return c;
}

// --------------------------------------------------------------- workspace --
struct Layout {
  size_t status, partial, logits, ids, w, bc, counts, offsets, s2e, e2s;
  // tensor-core router only: split weights, its work list
  size_t rsplit, rtasks, rstart, rcounts;
  bool tc_router;
  size_t wl_gemv_tasks, wl_gemv_gu, wl_gemv_dn, wl_tc_tasks, wl_tc_gu, wl_tc_dn, wl_counts;
  size_t wl_gu_done;  // single-launch FFN: per task count of stored gate/up tiles
  size_t x_perm, x_scale, h, y, h_s, y_s;
  size_t acc;  // fused combine with bf16 output: the tokens' fp32 accumulators
  // W8A8 only: integer-valued fp16 copies of the codes, row norms, fp32 h and
  // its codes/scales, and the guard-failure lists of the two passes
  size_t x16, xn2, h32, hq16, hsc, hn2, redo_gu, redo_dn;
  size_t x8, h8;  // int8 codes for the W8A8 streaming path (only when it may run)
  // W8A8 shared expert: the tokens' codes (one row per token), its fp32 h and
  // codes, and a work list and guard-failure lists of its own
  size_t xs16, xsn2, xss, hs32, hsq16, hssc, hsn2;
  size_t swl_tasks, swl_gu, swl_dn, swl_counts, sredo_gu, sredo_dn;
  int swl_cap, sredo_cap;
  int redo_cap;
  size_t total;
  int splits, nblk, wl_cap;
};

Layout make_layout(const moe_config& c, int T) {
  Layout L{};
  const size_t E = (size_t)c.n_routed + c.n_zero;
  const size_t R = (size_t)T * c.top_k;
  const size_t H = c.hidden, I = c.inter, Is = c.shared_inter;
  L.splits = router_splits_default(c, T);
  L.nblk = (T + kPermTokens - 1) / kPermTokens;
  L.wl_cap = c.n_routed + 4 + (int)(R + T);  // one-row tasks at worst
  const size_t xb = c.wdtype == MOE_W8A8 ? 1 : 2;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off = align256(off + bytes);
    return at;
  };
  L.status = take(256 + kRouterCounterBytes);  // status word, then router tile counters
  L.tc_router = router_on_tensor_cores(c, T);
  if (L.tc_router) {
    const size_t nt = ((size_t)T + kTcMaxN - 1) / kTcMaxN;
    L.splits = 1;
    L.rsplit = take(E * 3 * H * 2);
    L.rtasks = take(nt * sizeof(FfnTask));
    L.rstart = take(nt * 4);
    L.rcounts = take(kWlCount * 4);
  }
  L.partial = take(L.splits > 1 ? (size_t)L.splits * T * E * 4 : 0);
  L.logits = take((size_t)T * E * 4);
  L.ids = take(R * 4);
  L.w = take(R * 4);
  L.bc = take((size_t)L.nblk * E * 4);
  L.counts = take(E * 4);
  L.offsets = take((E + 1) * 4);
  L.s2e = take(R * 4);
  L.e2s = take(R * 4);
  L.wl_gemv_tasks = take((size_t)L.wl_cap * sizeof(FfnTask));
  L.wl_gemv_gu = take((size_t)L.wl_cap * 4);
  L.wl_gemv_dn = take((size_t)L.wl_cap * 4);
  L.wl_tc_tasks = take((size_t)L.wl_cap * sizeof(FfnTask));
  L.wl_tc_gu = take((size_t)L.wl_cap * 4);
  L.wl_tc_dn = take((size_t)L.wl_cap * 4);
  L.wl_counts = take(kWlCount * 4);
  L.wl_gu_done = take((size_t)L.wl_cap * 4);
  // W8A8 layers quantise straight into x16 and keep h in fp32 (h32), so the
  // int8 x_perm and the bf16 h are bf16-path buffers only
  const bool w8 = c.wdtype == MOE_W8A8;
  L.x_perm = take(w8 ? 0 : R * H * xb);
  L.x_scale = take(R * 4);
  L.h = take(w8 ? 0 : R * I * 2);
  // the ordered combine reads per-pick rows (and the shared expert's output);
  // the fused one adds into per-token accumulators (the caller's fp32 output, or
  // this buffer ahead of the bf16 rounding)
  const bool fused = fused_combine(c);
  L.y = take(fused ? 0 : R * H * 4);
  L.h_s = take((size_t)T * Is * 2);
  L.y_s = take(Is > 0 && !fused ? (size_t)T * H * 4 : 0);
  L.acc = take(fused && !c.out_fp32 ? (size_t)T * H * 4 : 0);
  if (c.wdtype == MOE_W8A8) {
    const size_t tc_tasks = c.n_routed + 4 + R / kTcMaxN;
    // one entry per CTA half of each two-SM tile of 256 channels
    const size_t tiles = 2 * ((std::max(I, H) + 2 * kTcM - 1) / (2 * kTcM));
    L.redo_cap = (int)(tc_tasks * tiles);
    L.x16 = take(R * H * 2);
    L.xn2 = take(R * 4);
    L.h32 = take(R * I * 4);
    L.hq16 = take(R * I * 2);
    L.hsc = take(R * 4);
    L.hn2 = take(R * 4);
    L.redo_gu = take((size_t)(1 + L.redo_cap) * 4);
    L.redo_dn = take((size_t)(1 + L.redo_cap) * 4);
    const bool gemv = gemv_possible(effective_gemv_max(c, T));
    L.x8 = take(gemv ? R * H : 0);
    L.h8 = take(gemv ? R * I : 0);
    if (Is > 0) {
      L.swl_cap = (int)(4 + ((size_t)T + kW8MaxN - 1) / kW8MaxN);
      L.sredo_cap = L.swl_cap * 2 * (int)((std::max(Is, H) + 2 * kTcM - 1) / (2 * kTcM));
      L.xs16 = take((size_t)T * H * 2);
      L.xsn2 = take((size_t)T * 4);
      L.xss = take((size_t)T * 4);
      L.hs32 = take((size_t)T * Is * 4);
      L.hsq16 = take((size_t)T * Is * 2);
      L.hssc = take((size_t)T * 4);
      L.hsn2 = take((size_t)T * 4);
      L.swl_tasks = take((size_t)L.swl_cap * sizeof(FfnTask));
      L.swl_gu = take((size_t)L.swl_cap * 4);
      L.swl_dn = take((size_t)L.swl_cap * 4);
      L.swl_counts = take(kWlCount * 4);
      L.sredo_gu = take((size_t)(1 + L.sredo_cap) * 4);
      L.sredo_dn = take((size_t)(1 + L.sredo_cap) * 4);
    }
  }
  L.total = off;
  return L;
}

template <class P>
P* at(void* ws, size_t off) {
  return reinterpret_cast<P*>(static_cast<char*>(ws) + off);
}

WorkList worklist_view(void* ws, const Layout& L) {
  WorkList wl;
  wl.gemv_tasks = at<FfnTask>(ws, L.wl_gemv_tasks);
  wl.gemv_start_gu = at<int32_t>(ws, L.wl_gemv_gu);
  wl.gemv_start_dn = at<int32_t>(ws, L.wl_gemv_dn);
  wl.tc_tasks = at<FfnTask>(ws, L.wl_tc_tasks);
  wl.tc_start_gu = at<int32_t>(ws, L.wl_tc_gu);
  wl.tc_start_dn = at<int32_t>(ws, L.wl_tc_dn);
  wl.counts = at<int32_t>(ws, L.wl_counts);
  wl.capacity = L.wl_cap;
  wl.redo_gu = L.redo_cap > 0 ? at<int32_t>(ws, L.redo_gu) : nullptr;
  wl.redo_dn = L.redo_cap > 0 ? at<int32_t>(ws, L.redo_dn) : nullptr;
  wl.gu_done = at<int32_t>(ws, L.wl_gu_done);
  return wl;
}

moe_status check_ws(const moe_config& c, int T, const void* ws, size_t ws_bytes, Layout* L) {
  *L = make_layout(c, T);
  if (!ws) return MOE_ERR_INVALID_ARG;
  if (!aligned(ws, 256)) return MOE_ERR_ALIGNMENT;
  if (ws_bytes < L->total) return MOE_ERR_WORKSPACE_TOO_SMALL;
  return MOE_OK;
}

moe_status finish() {
  const cudaError_t e = t_launch_error;
  t_launch_error = cudaSuccess;
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

Launch make_launch(moe_stream_t stream, void* ws, const Layout& L) {
  Launch ln;
  ln.stream = reinterpret_cast<cudaStream_t>(stream);
  ln.num_sms = sm_count(current_device());
  ln.status = at<DevStatus>(ws, L.status);
  return ln;
}

// ---------------------------------------------------------------- stages --
moe_status run_route(const Launch& ln, const moe_config& c, int T, const Layout& L, void* ws,
                     const void* x, const float* w_router, const float* bias, int32_t* ids,
                     float* w) {
  float* logits = at<float>(ws, L.logits);
  if (L.tc_router) {
    uint16_t* split = at<uint16_t>(ws, L.rsplit);
    launch_router_split(ln, w_router, c.n_routed + c.n_zero, c.hidden, split);
    if (!launch_tc_router(ln, c, T, x, split, at<FfnTask>(ws, L.rtasks), at<int32_t>(ws, L.rstart),
                          at<int32_t>(ws, L.rcounts), logits))
      return MOE_ERR_CUDA;
    launch_topk_only(ln, c, T, logits, bias, ids, w);
  } else {
    float* partial = at<float>(ws, L.partial);
    int* counters = at<int>(ws, L.status + 256);
    launch_route(ln, c, T, x, w_router, bias, partial, L.splits, logits, counters, ids, w);
  }
  return MOE_OK;
}

// How the grouped FFN's work list is cut: the config it sees (shared expert
// dropped when its weights are absent or in W8A8), the GEMV switch point and
// chunk, and the tensor-core chunk.
struct WlPlan {
  moe_config cw;
  int gemv_max, chunk, tc_chunk, dn_ch;
};
WlPlan wl_plan(const moe_config& c, int T, bool shared_weights) {
  WlPlan p;
  p.cw = c;
  if (!shared_weights || c.wdtype == MOE_W8A8) p.cw.shared_inter = 0;
  p.gemv_max = effective_gemv_max(c, T);
  p.chunk = gemv_chunk(p.gemv_max);
  p.tc_chunk = c.wdtype == MOE_W8A8 ? kW8MaxN : kTcMaxN;
  p.dn_ch = ffn_dn_wide(c, T) ? 2 * kTcM : 0;
  return p;
}

// Re-sort (and, for a plan, the work list).  Small batches take the one-CTA
// sort; returns whether the work list was built.
bool run_permute(const Launch& ln, const moe_config& c, int T, const Layout& L, void* ws,
                 const int32_t* ids, const void* x, int32_t* counts, int32_t* offsets,
                 int32_t* s2e, int32_t* e2s, void* x_perm, float* x_scale, const WlPlan* plan,
                 const float* w = nullptr, float* acc = nullptr,
                 const SmallRoute* route = nullptr, const TopkArgs* tk = nullptr) {
  const int E = c.n_routed + c.n_zero;
  bool built = false;
  if (sort_small_fits(T, E)) {
    const WorkList wl = worklist_view(ws, L);
    // small bf16 layers: the sort CTA also gathers the rows
    const size_t gather_bytes = (size_t)T * c.top_k * c.hidden * 2 + (size_t)T * c.hidden * 4;
    SmallGather g{};
    const bool small = x_perm && c.wdtype == MOE_W_BF16 && gather_bytes <= kSmallGatherBytes &&
                       folds_enabled();
    if (small) {
      g.x = static_cast<const uint16_t*>(x);
      g.x_perm = static_cast<uint16_t*>(x_perm);
      g.w = w;
      g.acc = acc;
      g.H = c.hidden;
      g.E_r = c.n_routed;
    }
    launch_sort_small(ln, plan ? plan->cw : c, T, ids, counts, offsets, s2e, e2s,
                      plan ? &wl : nullptr, plan ? plan->gemv_max : 0, plan ? plan->chunk : 1,
                      plan ? plan->tc_chunk : kTcMaxN, small ? &g : nullptr, route, tk,
                      plan ? plan->dn_ch : 0);
    built = plan != nullptr;
    if (small) return built;
  } else {
    int32_t* bc = at<int32_t>(ws, L.bc);
    launch_perm_count(ln, T, c.top_k, E, ids, bc);
    launch_perm_scan(ln, T, E, bc, counts, offsets);
    launch_perm_scatter(ln, T, c.top_k, E, ids, bc, s2e, e2s);
  }
  if (x_perm) launch_perm_gather(ln, c, T, ids, e2s, x, x_perm, x_scale, w, acc);
  return built;
}

// Grouped FFN over the sorted rows plus (optionally) the shared expert.
moe_status run_ffn(const Launch& ln, const moe_config& c, int T, const Layout& L, void* ws,
                   const int32_t* offsets, const void* x_perm, const void* w_gate,
                   const void* w_up, const void* w_down, float* y_perm, const void* x,
                   const void* sg, const void* su, const void* sd, float* y_shared,
                   bool wl_built, const ScatterAdd& sc = ScatterAdd{},
                   const SmallFinalize& fin = SmallFinalize{}) {
  const WorkList wl = worklist_view(ws, L);
  const bool shared = c.shared_inter > 0 && sg != nullptr;
  if (small_ffn_chosen(c, T) && !shared) {
    // the smallest layers: one CTA per expert, both projections in one launch
    SmallFfnArgs s{};
    s.x_perm = static_cast<const uint16_t*>(x_perm);
    s.offsets = offsets;
    s.w_gate = static_cast<const uint16_t*>(w_gate);
    s.w_up = static_cast<const uint16_t*>(w_up);
    s.w_down = static_cast<const uint16_t*>(w_down);
    s.sc = sc;
    s.out_y = y_perm;
    s.fin = fin;
    s.H = c.hidden;
    s.I = c.inter;
    s.E_r = c.n_routed;
    s.R = (int64_t)T * c.top_k;
    return launch_small_ffn(ln, s) ? MOE_OK : MOE_ERR_CUDA;
  }
  const WlPlan plan = wl_plan(c, T, shared);
  const int gemv_max = plan.gemv_max;
  const int chunk = plan.chunk;
  if (!wl_built)
    launch_worklist(ln, plan.cw, T, offsets, wl, gemv_max, chunk, plan.tc_chunk, plan.dn_ch);
  uint16_t* h = at<uint16_t>(ws, L.h);
  uint16_t* h_s = at<uint16_t>(ws, L.h_s);

  GemvPass gu{};
  gu.tasks = wl.gemv_tasks;
  gu.item_start = wl.gemv_start_gu;
  gu.counts = wl.counts;
  gu.task_slot = kWlGemvTasks;
  gu.item_slot = kWlGemvItemsGU;
  gu.w0 = static_cast<const uint16_t*>(w_gate);
  gu.w1 = static_cast<const uint16_t*>(w_up);
  gu.act = static_cast<const uint16_t*>(x_perm);
  gu.out_h = h;
  gu.sw0 = static_cast<const uint16_t*>(sg);
  gu.sw1 = static_cast<const uint16_t*>(su);
  gu.sact = static_cast<const uint16_t*>(x);
  gu.sout_h = h_s;
  gu.K = gu.Ks = c.hidden;
  gu.N = c.inter;
  gu.Ns = c.shared_inter;
  gu.max_rows = chunk;
  if (gemv_possible(gemv_max)) launch_gemv_gate_up(ln, gu);

  const int64_t R = (int64_t)T * c.top_k;
  TcPass tg{};
  tg.tasks = wl.tc_tasks;
  tg.tile_start = wl.tc_start_gu;
  tg.counts = wl.counts;
  tg.task_slot = kWlTcTasks;
  tg.tile_slot = kWlTcTilesGU;
  tg.sched_slot = kWlSchedGU;
  tg.w0 = w_gate;
  tg.w1 = w_up;
  tg.n_experts = c.n_routed;
  tg.act = x_perm;
  tg.act_rows = R;
  tg.out_h = h;
  tg.sw0 = shared ? sg : nullptr;
  tg.sw1 = shared ? su : nullptr;
  tg.sact = x;
  tg.sact_rows = T;
  tg.sout_h = h_s;
  tg.K = tg.Ks = c.hidden;
  tg.N = c.inter;
  tg.Ns = c.shared_inter;
  tg.task_cap = wl.capacity;
  const bool one_launch = ffn_one_launch(c, T);
  if (c.n_routed > 0 && !one_launch && !launch_tc_gate_up(ln, tg)) return MOE_ERR_CUDA;

  GemvPass dn{};
  dn.tasks = wl.gemv_tasks;
  dn.item_start = wl.gemv_start_dn;
  dn.counts = wl.counts;
  dn.task_slot = kWlGemvTasks;
  dn.item_slot = kWlGemvItemsDN;
  dn.w0 = static_cast<const uint16_t*>(w_down);
  dn.act = h;
  dn.out_y = y_perm;
  dn.sw0 = static_cast<const uint16_t*>(sd);
  dn.sact = h_s;
  dn.sout_y = y_shared;
  dn.K = c.inter;
  dn.Ks = c.shared_inter;
  dn.N = dn.Ns = c.hidden;
  dn.max_rows = chunk;
  dn.sc = sc;
  if (gemv_possible(gemv_max)) launch_gemv_down(ln, dn);

  TcPass td{};
  td.tasks = wl.tc_tasks;
  td.tile_start = wl.tc_start_dn;
  td.counts = wl.counts;
  td.task_slot = kWlTcTasks;
  td.tile_slot = kWlTcTilesDN;
  td.sched_slot = kWlSchedDN;
  td.w0 = w_down;
  td.n_experts = c.n_routed;
  td.act = h;
  td.act_rows = R;
  td.out_y = y_perm;
  td.sw0 = shared ? sd : nullptr;
  td.sact = h_s;
  td.sact_rows = T;
  td.sout_y = y_shared;
  td.K = c.inter;
  td.Ks = c.shared_inter;
  td.N = td.Ns = c.hidden;
  td.sc = sc;
  td.fin = fin;
  td.dn_wide = plan.dn_ch > 0;
  td.task_cap = wl.capacity;
  if (c.n_routed > 0) {
    const bool ok = one_launch ? launch_tc_ffn(ln, tg, td, wl.gu_done) : launch_tc_down(ln, td);
    if (!ok) return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

// W8A8 grouped FFN over the sorted rows (int8 codes + per-row scales).  With
// x_perm == nullptr the codes are already in the workspace's x16 rows (and x8,
// when the streaming path may run), with their norms and scales, as the layer
// path's quantising gather leaves them.  Experts with at most gemv_max rows
// stream through the dp4a GEMV, the others run on tensor-core tiles.
moe_status run_ffn_w8a8(const Launch& ln, const moe_config& c, int T, const Layout& L, void* ws,
                        const int32_t* offsets, const void* x_perm, const float* x_scale,
                        const void* w_gate, const void* w_up, const void* w_down,
                        const float* s_gate, const float* s_up, const float* s_down,
                        float* y_perm, bool wl_built, const ScatterAdd& sc = ScatterAdd{}) {
  const WorkList wl = worklist_view(ws, L);
  const WlPlan plan = wl_plan(c, T, false);
  const int gemv_max = plan.gemv_max;
  const bool gemv = gemv_possible(gemv_max);
  if (!wl_built)
    launch_worklist(ln, plan.cw, T, offsets, wl, gemv_max, plan.chunk, plan.tc_chunk);
  const int64_t R = (int64_t)T * c.top_k;
  const int32_t* n_real = offsets + c.n_routed;   // rows that belong to FFN experts
  uint16_t* x16 = at<uint16_t>(ws, L.x16);
  int32_t* xn2 = at<int32_t>(ws, L.xn2);
  float* h32 = at<float>(ws, L.h32);
  uint16_t* hq16 = at<uint16_t>(ws, L.hq16);
  float* hsc = at<float>(ws, L.hsc);
  int32_t* hn2 = at<int32_t>(ws, L.hn2);
  if (x_perm)
    launch_i8_rows_to_f16(ln, static_cast<const int8_t*>(x_perm), x16, xn2, (int)R, c.hidden,
                          n_real);
  const int8_t* x8 = x_perm ? static_cast<const int8_t*>(x_perm) : at<int8_t>(ws, L.x8);
  int8_t* h8 = gemv ? at<int8_t>(ws, L.h8) : nullptr;

  GemvI8Pass vg{};
  vg.tasks = wl.gemv_tasks;
  vg.item_start = wl.gemv_start_gu;
  vg.counts = wl.counts;
  vg.task_slot = kWlGemvTasks;
  vg.item_slot = kWlGemvItemsGU;
  vg.w0 = static_cast<const int8_t*>(w_gate);
  vg.w1 = static_cast<const int8_t*>(w_up);
  vg.n_experts = c.n_routed;
  vg.s0 = s_gate;
  vg.s1 = s_up;
  vg.act = x8;
  vg.act_rows = R;
  vg.row_scale = x_scale;
  vg.out_f32 = at<float>(ws, L.h32);
  vg.K = c.hidden;
  vg.N = c.inter;
  if (gemv && !launch_gemv_i8_gate_up(ln, vg)) return MOE_ERR_CUDA;

  W8Pass g{};
  g.mode = kW8GateUp;
  g.tasks = wl.tc_tasks;
  g.tile_start = wl.tc_start_gu;
  g.counts = wl.counts;
  g.task_slot = kWlTcTasks;
  g.tile_slot = kWlTcTilesGU;
  g.sched_slot = kWlSchedGU;
  g.w0 = w_gate;
  g.w1 = w_up;
  g.n_experts = c.n_routed;
  g.s0 = s_gate;
  g.s1 = s_up;
  g.act = x16;
  g.act_rows = R;
  g.row_norm2 = xn2;
  g.row_scale = x_scale;
  g.out_f32 = h32;
  g.redo = wl.redo_gu;
  g.redo_cap = L.redo_cap;
  g.K = c.hidden;
  g.N = c.inter;
  if (!launch_w8a8(ln, g)) return MOE_ERR_CUDA;

  launch_quant_rows(ln, h32, hq16, h8, hsc, hn2, (int)R, c.inter, offsets, c.n_routed, gemv_max);

  GemvI8Pass vd = vg;
  vd.item_start = wl.gemv_start_dn;
  vd.item_slot = kWlGemvItemsDN;
  vd.w0 = static_cast<const int8_t*>(w_down);
  vd.w1 = nullptr;
  vd.s0 = s_down;
  vd.s1 = nullptr;
  vd.act = h8;
  vd.row_scale = hsc;
  vd.out_f32 = y_perm;
  vd.K = c.inter;
  vd.N = c.hidden;
  vd.sc = sc;
  if (gemv && !launch_gemv_i8_down(ln, vd)) return MOE_ERR_CUDA;

  W8Pass d = g;
  d.mode = kW8Down;
  d.tile_start = wl.tc_start_dn;
  d.tile_slot = kWlTcTilesDN;
  d.sched_slot = kWlSchedDN;
  d.w0 = w_down;
  d.w1 = nullptr;
  d.s0 = s_down;
  d.s1 = nullptr;
  d.act = hq16;
  d.row_norm2 = hn2;
  d.row_scale = hsc;
  d.out_f32 = y_perm;
  d.redo = wl.redo_dn;
  d.K = c.inter;
  d.N = c.hidden;
  d.sc = sc;
  if (!launch_w8a8(ln, d)) return MOE_ERR_CUDA;
  return MOE_OK;
}

// The W8A8 shared expert: a one-expert grouped FFN over every token, on the
// tokens' own codes (written by the quantising gather), with its weights after
// the routed experts' scales in s_gate / s_up / s_down.  Its outputs add into
// the tokens' accumulators at weight 1 (fused combine) or fill y_shared.
moe_status run_shared_w8a8(const Launch& ln, const moe_config& c, int T, const Layout& L,
                           void* ws, const void* sg, const void* su, const void* sd,
                           const float* s_gate, const float* s_up, const float* s_down,
                           float* y_shared, const ScatterAdd& sc) {
  const int Is = c.shared_inter;
  WorkList wl{};
  wl.gemv_tasks = at<FfnTask>(ws, L.swl_tasks);  // no streaming tasks: shares the array
  wl.gemv_start_gu = at<int32_t>(ws, L.swl_gu);
  wl.gemv_start_dn = at<int32_t>(ws, L.swl_dn);
  wl.tc_tasks = at<FfnTask>(ws, L.swl_tasks);
  wl.tc_start_gu = at<int32_t>(ws, L.swl_gu);
  wl.tc_start_dn = at<int32_t>(ws, L.swl_dn);
  wl.counts = at<int32_t>(ws, L.swl_counts);
  wl.capacity = L.swl_cap;
  wl.redo_gu = at<int32_t>(ws, L.sredo_gu);
  wl.redo_dn = at<int32_t>(ws, L.sredo_dn);
  wl.gu_done = nullptr;
  // one unit: the shared expert over all T tokens, in 256-row two-SM tiles
  moe_config cs = c;
  cs.n_routed = 0;
  cs.n_zero = 1;
  launch_worklist(ln, cs, T, nullptr, wl, 0, 1, kW8MaxN);

  W8Pass g{};
  g.mode = kW8GateUp;
  g.tasks = wl.tc_tasks;
  g.tile_start = wl.tc_start_gu;
  g.counts = wl.counts;
  g.task_slot = kWlTcTasks;
  g.tile_slot = kWlTcTilesGU;
  g.sched_slot = kWlSchedGU;
  g.w0 = sg;
  g.w1 = su;
  g.n_experts = 1;
  g.s0 = s_gate + (size_t)c.n_routed * c.inter;
  g.s1 = s_up + (size_t)c.n_routed * c.inter;
  g.act = at<uint16_t>(ws, L.xs16);
  g.act_rows = T;
  g.row_norm2 = at<int32_t>(ws, L.xsn2);
  g.row_scale = at<float>(ws, L.xss);
  g.out_f32 = at<float>(ws, L.hs32);
  g.redo = wl.redo_gu;
  g.redo_cap = L.sredo_cap;
  g.K = c.hidden;
  g.N = Is;
  if (!launch_w8a8(ln, g)) return MOE_ERR_CUDA;

  launch_quant_rows(ln, at<float>(ws, L.hs32), at<uint16_t>(ws, L.hsq16), nullptr,
                    at<float>(ws, L.hssc), at<int32_t>(ws, L.hsn2), T, Is, nullptr, 0, 0);

  W8Pass d = g;
  d.mode = kW8Down;
  d.tile_start = wl.tc_start_dn;
  d.tile_slot = kWlTcTilesDN;
  d.sched_slot = kWlSchedDN;
  d.w0 = sd;
  d.w1 = nullptr;
  d.s0 = s_down + (size_t)c.n_routed * c.hidden;
  d.s1 = nullptr;
  d.act = at<uint16_t>(ws, L.hsq16);
  d.row_norm2 = at<int32_t>(ws, L.hsn2);
  d.row_scale = at<float>(ws, L.hssc);
  d.out_f32 = y_shared;
  d.redo = wl.redo_dn;
  d.K = Is;
  d.N = c.hidden;
  d.sc = sc;
  d.sc.s2e = nullptr;  // the shared expert's rows are the tokens, at weight 1
  if (!launch_w8a8(ln, d)) return MOE_ERR_CUDA;
  return MOE_OK;
}

}  // namespace

void set_smem_attr_once(const void* func, int bytes, int slot) {
  const int d = current_device();
  if (d < 0 || d >= kMaxDevices || slot < 0 || slot >= kAttrSlots) {
    cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    return;
  }
  if (g_attr_done[slot][d].load(std::memory_order_acquire)) return;
  if (cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) ==
      cudaSuccess)
    g_attr_done[slot][d].store(1, std::memory_order_release);
}

moe_status launch_status_take() { return finish(); }

void launch_note(cudaError_t e) {
  if (e != cudaSuccess && t_launch_error == cudaSuccess) t_launch_error = e;
}

bool folds_enabled() {
  static const bool on = [] {
    const char* v = getenv("MOE_FOLDS");
    return !(v && v[0] == '0' && v[1] == 0);
  }();
  return on;
}

bool pdl_enabled() {
  static const bool on = [] {
    const char* v = getenv("MOE_PDL");
    return !(v && v[0] == '0' && v[1] == 0);
  }();
  return on;
}

void launch_begin(const Launch& L, int kind) {
  g_launches[kind].fetch_add(1, std::memory_order_relaxed);
  t_open_event = nullptr;
  if (g_timing.load(std::memory_order_relaxed)) {
    t_open_event = take_event();
    if (t_open_event) cudaEventRecord(t_open_event, L.stream);
  }
}

void launch_end(const Launch& L, int kind) {
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess && t_launch_error == cudaSuccess) t_launch_error = e;
  if (t_open_event) {
    cudaEvent_t b = take_event();
    if (b) {
      cudaEventRecord(b, L.stream);
      std::lock_guard<std::mutex> lk(g_tmu);
      g_records.push_back({kind, t_open_event, b});
    }
    t_open_event = nullptr;
  }
}

}  // namespace moe

using namespace moe;

extern "C" {

const char* moe_status_string(moe_status s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported configuration";
    case MOE_ERR_ALIGNMENT: return "misaligned pointer";
    case MOE_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_DEVICE_CHECK: return "device-side data check failed";
    case MOE_ERR_DEVICE_TIMEOUT: return "device-side wait timed out";
  }
  return "unknown status";
}

const char* moe_kernel_name(int32_t kind) {
  static const char* names[MOE_K_COUNT] = {
      "router", "topk", "perm_count", "perm_scan", "perm_scatter", "perm_gather", "worklist",
      "gemv_gate_up", "gemv_down", "tc_gate_up", "tc_down", "quant_h", "combine", "w8_exact",
      "sort"};
  return (kind >= 0 && kind < MOE_K_COUNT) ? names[kind] : "unknown";
}

moe_status moe_workspace_size(const moe_config* cfg, int32_t T, size_t* bytes) {
  const moe_status s = check_cfg(cfg, T);
  if (s != MOE_OK) return s;
  if (!bytes) return MOE_ERR_INVALID_ARG;
  *bytes = make_layout(*cfg, T).total;
  return MOE_OK;
}

moe_status moe_route(const moe_config* cfg, int32_t T, const void* x, const float* w_router,
                     const float* bias, int32_t* topk_ids, float* topk_w, void* ws,
                     size_t ws_bytes, moe_stream_t stream) {
  moe_status s = check_cfg(cfg, T);
  if (s != MOE_OK) return s;
  Layout L;
  if ((s = check_ws(*cfg, T, ws, ws_bytes, &L)) != MOE_OK) return s;
  if (T == 0) return MOE_OK;
  if (!x || !w_router || !topk_ids || !topk_w) return MOE_ERR_INVALID_ARG;
  if (cfg->bias_mode != MOE_BIAS_NONE && !bias) return MOE_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(w_router, 16) || !aligned(topk_ids, 16) || !aligned(topk_w, 16))
    return MOE_ERR_ALIGNMENT;
  const Launch ln = make_launch(stream, ws, L);
  const moe_status rs = run_route(ln, *cfg, T, L, ws, x, w_router, bias, topk_ids, topk_w);
  const moe_status f = finish();
  return rs != MOE_OK ? rs : f;
}

moe_status moe_permute(const moe_config* cfg, int32_t T, const int32_t* topk_ids, const void* x,
                       int32_t* counts, int32_t* offsets, int32_t* sorted_to_expanded,
                       int32_t* expanded_to_sorted, void* x_perm, float* x_perm_scale, void* ws,
                       size_t ws_bytes, moe_stream_t stream) {
  moe_status s = check_cfg(cfg, T);
  if (s != MOE_OK) return s;
  Layout L;
  if ((s = check_ws(*cfg, T, ws, ws_bytes, &L)) != MOE_OK) return s;
  if (!counts || !offsets) return MOE_ERR_INVALID_ARG;
  if (T > 0 && (!topk_ids || !x || !sorted_to_expanded || !expanded_to_sorted || !x_perm))
    return MOE_ERR_INVALID_ARG;
  if (cfg->wdtype == MOE_W8A8 && T > 0 && !x_perm_scale) return MOE_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(x_perm, 16) || !aligned(counts, 4) || !aligned(offsets, 4))
    return MOE_ERR_ALIGNMENT;
  const Launch ln = make_launch(stream, ws, L);
  if (T == 0) {
    const int E = cfg->n_routed + cfg->n_zero;
    if (cudaMemsetAsync(counts, 0, E * 4, ln.stream) != cudaSuccess ||
        cudaMemsetAsync(offsets, 0, (E + 1) * 4, ln.stream) != cudaSuccess)
      return MOE_ERR_CUDA;
    return MOE_OK;
  }
  run_permute(ln, *cfg, T, L, ws, topk_ids, x, counts, offsets, sorted_to_expanded,
              expanded_to_sorted, x_perm, x_perm_scale, nullptr);
  return finish();
}

moe_status moe_grouped_ffn(const moe_config* cfg, int32_t T, const int32_t* offsets,
                           const void* x_perm, const float* x_perm_scale, const void* w_gate,
                           const void* w_up, const void* w_down, const float* s_gate,
                           const float* s_up, const float* s_down, float* y_perm, void* ws,
                           size_t ws_bytes, moe_stream_t stream) {
  moe_status s = check_cfg(cfg, T);
  if (s != MOE_OK) return s;
  Layout L;
  if ((s = check_ws(*cfg, T, ws, ws_bytes, &L)) != MOE_OK) return s;
  if (T == 0 || cfg->n_routed == 0) return MOE_OK;
  if (!offsets || !x_perm || !w_gate || !w_up || !w_down || !y_perm) return MOE_ERR_INVALID_ARG;
  const bool w8 = cfg->wdtype == MOE_W8A8;
  if (w8 && (!x_perm_scale || !s_gate || !s_up || !s_down)) return MOE_ERR_INVALID_ARG;
  if (!aligned(x_perm, 16) || !aligned(w_gate, 16) || !aligned(w_up, 16) || !aligned(w_down, 16) ||
      !aligned(y_perm, 16) || !aligned(x_perm_scale, 4) || !aligned(s_gate, 4) ||
      !aligned(s_up, 4) || !aligned(s_down, 4))
    return MOE_ERR_ALIGNMENT;
  const Launch ln = make_launch(stream, ws, L);
  moe_config c = *cfg;
  c.shared_inter = 0;
  if (w8)
    s = run_ffn_w8a8(ln, c, T, L, ws, offsets, x_perm, x_perm_scale, w_gate, w_up, w_down, s_gate,
                     s_up, s_down, y_perm, false);
  else
    s = run_ffn(ln, c, T, L, ws, offsets, x_perm, w_gate, w_up, w_down, y_perm, nullptr, nullptr,
                nullptr, nullptr, nullptr, false);
  const moe_status f = finish();
  return s != MOE_OK ? s : f;
}

moe_status moe_combine(const moe_config* cfg, int32_t T, const float* y_perm,
                       const int32_t* expanded_to_sorted, const int32_t* topk_ids,
                       const float* topk_w, const void* x, const float* shared_out, void* out,
                       moe_stream_t stream) {
  const moe_status s = check_cfg(cfg, T);
  if (s != MOE_OK) return s;
  if (T == 0) return MOE_OK;
  if (!expanded_to_sorted || !topk_ids || !topk_w || !x || !out) return MOE_ERR_INVALID_ARG;
  if (cfg->n_routed > 0 && !y_perm) return MOE_ERR_INVALID_ARG;
  if (!aligned(y_perm, 16) || !aligned(x, 16) || !aligned(shared_out, 16) || !aligned(out, 16))
    return MOE_ERR_ALIGNMENT;
  Launch ln;
  ln.stream = reinterpret_cast<cudaStream_t>(stream);
  ln.num_sms = sm_count(current_device());
  ln.status = nullptr;
  launch_combine(ln, *cfg, T, y_perm, expanded_to_sorted, topk_ids, topk_w, x, shared_out, out);
  return finish();
}

moe_status moe_layer_forward(const moe_config* cfg, int32_t T, const void* x,
                             const float* w_router, const float* bias, const void* w_gate,
                             const void* w_up, const void* w_down, const float* s_gate,
                             const float* s_up, const float* s_down, const void* ws_gate,
                             const void* ws_up, const void* ws_down, void* out, void* ws,
                             size_t ws_bytes, moe_stream_t stream) {
  moe_status s = check_cfg(cfg, T);
  if (s != MOE_OK) return s;
  Layout L;
  if ((s = check_ws(*cfg, T, ws, ws_bytes, &L)) != MOE_OK) return s;
  if (T == 0) return MOE_OK;
  if (!x || !w_router || !out) return MOE_ERR_INVALID_ARG;
  if (cfg->bias_mode != MOE_BIAS_NONE && !bias) return MOE_ERR_INVALID_ARG;
  if (cfg->n_routed > 0 && (!w_gate || !w_up || !w_down)) return MOE_ERR_INVALID_ARG;
  const bool w8 = cfg->wdtype == MOE_W8A8;
  if (w8 && cfg->n_routed > 0 && (!s_gate || !s_up || !s_down)) return MOE_ERR_INVALID_ARG;
  if (!aligned(s_gate, 4) || !aligned(s_up, 4) || !aligned(s_down, 4)) return MOE_ERR_ALIGNMENT;
  if (cfg->shared_inter > 0 && (!ws_gate || !ws_up || !ws_down)) return MOE_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(w_router, 16) || !aligned(w_gate, 16) || !aligned(w_up, 16) ||
      !aligned(w_down, 16) || !aligned(ws_gate, 16) || !aligned(ws_up, 16) ||
      !aligned(ws_down, 16) || !aligned(out, 16))
    return MOE_ERR_ALIGNMENT;
  const Launch ln = make_launch(stream, ws, L);
  const moe_config& c = *cfg;
  int32_t* ids = at<int32_t>(ws, L.ids);
  float* w = at<float>(ws, L.w);
  int32_t* counts = at<int32_t>(ws, L.counts);
  int32_t* offsets = at<int32_t>(ws, L.offsets);
  int32_t* s2e = at<int32_t>(ws, L.s2e);
  int32_t* e2s = at<int32_t>(ws, L.e2s);
  void* x_perm = w8 ? nullptr : at<void>(ws, L.x_perm);
  float* x_scale = at<float>(ws, L.x_scale);
  const bool fused = fused_combine(c);
  float* y = fused ? nullptr : at<float>(ws, L.y);
  float* y_s = c.shared_inter > 0 && !fused ? at<float>(ws, L.y_s) : nullptr;
  // fused combine: the tokens' fp32 accumulators (the output itself when fp32)
  float* acc = !fused ? nullptr : c.out_fp32 ? static_cast<float*>(out) : at<float>(ws, L.acc);
  ScatterAdd sc{};
  if (fused) {
    sc.acc = acc;
    sc.s2e = s2e;
    sc.w = w;
    sc.k = c.top_k;
  }
  // small layers: the one-CTA re-sort routes the tokens first (one launch fewer)
  const bool route_in_sort = route_small_fits(c, T) && folds_enabled();
  const SmallRoute sroute{static_cast<const uint16_t*>(x), w_router, c.hidden};
  const TopkArgs stk = topk_args(ln, c, T, nullptr, bias, ids, w);
  if (!route_in_sort) {
    const moe_status rs = run_route(ln, c, T, L, ws, x, w_router, bias, ids, w);
    if (rs != MOE_OK) {
      finish();
      return rs;
    }
  }
  // the FFN's work list is built with the re-sort when that runs as one CTA
  // (the small-layer FFN reads only the offsets)
  const bool ffn = w8 ? c.n_routed > 0
                      : ((c.n_routed > 0 || c.shared_inter > 0) &&
                         !(c.shared_inter == 0 && small_ffn_chosen(c, T)));
  const WlPlan plan = wl_plan(c, T, !w8 && c.shared_inter > 0);
  const bool wl_built =
      run_permute(ln, c, T, L, ws, ids, x, counts, offsets, s2e, e2s, x_perm, x_scale,
                  ffn ? &plan : nullptr, w, acc, route_in_sort ? &sroute : nullptr,
                  route_in_sort ? &stk : nullptr);
  const bool w8_shared = w8 && c.shared_inter > 0;
  if (w8 && c.n_routed > 0) {
    QuantGatherOut qo{};
    qo.x16 = at<uint16_t>(ws, L.x16);
    qo.x8 = gemv_possible(plan.gemv_max) ? at<int8_t>(ws, L.x8) : nullptr;
    qo.scale = x_scale;
    qo.norm2 = at<int32_t>(ws, L.xn2);
    if (w8_shared) {
      qo.tok16 = at<uint16_t>(ws, L.xs16);
      qo.tok_scale = at<float>(ws, L.xss);
      qo.tok_norm2 = at<int32_t>(ws, L.xsn2);
    }
    launch_quant_gather(ln, c, T, x, ids, e2s, offsets, plan.gemv_max, qo, w, acc);
  }
  // small bf16 layers: the down pass's last CTA rounds the output itself
  SmallFinalize fin{};
  if (fused && !c.out_fp32 && !w8 && c.n_routed > 0 &&
      (long long)T * c.hidden <= kSmallFinalizeElems && folds_enabled()) {
    fin.ctr = reinterpret_cast<int*>(static_cast<char*>(ws) + L.status + kFinalizeCtrOffset);
    fin.acc = acc;
    fin.out = static_cast<uint16_t*>(out);
    fin.n8 = T * c.hidden / 8;
  }
  moe_status fs = MOE_OK;
  if (w8 && c.n_routed > 0) {
    fs = run_ffn_w8a8(ln, c, T, L, ws, offsets, x_perm, x_scale, w_gate, w_up, w_down, s_gate,
                      s_up, s_down, y, wl_built, sc);
    if (fs == MOE_OK && w8_shared)
      fs = run_shared_w8a8(ln, c, T, L, ws, ws_gate, ws_up, ws_down, s_gate, s_up, s_down, y_s,
                           sc);
  } else if (!w8 && (c.n_routed > 0 || c.shared_inter > 0)) {
    fs = run_ffn(ln, c, T, L, ws, offsets, x_perm, w_gate, w_up, w_down, y, x, ws_gate, ws_up,
                 ws_down, y_s, wl_built, sc, fin);
  }
  if (!fused)
    launch_combine(ln, c, T, y, e2s, ids, w, x, y_s, out);
  else if (!c.out_fp32 && !fin.ctr)
    launch_finalize(ln, T, c.hidden, acc, out);
  const moe_status f = finish();
  return fs != MOE_OK ? fs : f;
}

namespace {
struct QLayout {
  size_t tasks, start_gu, start_dn, tc_tasks, tc_gu, tc_dn, counts, a16, an2, redo, total;
  int cap, redo_cap;
};
QLayout qgemm_layout(int E, int K, int N, int R) {
  QLayout Q{};
  Q.cap = E + 4 + R / kTcMaxN;
  // one exact-fallback entry per CTA half of each two-SM tile of 256 channels
  Q.redo_cap = Q.cap * 2 * ((N + 2 * kTcM - 1) / (2 * kTcM));
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off = align256(off + bytes);
    return at;
  };
  take(256 + kRouterCounterBytes);  // status word (same head as the layer workspace)
  Q.tasks = take((size_t)Q.cap * sizeof(FfnTask));
  Q.start_gu = take((size_t)Q.cap * 4);
  Q.start_dn = take((size_t)Q.cap * 4);
  Q.tc_tasks = take((size_t)Q.cap * sizeof(FfnTask));
  Q.tc_gu = take((size_t)Q.cap * 4);
  Q.tc_dn = take((size_t)Q.cap * 4);
  Q.counts = take(kWlCount * 4);
  Q.a16 = take((size_t)R * K * 2);
  Q.an2 = take((size_t)R * 4);
  Q.redo = take((size_t)(1 + Q.redo_cap) * 4);
  Q.total = off;
  return Q;
}
moe_status check_qgemm(int E, int K, int N, int R) {
  if (E < 1 || K < 16 || K % 16 || N < 1 || R < 0) return MOE_ERR_INVALID_ARG;
  if (E > kMaxExperts || K > 131071 || (long long)R * (K > N ? K : N) > (1LL << 40))
    return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}
}  // namespace

moe_status moe_qgemm_s8_workspace_size(int32_t n_experts, int32_t K, int32_t N, int32_t R,
                                       size_t* bytes) {
  const moe_status s = check_qgemm(n_experts, K, N, R);
  if (s != MOE_OK) return s;
  if (!bytes) return MOE_ERR_INVALID_ARG;
  *bytes = qgemm_layout(n_experts, K, N, R).total;
  return MOE_OK;
}

moe_status moe_qgemm_s8(int32_t n_experts, int32_t K, int32_t N, int32_t R, const int32_t* offsets,
                        const void* a, const void* w, int32_t* acc, void* ws, size_t ws_bytes,
                        moe_stream_t stream) {
  moe_status s = check_qgemm(n_experts, K, N, R);
  if (s != MOE_OK) return s;
  const QLayout Q = qgemm_layout(n_experts, K, N, R);
  if (!ws || !offsets || !w || !acc || (R > 0 && !a)) return MOE_ERR_INVALID_ARG;
  if (!aligned(ws, 256)) return MOE_ERR_ALIGNMENT;
  if (ws_bytes < Q.total) return MOE_ERR_WORKSPACE_TOO_SMALL;
  if (!aligned(a, 16) || !aligned(w, 16) || !aligned(acc, 4) || !aligned(offsets, 4))
    return MOE_ERR_ALIGNMENT;
  if (R == 0) return MOE_OK;
  Launch ln;
  ln.stream = reinterpret_cast<cudaStream_t>(stream);
  ln.num_sms = sm_count(current_device());
  ln.status = at<DevStatus>(ws, 0);
  WorkList wl;
  wl.gemv_tasks = at<FfnTask>(ws, Q.tasks);
  wl.gemv_start_gu = at<int32_t>(ws, Q.start_gu);
  wl.gemv_start_dn = at<int32_t>(ws, Q.start_dn);
  wl.tc_tasks = at<FfnTask>(ws, Q.tc_tasks);
  wl.tc_start_gu = at<int32_t>(ws, Q.tc_gu);
  wl.tc_start_dn = at<int32_t>(ws, Q.tc_dn);
  wl.counts = at<int32_t>(ws, Q.counts);
  wl.capacity = Q.cap;
  wl.redo_gu = nullptr;
  wl.redo_dn = at<int32_t>(ws, Q.redo);
  wl.gu_done = nullptr;
  // Tasks: the experts' row ranges in <= 256-row chunks, N/256 two-SM tiles
  // each (the work-list kernel's W8A8 "down" tiling, hidden = N).
  moe_config c{};
  c.hidden = N;
  c.inter = 16;
  c.n_routed = n_experts;
  c.top_k = 1;
  c.n_group = 1;
  c.wdtype = MOE_W8A8;
  launch_worklist(ln, c, R, offsets, wl, 0, 1, kW8MaxN);
  uint16_t* a16 = at<uint16_t>(ws, Q.a16);
  int32_t* an2 = at<int32_t>(ws, Q.an2);
  launch_i8_rows_to_f16(ln, static_cast<const int8_t*>(a), a16, an2, R, K, offsets + n_experts);
  W8Pass p{};
  p.mode = kW8Raw;
  p.tasks = wl.tc_tasks;
  p.tile_start = wl.tc_start_dn;
  p.counts = wl.counts;
  p.task_slot = kWlTcTasks;
  p.tile_slot = kWlTcTilesDN;
  p.sched_slot = kWlSchedDN;
  p.w0 = w;
  p.n_experts = n_experts;
  p.act = a16;
  p.act_rows = R;
  p.row_norm2 = an2;
  p.out_i32 = acc;
  p.redo = wl.redo_dn;
  p.redo_cap = Q.redo_cap;
  p.K = K;
  p.N = N;
  const bool ok = launch_w8a8(ln, p);
  const moe_status f = finish();
  return ok ? f : MOE_ERR_CUDA;
}

moe_status moe_tile_choice(const moe_config* cfg, int32_t T, int32_t* gemv_max_rows,
                           int32_t* one_launch) {
  const moe_status s = check_cfg(cfg, T);
  if (s != MOE_OK) return s;
  if (!gemv_max_rows || !one_launch) return MOE_ERR_INVALID_ARG;
  *gemv_max_rows = effective_gemv_max(*cfg, T);
  // 0 two launches, 1 one, 2 one with wide down tiles
  *one_launch = ffn_dn_wide(*cfg, T) ? 2 : ffn_one_launch(*cfg, T) ? 1 : 0;
  return MOE_OK;
}

moe_status moe_check_device_status(void* ws, moe_stream_t stream) {
  if (!ws) return MOE_ERR_INVALID_ARG;
  if (!aligned(ws, 256)) return MOE_ERR_ALIGNMENT;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  DevStatus h{};
  if (cudaMemcpyAsync(&h, ws, sizeof h, cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return MOE_ERR_CUDA;
  if (h.bits == 0u) return MOE_OK;
  if (cudaMemsetAsync(ws, 0, sizeof h, st) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return MOE_ERR_CUDA;
  return (h.bits & kStTimeout) ? MOE_ERR_DEVICE_TIMEOUT : MOE_ERR_DEVICE_CHECK;
}

moe_status moe_selftest_wait_timeout(void* ws, int64_t limit_cycles, moe_stream_t stream) {
  if (!ws || limit_cycles < 1 || limit_cycles > kWaitCycles) return MOE_ERR_INVALID_ARG;
  if (!aligned(ws, 256)) return MOE_ERR_ALIGNMENT;
  Launch ln;
  ln.stream = reinterpret_cast<cudaStream_t>(stream);
  ln.num_sms = sm_count(current_device());
  ln.status = at<DevStatus>(ws, 0);
  launch_wait_timeout_selftest(ln, limit_cycles);
  return finish();
}

moe_status moe_timing_enable(int32_t enable) {
  g_timing.store(enable != 0);
  return MOE_OK;
}

moe_status moe_timing_collect(float* ms, int32_t* launches, int32_t n) {
  if (!ms || !launches || n < MOE_K_COUNT) return MOE_ERR_INVALID_ARG;
  std::vector<TimedLaunch> recs;
  {
    std::lock_guard<std::mutex> lk(g_tmu);
    recs.swap(g_records);
  }
  for (int i = 0; i < n; ++i) {
    ms[i] = 0.f;
    launches[i] = 0;
  }
  moe_status s = MOE_OK;
  for (const TimedLaunch& r : recs) {
    float t = 0.f;
    if (cudaEventSynchronize(r.b) != cudaSuccess || cudaEventElapsedTime(&t, r.a, r.b) != cudaSuccess)
      s = MOE_ERR_CUDA;
    ms[r.kind] += t;
    launches[r.kind] += 1;
  }
  std::lock_guard<std::mutex> lk(g_tmu);
  for (const TimedLaunch& r : recs) {
    g_event_pool.push_back(r.a);
    g_event_pool.push_back(r.b);
  }
  return s;
}

moe_status moe_launch_counts(int64_t* launches, int32_t n) {
  if (!launches || n < MOE_K_COUNT) return MOE_ERR_INVALID_ARG;
  for (int i = 0; i < MOE_K_COUNT; ++i) launches[i] = g_launches[i].load();
  for (int i = MOE_K_COUNT; i < n; ++i) launches[i] = 0;
  return MOE_OK;
}

}  // extern "C"
