// Grouped SwiGLU FFN of the smallest layers (a few tokens, experts of a few
// hundred KB): latency, not bandwidth, sets their pace.  The persistent
// tensor-core kernel spends most of such a layer in its claim / hand-off /
// fence chain between a gate/up tile and the down tiles of other CTAs; here a
// cluster of kSfCluster CTAs takes a whole expert instead, CTA q a quarter:
//   - its rows, a quarter of the gate and up rows and a quarter of the down
//     rows land in shared memory as a few TMA boxes of 64 columns (128-byte
//     rows, 128-byte swizzle, so the MMA fragment loads of eight rows hit
//     different banks);
//   - warps run gate/up as warp-level bf16 MMAs (m16n8k16, fp32 accumulate),
//     a 16-channel tile of both matrices each, SwiGLU in registers, and write
//     h, rounded to bf16 as on the tensor-core path, into the shared memory of
//     every CTA of the cluster;
//   - after one cluster barrier each CTA runs its quarter of the down
//     projection over the whole h and adds w * y into the tokens' fp32
//     accumulators (or stores the y rows for the ordered combine).
// The products are the grouped FFN of the Pangu Pro MoE disclosure, section
// SwiftGMM, for experts whose weights stay in L2.
#include <cudaTypedefs.h>

#include <atomic>
#include <cstring>
#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "small_ffn.h"

namespace moe {

namespace {

constexpr int kSfThreads = 256;  // 8 warps
constexpr int kSfWarps = kSfThreads / 32;
constexpr int kSfBoxK = 64;      // columns of a TMA box: one 128-byte row
constexpr int kSfCluster = 4;    // CTAs per expert (a cluster)
constexpr int kSfSmemMax = 220 * 1024;

struct SfMaps {
  CUtensorMap wg, wu;  // [E_r * I rows][H], boxes of 64 columns x I / 4 rows
  CUtensorMap wd;      // [E_r * H rows][I], boxes of 64 columns x H / 4 rows
  CUtensorMap x;       // [R rows][H], boxes of 64 columns x 16 rows
};

// Shared-memory plan of one CTA: its gate and up rows (H / 64 boxes of I / 4
// rows each), its down rows (I / 64 boxes of H / 4 rows), x and the whole h
// (16 rows), every box 1024-byte aligned, then the copy barrier.
struct SfPlan {
  uint32_t wg, wu, wd, x, h, bar, total;
};
__host__ __device__ inline SfPlan sf_plan(int H, int I) {
  SfPlan p;
  const uint32_t Is = (uint32_t)I / kSfCluster, Hs = (uint32_t)H / kSfCluster;
  p.wg = 0;
  p.wu = p.wg + Is * H * 2;
  p.wd = p.wu + Is * H * 2;
  p.x = p.wd + Hs * I * 2;
  p.h = p.x + (uint32_t)kSmallFfnMaxRows * H * 2;
  p.bar = p.h + (uint32_t)kSmallFfnMaxRows * I * 2;
  p.total = p.bar + 16;
  return p;
}

// Byte offset of element (r, k) of a matrix staged as 64-column boxes of
// `rows` rows each: 128-byte rows whose 16-byte chunks are swizzled by the row
// (chunk c of row r sits at c ^ (r % 8)).
__device__ __forceinline__ uint32_t swz(uint32_t rows, int r, int k) {
  const int b = k >> 6, kk = k & 63;
  return (uint32_t)b * rows * 128u + (uint32_t)r * 128u +
         ((uint32_t)(((kk >> 3) ^ (r & 7)) << 4) | (uint32_t)((kk & 7) << 1));
}

__device__ __forceinline__ uint32_t ld_s32(const uint8_t* p) {
  return *reinterpret_cast<const uint32_t*>(p);
}
__device__ __forceinline__ void st_cluster_u16(uint32_t cluster_addr, uint16_t v) {
  asm volatile("st.shared::cluster.u16 [%0], %1;" ::"r"(cluster_addr), "h"(v) : "memory");
}

// D (16 x 8, fp32) += A (16 x 16, bf16, row-major) * B (16 x 8, bf16, given as
// its transpose's rows): the warp-level MMA fragment layout, lane = 4 g + t.
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4],
                                               const uint32_t (&b)[2]) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// A fragment: rows r0 .. r0 + 15, columns k0 .. k0 + 15 of a staged matrix
// whose boxes hold `rows` rows.
__device__ __forceinline__ void load_a(const uint8_t* base, uint32_t rows, int r0, int k0, int g,
                                       int t, uint32_t (&a)[4]) {
  a[0] = ld_s32(base + swz(rows, r0 + g, k0 + 2 * t));
  a[1] = ld_s32(base + swz(rows, r0 + g + 8, k0 + 2 * t));
  a[2] = ld_s32(base + swz(rows, r0 + g, k0 + 2 * t + 8));
  a[3] = ld_s32(base + swz(rows, r0 + g + 8, k0 + 2 * t + 8));
}
// B fragment: columns n0 .. n0 + 7 are rows n0 .. n0 + 7 of a staged matrix
// (its K along the row), K range k0 .. k0 + 15.
__device__ __forceinline__ void load_b(const uint8_t* base, uint32_t rows, int n0, int k0, int g,
                                       int t, uint32_t (&b)[2]) {
  b[0] = ld_s32(base + swz(rows, n0 + g, k0 + 2 * t));
  b[1] = ld_s32(base + swz(rows, n0 + g, k0 + 2 * t + 8));
}

__global__ void __launch_bounds__(kSfThreads, 1)
    small_ffn_kernel(const __grid_constant__ SfMaps maps, const SmallFfnArgs a, DevStatus* st) {
  extern __shared__ uint8_t sm_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(sm_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  __shared__ int last;
  const SfPlan p = sf_plan(a.H, a.I);
  const int e = blockIdx.x / kSfCluster, q = (int)cluster_rank();
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const int g = lane / 4, t = lane % 4;
  const uint32_t bar = smem_u32(sm + p.bar);
  if (tid == 0) {
    mbar_init(bar, 1);
    fence_barrier_init();
    prefetch_tensormap(&maps.wg);
    prefetch_tensormap(&maps.wu);
    prefetch_tensormap(&maps.wd);
    prefetch_tensormap(&maps.x);
  }
  __syncthreads();
  cluster_sync_all();  // every CTA of the cluster runs before any writes into another
  pdl_enter();
  const int H = a.H, I = a.I, Is = I / kSfCluster, Hs = H / kSfCluster;
  const int r0 = a.offsets[e];
  int n = a.offsets[e + 1] - r0;  // the same in every CTA of the cluster
  if (n > kSmallFfnMaxRows) {     // more rows than tokens: bad offsets
    if (tid == 0) raise_status(st, kStInternal, MOE_K_TC_GATE_UP);
    n = 0;
  }
  if (n > 0) {
    if (tid == 0) {
      // this CTA's gate, up and down rows and the expert's rows (16 from r0;
      // rows of other experts or past the end only feed output columns that
      // are not kept)
      mbar_arrive_expect_tx(bar, (uint32_t)(4 * Is * H + 2 * Hs * I + 2 * kSmallFfnMaxRows * H));
      const uint64_t pol = policy_evict_last();
      for (int b = 0; b < H / kSfBoxK; ++b) {
        tma_load_2d(smem_u32(sm + p.wg + b * Is * 128), &maps.wg, b * kSfBoxK, e * I + q * Is,
                    bar, pol);
        tma_load_2d(smem_u32(sm + p.wu + b * Is * 128), &maps.wu, b * kSfBoxK, e * I + q * Is,
                    bar, pol);
        tma_load_2d(smem_u32(sm + p.x + b * kSmallFfnMaxRows * 128), &maps.x, b * kSfBoxK, r0,
                    bar, pol);
      }
      for (int b = 0; b < I / kSfBoxK; ++b)
        tma_load_2d(smem_u32(sm + p.wd + b * Hs * 128), &maps.wd, b * kSfBoxK, e * H + q * Hs,
                    bar, pol);
    }
    const bool ok = __syncthreads_and(mbar_wait(bar, 0));
    if (!ok) {
      // report, and give the copies in flight one more bounded wait
      if (tid == 0) raise_status(st, kStTimeout, MOE_K_TC_GATE_UP);
      mbar_wait(bar, 0);
    }
    const int ntn = n > 8 ? 2 : 1;  // 8-row MMA column tiles with rows
    if (ok) {
      // gate/up: warp w takes this CTA's channel tile w (of Is / 16), and
      // writes h into the same place in every CTA of the cluster
      uint32_t hbase[kSfCluster];
#pragma unroll
      for (int j = 0; j < kSfCluster; ++j) hbase[j] = mapa_shared(smem_u32(sm + p.h), (uint32_t)j);
      for (int m = warp; m < Is / 16; m += kSfWarps) {
        float cg[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
        float cu[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
        for (int k0 = 0; k0 < H; k0 += 16) {
          uint32_t ag[4], au[4];
          load_a(sm + p.wg, Is, m * 16, k0, g, t, ag);
          load_a(sm + p.wu, Is, m * 16, k0, g, t, au);
          for (int nt = 0; nt < ntn; ++nt) {
            uint32_t b[2];
            load_b(sm + p.x, kSmallFfnMaxRows, nt * 8, k0, g, t, b);
            mma_bf16_16816(cg[nt], ag, b);
            mma_bf16_16816(cu[nt], au, b);
          }
        }
        // element j of a tile: channel m * 16 + g (+ 8 for j >= 2), row 2t (+ 1 for odd j)
        for (int nt = 0; nt < ntn; ++nt)
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int ch = q * Is + m * 16 + g + (j >= 2 ? 8 : 0), r = nt * 8 + 2 * t + (j & 1);
            const float gv = cg[nt][j];
            const uint16_t h = f_to_bf16(gv * __frcp_rn(1.f + __expf(-gv)) * cu[nt][j]);
            const uint32_t off = swz(kSmallFfnMaxRows, r, ch);
#pragma unroll
            for (int c = 0; c < kSfCluster; ++c) st_cluster_u16(hbase[c] + off, h);
          }
      }
    }
    cluster_sync_all();  // h complete in every CTA (reached by every CTA of the cluster)
    if (ok) {
      // down: warp w takes this CTA's output-channel tile w (of Hs / 16)
      const bool fused = a.sc.acc != nullptr;
      for (int m = warp; m < Hs / 16; m += kSfWarps) {
        float c[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
        for (int k0 = 0; k0 < I; k0 += 16) {
          uint32_t ad[4];
          load_a(sm + p.wd, Hs, m * 16, k0, g, t, ad);
          for (int nt = 0; nt < ntn; ++nt) {
            uint32_t b[2];
            load_b(sm + p.h, kSmallFfnMaxRows, nt * 8, k0, g, t, b);
            mma_bf16_16816(c[nt], ad, b);
          }
        }
        for (int nt = 0; nt < ntn; ++nt)
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int ch = q * Hs + m * 16 + g + (j >= 2 ? 8 : 0), r = nt * 8 + 2 * t + (j & 1);
            if (r >= n) continue;
            if (fused) {
              int tk;
              float wt;
              scatter_target(a.sc, r0 + r, false, &tk, &wt);
              atomicAdd(a.sc.acc + (size_t)tk * H + ch, wt * c[nt][j]);
            } else {
              a.out_y[(size_t)(r0 + r) * H + ch] = c[nt][j];
            }
          }
      }
    }
  }
  if (!a.fin.ctr) return;
  // the last CTA to finish rounds the accumulators (each thread's adds are
  // fenced before its CTA counts itself done)
  __threadfence();
  __syncthreads();
  if (tid == 0) last = atomicAdd(a.fin.ctr, 1) == (int)gridDim.x - 1;
  __syncthreads();
  if (!last) return;
  __threadfence();
  for (int i = tid; i < a.fin.n8; i += kSfThreads) {
    const float4 v0 = __ldcg(reinterpret_cast<const float4*>(a.fin.acc) + 2 * i);
    const float4 v1 = __ldcg(reinterpret_cast<const float4*>(a.fin.acc) + 2 * i + 1);
    const uint32_t q0 = (uint32_t)f_to_bf16(v0.x) | ((uint32_t)f_to_bf16(v0.y) << 16);
    const uint32_t q1 = (uint32_t)f_to_bf16(v0.z) | ((uint32_t)f_to_bf16(v0.w) << 16);
    const uint32_t q2 = (uint32_t)f_to_bf16(v1.x) | ((uint32_t)f_to_bf16(v1.y) << 16);
    const uint32_t q3 = (uint32_t)f_to_bf16(v1.z) | ((uint32_t)f_to_bf16(v1.w) << 16);
    reinterpret_cast<uint4*>(a.fin.out)[i] = make_uint4(q0, q1, q2, q3);
  }
  if (tid == 0) *a.fin.ctr = 0;  // ready for the next call
}

constexpr int kSfMaxDevices = 64;
std::atomic<int> g_sf_attr[kSfMaxDevices];

PFN_cuTensorMapEncodeTiled_v12000 sf_encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* q = nullptr;
    cudaDriverEntryPointQueryResult r;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &q, 12000, cudaEnableDefault,
                                         &r) == cudaSuccess &&
        r == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(q);
  });
  return fn;
}

// bf16 matrix [rows][cols] (cols contiguous) in boxes of 64 columns x box_rows
// rows, 128-byte swizzle; rows and columns past the matrix read as zero.
bool sf_map(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows, uint32_t box_rows) {
  auto fn = sf_encode_fn();
  if (!fn || !base) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 2};
  const cuuint32_t box[2] = {(cuuint32_t)kSfBoxK, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool small_ffn_fits(const moe_config& c, int T) {
  // (a cluster per routed expert, empty or not: at most kSmallFfnMaxExperts)
  if (c.wdtype != MOE_W_BF16 || c.shared_inter > 0 || c.n_routed < 1 ||
      c.n_routed > kSmallFfnMaxExperts)
    return false;
  if (T < 1 || T > kSmallFfnMaxRows) return false;
  // whole 64-column boxes, at most 256 rows a box
  if (c.hidden % kSfBoxK != 0 || c.inter % kSfBoxK != 0 || c.hidden > 256 || c.inter > 256)
    return false;
  return sf_plan(c.hidden, c.inter).total + 1024 <= (uint32_t)kSfSmemMax;
}

bool launch_small_ffn(const Launch& L, const SmallFfnArgs& a) {
  SfMaps maps;
  memset(&maps, 0, sizeof maps);
  const uint64_t er = (uint64_t)a.E_r;
  if (!sf_map(&maps.wg, a.w_gate, a.H, er * a.I, a.I / kSfCluster) ||
      !sf_map(&maps.wu, a.w_up, a.H, er * a.I, a.I / kSfCluster) ||
      !sf_map(&maps.wd, a.w_down, a.I, er * a.H, a.H / kSfCluster) ||
      !sf_map(&maps.x, a.x_perm, a.H, a.R, kSmallFfnMaxRows))
    return false;
  const uint32_t smem = sf_plan(a.H, a.I).total + 1024;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kSfMaxDevices) dev = -1;
  if (dev < 0 || !g_sf_attr[dev].load(std::memory_order_acquire)) {
    if (cudaFuncSetAttribute(reinterpret_cast<const void*>(small_ffn_kernel),
                             cudaFuncAttributeMaxDynamicSharedMemorySize, kSfSmemMax) ==
            cudaSuccess &&
        dev >= 0)
      g_sf_attr[dev].store(1, std::memory_order_release);
  }
  launch_begin(L, MOE_K_TC_GATE_UP);
  launch_kernel_cluster(small_ffn_kernel, dim3(a.E_r * kSfCluster), dim3(kSfCluster), kSfThreads,
                        smem, L.stream, maps, a, L.status);
  launch_end(L, MOE_K_TC_GATE_UP);
  return true;
}

}  // namespace moe
