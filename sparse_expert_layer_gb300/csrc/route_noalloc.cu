// moe_route_noalloc: routing for callers that cannot hand the library any
// device memory beyond the tensors themselves.
//
// Who needs it: a host framework that gives an operator only its input and
// output buffers (and owns every other allocation), or a latency-bound decode
// loop that must not call cudaMalloc, which can synchronise the device and take
// milliseconds.  moe_route needs a caller-provided workspace for the router's
// split-K partial logits; this entry point keeps that scratch in a fixed array
// compiled into the library instead, so the caller passes x, the router
// weights, the bias and the two outputs, and nothing is allocated.
//
// It always runs the small-batch routers (the decode router on tensor cores,
// or the CUDA-core router), also for batches where moe_route switches to its
// large-batch router (at least 1024 tokens, H a multiple of 64, 64 or more
// 128 x 128 tiles), which needs a split copy of the router weights.  There the
// two entry points sum the same products in different orders: routing ids are
// the same unless two keys are closer than the logits' rounding, and weights
// agree to about 1e-5 relative.
//
// The array (4 MiB of logits and split-K partials after a 4 KB head: status
// word and router tile counters) exists on every GPU that loads the library and
// stays there until the process exits.  All calls on a device share it: two
// calls whose work overlaps on that GPU (different streams, or different host
// threads) race on it and may return wrong results.  Logits and partials are
// fully rewritten by every call, the counters start at zero and the router
// leaves them zero, and the status word is zeroed at the start of every call.
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace moe {

namespace {

constexpr size_t kNoAllocStatusBytes = 256;
constexpr size_t kNoAllocHeadBytes = kNoAllocStatusBytes + kRouterCounterBytes;
constexpr size_t kNoAllocScratchBytes = (size_t)4 << 20;  // 4 MiB of fp32 logits + partials
constexpr int kNoAllocMaxDevices = 64;

// Status word, router tile counters (zero at load time; the router leaves them
// zero after every call), then final and split-K partial logits.
static __device__ __align__(256) unsigned char g_route_scratch[kNoAllocHeadBytes +
                                                               kNoAllocScratchBytes];

std::mutex g_setup_mu;
void* g_scratch_ptr[kNoAllocMaxDevices] = {};

// Device address of the array for the current device.  The host-side symbol is
// only a stand-in; the address must come from cudaGetSymbolAddress, called once
// per device with that device current.
moe_status scratch_for_current_device(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  if (dev < 0 || dev >= kNoAllocMaxDevices) return MOE_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_setup_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_route_scratch) != cudaSuccess || !p) return MOE_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return MOE_OK;
}

}  // namespace

}  // namespace moe

using namespace moe;

extern "C" moe_status moe_route_noalloc(const moe_config* cfg, int32_t T, const void* x,
                                        const float* w_router, const float* bias,
                                        int32_t* topk_ids, float* topk_w, moe_stream_t stream) {
  size_t need = 0;
  moe_status s = moe_workspace_size(cfg, T, &need);  // validates cfg and T
  if (s != MOE_OK) return s;
  if (T == 0) return MOE_OK;
  if (!x || !w_router || !topk_ids || !topk_w) return MOE_ERR_INVALID_ARG;
  if (cfg->bias_mode != MOE_BIAS_NONE && !bias) return MOE_ERR_INVALID_ARG;
  const uintptr_t mis = reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(w_router) |
                        reinterpret_cast<uintptr_t>(topk_ids) |
                        reinterpret_cast<uintptr_t>(topk_w);
  if (mis & 15u) return MOE_ERR_ALIGNMENT;
  const int E = cfg->n_routed + cfg->n_zero;
  // The decode router on tensor cores needs no split-K partials; the CUDA-core
  // router splits K as moe_route does.  (Should the tensor-core router's maps
  // fail to encode, the fallback runs unsplit, so it needs no partials either.)
  const int splits = router_tc_decode_chosen(*cfg, T) ? 1 : router_splits_default(*cfg, T);
  const size_t logit_bytes = (size_t)T * E * sizeof(float);
  const size_t partial_bytes = splits > 1 ? (size_t)splits * logit_bytes : 0;
  if (logit_bytes + partial_bytes > kNoAllocScratchBytes) return MOE_ERR_WORKSPACE_TOO_SMALL;

  void* base = nullptr;
  if ((s = scratch_for_current_device(&base)) != MOE_OK) return s;
  Launch L;
  L.stream = reinterpret_cast<cudaStream_t>(stream);
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return MOE_ERR_CUDA;
  L.num_sms = sms;
  L.status = static_cast<DevStatus*>(base);
  unsigned char* b = static_cast<unsigned char*>(base);
  int* counters = reinterpret_cast<int*>(b + kNoAllocStatusBytes);
  float* logits = reinterpret_cast<float*>(b + kNoAllocHeadBytes);
  float* partial = reinterpret_cast<float*>(b + kNoAllocHeadBytes + logit_bytes);
  if (cudaMemsetAsync(base, 0, kNoAllocStatusBytes, L.stream) != cudaSuccess) return MOE_ERR_CUDA;
  launch_route(L, *cfg, T, x, w_router, bias, partial, splits, logits, counters, topk_ids, topk_w);
  return launch_status_take();
}
