// Grouped SwiGLU FFN of the smallest layers in one launch (small_ffn.cu).
#pragma once

#include "internal.h"

namespace moe {

// Whether (c, T) takes the small-layer FFN: bf16 weights, no shared expert, at
// most kSmallFfnMaxRows tokens (so at most that many rows per expert) and
// kSmallFfnMaxExperts routed experts, H and I multiples of 64 and at most 256,
// and a quarter of one expert's weights plus its rows fit one CTA's shared
// memory.
constexpr int kSmallFfnMaxRows = 16;
constexpr int kSmallFfnMaxExperts = 64;
bool small_ffn_fits(const moe_config& c, int T);

// A cluster of four CTAs per routed expert: its rows x_perm[offsets[e] ..
// offsets[e + 1]) and a quarter of its weights in each CTA's shared memory by
// TMA, gate/up and down as warp-level bf16 MMAs (h exchanged through the
// cluster's shared memory, rounded to bf16 as on the tensor-core path), then
// w * y added into the tokens' fp32 accumulators (sc.acc set) or the y rows
// written to out_y [R, H].  With fin.ctr set the last CTA rounds the
// accumulators to bf16.
struct SmallFfnArgs {
  const uint16_t* x_perm;   // bf16 [R, H], rows sorted by expert
  const int32_t* offsets;   // [E + 1]
  const uint16_t* w_gate;   // bf16 [E_r, I, H]
  const uint16_t* w_up;     // bf16 [E_r, I, H]
  const uint16_t* w_down;   // bf16 [E_r, H, I]
  ScatterAdd sc;
  float* out_y;
  SmallFinalize fin;
  int H, I, E_r;
  int64_t R;                // rows of x_perm (T * k)
};
// false: a tensor map could not be encoded (nothing launched)
bool launch_small_ffn(const Launch& L, const SmallFfnArgs& a);

}  // namespace moe
