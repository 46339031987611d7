/*
 * moe_oracle.c -- plain fp64 CPU reference of the sparse MoE expert layer.
 *
 * TEST INFRASTRUCTURE ONLY (see moe_oracle.h): used by the test-suite, the
 * smoke check and the benchmark's CPU-baseline leg; never by the product path.
 *
 * Built with: gcc -O2 -fopenmp -fno-fast-math -ffp-contract=off -shared -fPIC
 * so that every floating-point operation is the IEEE operation written here.
 * Loops are written out; there is no blocking, fusion or reordering beyond the
 * definition.  OpenMP splits independent tokens only.
 */
#include "moe_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

static double bf16_to_f64(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

static float bf16_to_f32(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

static int cfg_ok(const orc_cfg* c) {
  if (!c || c->hidden <= 0 || c->n_routed < 0 || c->n_zero < 0 || c->top_k <= 0) return 0;
  int E = c->n_routed + c->n_zero;
  if (E <= 0 || c->top_k > E) return 0;
  if (c->n_routed > 0 && c->inter <= 0) return 0;
  if (c->n_group < 1 || E % c->n_group != 0) return 0;
  if (c->n_group > 1) {
    int G = E / c->n_group;
    if (c->per_group_k > 0) {
      if (c->per_group_k > G || c->per_group_k * c->n_group != c->top_k) return 0;
    } else {
      if (c->topk_group < 1 || c->topk_group > c->n_group) return 0;
      if (c->top_k > c->topk_group * G) return 0;
    }
  }
  return 1;
}

/* Step 1 -- router logits.  The router is a plain matmul of the token row with
 * the router weights ([LC-A3] section 优化措施三 names it "Router Matmul").  A
 * per-expert bias in LOGIT mode is added before scoring, so it moves both the
 * selection and the weights. */
int orc_router_logits(const orc_cfg* c, int T, const uint16_t* x, const float* w_router,
                      const float* bias, double* logits) {
  if (!cfg_ok(c) || T < 0 || (T > 0 && (!x || !w_router || !logits))) return -1;
  if (c->bias_mode != ORC_BIAS_NONE && !bias) return -1;
  const int H = c->hidden, E = c->n_routed + c->n_zero;
#pragma omp parallel for schedule(static)
  for (int t = 0; t < T; ++t) {
    for (int e = 0; e < E; ++e) {
      double s = 0.0;
      for (int h = 0; h < H; ++h)
        s += bf16_to_f64(x[(size_t)t * H + h]) * (double)w_router[(size_t)e * H + h];
      if (c->bias_mode == ORC_BIAS_LOGIT) s += (double)bias[e];
      logits[(size_t)t * E + e] = s;
    }
  }
  return 0;
}

/* Index of the largest key among allowed, not-yet-taken entries of [lo, hi);
 * ties go to the lower index (strict '>' while scanning upwards).  -1 if none. */
static int best_index(int lo, int hi, const double* key, const unsigned char* allowed,
                      const unsigned char* taken) {
  int best = -1;
  for (int e = lo; e < hi; ++e) {
    if ((allowed && !allowed[e]) || (taken && taken[e])) continue;
    if (best < 0 || key[e] > key[best]) best = e;
  }
  return best;
}

/* Steps 2-5 -- scoring, group stage, top-k and weights, per token.
 *  - Scores: softmax over ALL experts including zero-computation ones (the
 *    768-way choice of [LC-CANN] section 拆解MoE困局), or an elementwise sigmoid.
 *  - Group stage ([PANGU] opening section and section H2P: routed experts are
 *    split into groups): groups are contiguous blocks of E/n_group experts.
 *    per_group_k == 0: a group's score is the sum of its two largest keys and
 *    the topk_group best groups stay eligible; per_group_k > 0 (MoGE): exactly
 *    per_group_k winners are taken inside every group.
 *  - Top-k: order eligible experts by (key descending, index ascending); slot j
 *    holds the j-th of that order.
 *  - Weight of a pick: its (unbiased) score; optionally divided by the sum of the
 *    k picked scores; then multiplied by routed_scale. */
int orc_select(const orc_cfg* c, int T, const double* logits, const float* bias, int32_t* ids,
               double* weights, double* scores_out, double* keys_out) {
  if (!cfg_ok(c) || T < 0 || (T > 0 && (!logits || !ids || !weights))) return -1;
  if (c->bias_mode == ORC_BIAS_SELECT && !bias) return -1;
  const int E = c->n_routed + c->n_zero, k = c->top_k;
  int bad = 0;
#pragma omp parallel
  {
    double* s = (double*)malloc(sizeof(double) * E);
    double* key = (double*)malloc(sizeof(double) * E);
    unsigned char* allowed = (unsigned char*)malloc(E);
    unsigned char* taken = (unsigned char*)malloc(E);
    double* gscore = (double*)malloc(sizeof(double) * (c->n_group + 1));
    unsigned char* gkeep = (unsigned char*)malloc(c->n_group + 1);
    unsigned char* gtaken = (unsigned char*)malloc(c->n_group + 1);
#pragma omp for schedule(static)
    for (int t = 0; t < T; ++t) {
      const double* l = logits + (size_t)t * E;
      if (c->score == ORC_SOFTMAX) {
        double m = l[0];
        for (int e = 1; e < E; ++e)
          if (l[e] > m) m = l[e];
        double z = 0.0;
        for (int e = 0; e < E; ++e) z += exp(l[e] - m);
        for (int e = 0; e < E; ++e) s[e] = exp(l[e] - m) / z;
      } else {
        for (int e = 0; e < E; ++e) s[e] = 1.0 / (1.0 + exp(-l[e]));
      }
      for (int e = 0; e < E; ++e)
        key[e] = s[e] + (c->bias_mode == ORC_BIAS_SELECT ? (double)bias[e] : 0.0);

      for (int e = 0; e < E; ++e) allowed[e] = 1;
      if (c->n_group > 1) {
        const int G = E / c->n_group;
        if (c->per_group_k == 0) {
          for (int g = 0; g < c->n_group; ++g) {
            memset(taken, 0, E);
            double sum = 0.0;
            int top = G < 2 ? G : 2;
            for (int i = 0; i < top; ++i) {
              int b = best_index(g * G, (g + 1) * G, key, NULL, taken);
              taken[b] = 1;
              sum += key[b];
            }
            gscore[g] = sum;
          }
          memset(gkeep, 0, c->n_group);
          memset(gtaken, 0, c->n_group);
          for (int i = 0; i < c->topk_group; ++i) {
            int b = best_index(0, c->n_group, gscore, NULL, gtaken);
            gtaken[b] = 1;
            gkeep[b] = 1;
          }
          for (int e = 0; e < E; ++e) allowed[e] = gkeep[e / G];
        } else {
          memset(allowed, 0, E);
          memset(taken, 0, E);
          for (int g = 0; g < c->n_group; ++g)
            for (int i = 0; i < c->per_group_k; ++i) {
              int b = best_index(g * G, (g + 1) * G, key, NULL, taken);
              taken[b] = 1;
              allowed[b] = 1;
            }
        }
      }

      memset(taken, 0, E);
      double wsum = 0.0;
      for (int j = 0; j < k; ++j) {
        int b = best_index(0, E, key, allowed, taken);
        if (b < 0) {
#pragma omp atomic write
          bad = 1;
          b = 0;
        }
        taken[b] = 1;
        ids[(size_t)t * k + j] = b;
        weights[(size_t)t * k + j] = s[b];
        wsum += s[b];
      }
      for (int j = 0; j < k; ++j) {
        double w = weights[(size_t)t * k + j];
        if (c->renormalize) w = w / wsum;
        weights[(size_t)t * k + j] = w * c->routed_scale;
      }
      if (scores_out) memcpy(scores_out + (size_t)t * E, s, sizeof(double) * E);
      if (keys_out) memcpy(keys_out + (size_t)t * E, key, sizeof(double) * E);
    }
    free(s);
    free(key);
    free(allowed);
    free(taken);
    free(gscore);
    free(gkeep);
    free(gtaken);
  }
  return bad ? -1 : 0;
}

/* Step 6 -- InitialRouting-style re-sort of all picks by expert ([DS-ASC]
 * section "2. MOE 算子优化").  A counting sort that visits the expanded index
 * r = t*k + j in increasing order is stable, so within an expert the picks are
 * in token order. */
int orc_permute(int T, int k, int E_tot, const int32_t* ids, int32_t* counts, int32_t* offsets,
                int32_t* sorted_to_expanded, int32_t* expanded_to_sorted) {
  if (T < 0 || k <= 0 || E_tot <= 0) return -1;
  const int R = T * k;
  for (int e = 0; e < E_tot; ++e) counts[e] = 0;
  for (int r = 0; r < R; ++r) {
    if (ids[r] < 0 || ids[r] >= E_tot) return -1;
    counts[ids[r]]++;
  }
  offsets[0] = 0;
  for (int e = 0; e < E_tot; ++e) offsets[e + 1] = offsets[e] + counts[e];
  int32_t* fill = (int32_t*)calloc((size_t)E_tot, sizeof(int32_t));
  for (int r = 0; r < R; ++r) {
    int e = ids[r];
    int p = offsets[e] + fill[e]++;
    sorted_to_expanded[p] = r;
    expanded_to_sorted[r] = p;
  }
  free(fill);
  return 0;
}

static double silu(double g) { return g / (1.0 + exp(-g)); }

/* Step 7 -- one SwiGLU expert ([PANGU] section SwiftGMM: each routed expert is a
 * gate/up/down matmul group): g = Wg x, u = Wu x, h_i = silu(g_i) * u_i, y = Wd h.
 * All in fp64 with no intermediate rounding. */
void orc_swiglu_expert(int H, int I, const double* x, const uint16_t* wg, const uint16_t* wu,
                       const uint16_t* wd, double* y, double* h_out) {
  double* h = h_out ? h_out : (double*)malloc(sizeof(double) * I);
  for (int i = 0; i < I; ++i) {
    double g = 0.0, u = 0.0;
    for (int c = 0; c < H; ++c) {
      g += bf16_to_f64(wg[(size_t)i * H + c]) * x[c];
      u += bf16_to_f64(wu[(size_t)i * H + c]) * x[c];
    }
    h[i] = silu(g) * u;
  }
  for (int c = 0; c < H; ++c) {
    double s = 0.0;
    for (int i = 0; i < I; ++i) s += bf16_to_f64(wd[(size_t)c * I + i]) * h[i];
    y[c] = s;
  }
  if (!h_out) free(h);
}

/* Step 8 -- combine ([LC-CANN] section 拆解MoE困局: results are gathered back to
 * their token).  out[t] = sum_j w_j * (expert output, or x_t unchanged for a
 * zero-computation expert, [LC-A3] section 背景介绍) + shared expert output at
 * weight 1 ([DS-ASC] deployment paragraph: routed experts plus one shared
 * expert).  Slots are summed in slot order, then the shared expert. */
int orc_layer(const orc_cfg* c, int T, const uint16_t* x, const float* w_router, const float* bias,
              const uint16_t* const* wg, const uint16_t* const* wu, const uint16_t* const* wd,
              const uint16_t* sg, const uint16_t* su, const uint16_t* sd, double* out,
              int32_t* ids_out, double* weights_out) {
  if (!cfg_ok(c) || T < 0 || !out) return -1;
  if (c->shared_inter > 0 && (!sg || !su || !sd)) return -1;
  if (T == 0) return 0;
  const int H = c->hidden, I = c->inter, E = c->n_routed + c->n_zero, k = c->top_k;
  double* logits = (double*)malloc(sizeof(double) * (size_t)T * E);
  int32_t* ids = (int32_t*)malloc(sizeof(int32_t) * (size_t)T * k);
  double* w = (double*)malloc(sizeof(double) * (size_t)T * k);
  int rc = orc_router_logits(c, T, x, w_router, bias, logits);
  if (rc == 0) rc = orc_select(c, T, logits, bias, ids, w, NULL, NULL);
  for (size_t r = 0; rc == 0 && r < (size_t)T * k; ++r) {
    int e = ids[r];
    if (e < c->n_routed && (!wg || !wu || !wd || !wg[e] || !wu[e] || !wd[e])) rc = -1;
  }
  if (rc == 0) {
#pragma omp parallel
    {
      double* xt = (double*)malloc(sizeof(double) * H);
      double* y = (double*)malloc(sizeof(double) * H);
      int Imax = I > c->shared_inter ? I : c->shared_inter;
      double* h = (double*)malloc(sizeof(double) * (Imax > 0 ? Imax : 1));
#pragma omp for schedule(dynamic, 1)
      for (int t = 0; t < T; ++t) {
        double* o = out + (size_t)t * H;
        for (int i = 0; i < H; ++i) {
          xt[i] = bf16_to_f64(x[(size_t)t * H + i]);
          o[i] = 0.0;
        }
        for (int j = 0; j < k; ++j) {
          int e = ids[(size_t)t * k + j];
          double wj = w[(size_t)t * k + j];
          if (e < c->n_routed) {
            orc_swiglu_expert(H, I, xt, wg[e], wu[e], wd[e], y, h);
            for (int i = 0; i < H; ++i) o[i] += wj * y[i];
          } else {
            for (int i = 0; i < H; ++i) o[i] += wj * xt[i];
          }
        }
        if (c->shared_inter > 0) {
          orc_swiglu_expert(H, c->shared_inter, xt, sg, su, sd, y, h);
          for (int i = 0; i < H; ++i) o[i] += y[i];
        }
      }
      free(xt);
      free(y);
      free(h);
    }
  }
  if (rc == 0 && ids_out) memcpy(ids_out, ids, sizeof(int32_t) * (size_t)T * k);
  if (rc == 0 && weights_out) memcpy(weights_out, w, sizeof(double) * (size_t)T * k);
  free(logits);
  free(ids);
  free(w);
  return rc;
}

/* ---- W8A8 ----
 * [LC-A3] section 优化措施三 names QuantBatchMatmul for the expert matmuls and
 * [DS-ASC] section "2. 模型侧并发优化" sends quantised activations together with
 * their scales.  Reading taken: symmetric per-row int8 with one fp32 scale per
 * row (token, or token-expert row for the intermediate), +-127, round half to
 * even; integer accumulation; dequantisation acc * s_row * s_channel. */
void orc_quantize_rows(int R, int K, const float* v, int8_t* q, float* scale) {
  for (int r = 0; r < R; ++r) {
    const float* row = v + (size_t)r * K;
    float amax = 0.0f;
    for (int i = 0; i < K; ++i) {
      float a = fabsf(row[i]);
      if (a > amax) amax = a;
    }
    float s = amax / 127.0f;
    scale[r] = s;
    for (int i = 0; i < K; ++i) {
      if (amax == 0.0f) {
        q[(size_t)r * K + i] = 0;
        continue;
      }
      float z = rintf(row[i] / s); /* default rounding mode: to nearest, ties to even */
      if (z > 127.0f) z = 127.0f;
      if (z < -127.0f) z = -127.0f;
      q[(size_t)r * K + i] = (int8_t)z;
    }
  }
}

void orc_int8_matmul(int R, int N, int K, const int8_t* a, const int8_t* w, int64_t* acc) {
#pragma omp parallel for schedule(static)
  for (int r = 0; r < R; ++r)
    for (int n = 0; n < N; ++n) {
      int64_t s = 0;
      for (int i = 0; i < K; ++i)
        s += (int64_t)a[(size_t)r * K + i] * (int64_t)w[(size_t)n * K + i];
      acc[(size_t)r * N + n] = s;
    }
}

/* One W8A8 SwiGLU expert on one token's codes q (scale sx): integer gate and up
 * matmuls, dequantised acc * sx * s_channel in fp64, h = silu(g) * u rounded to
 * fp32 and quantised per row like the token, integer down matmul, dequantised
 * acc * s_h * s_channel.  y fp64 [H]; hf, qh scratch of I entries. */
static void w8a8_expert(int H, int I, const int8_t* q, float sx, const int8_t* qg,
                        const float* sg, const int8_t* qu, const float* su, const int8_t* qd,
                        const float* sd, double* y, float* hf, int8_t* qh) {
  for (int i = 0; i < I; ++i) {
    int64_t ag = 0, au = 0;
    for (int h = 0; h < H; ++h) {
      ag += (int64_t)q[h] * qg[(size_t)i * H + h];
      au += (int64_t)q[h] * qu[(size_t)i * H + h];
    }
    double g = (double)ag * (double)sx * (double)sg[i];
    double u = (double)au * (double)sx * (double)su[i];
    hf[i] = (float)(silu(g) * u);
  }
  float sh;
  orc_quantize_rows(1, I, hf, qh, &sh);
  for (int ch = 0; ch < H; ++ch) {
    int64_t ad = 0;
    for (int i = 0; i < I; ++i) ad += (int64_t)qh[i] * qd[(size_t)ch * I + i];
    y[ch] = (double)ad * (double)sh * (double)sd[ch];
  }
}

/* The shared expert of a W8A8 layer takes the same quantised token codes as the
 * routed experts: [DS-ASC] section "2. 模型侧并发优化" moves the quantisation
 * ahead of the token AllGather, so the MoE layer (shared expert included)
 * receives int8 activations with their scales.  Reading taken: the shared
 * expert is an int8 SwiGLU expert with per-output-channel scales like the
 * routed ones, added at weight 1. */
int orc_layer_w8a8(const orc_cfg* c, int T, const uint16_t* x, const float* w_router,
                   const float* bias, const int8_t* const* qg, const float* const* sg,
                   const int8_t* const* qu, const float* const* su, const int8_t* const* qd,
                   const float* const* sd, const int8_t* qsg, const float* ssg,
                   const int8_t* qsu, const float* ssu, const int8_t* qsd, const float* ssd,
                   double* out, int32_t* ids_out, double* weights_out, int8_t* q_x_out,
                   float* s_x_out) {
  if (!cfg_ok(c) || T < 0 || !out) return -1;
  if (c->shared_inter > 0 && (!qsg || !ssg || !qsu || !ssu || !qsd || !ssd)) return -1;
  if (T == 0) return 0;
  const int H = c->hidden, I = c->inter, E = c->n_routed + c->n_zero, k = c->top_k;
  const int Is = c->shared_inter;
  double* logits = (double*)malloc(sizeof(double) * (size_t)T * E);
  int32_t* ids = (int32_t*)malloc(sizeof(int32_t) * (size_t)T * k);
  double* w = (double*)malloc(sizeof(double) * (size_t)T * k);
  int8_t* qx = (int8_t*)malloc((size_t)T * H);
  float* sx = (float*)malloc(sizeof(float) * (size_t)T);
  int rc = orc_router_logits(c, T, x, w_router, bias, logits);
  if (rc == 0) rc = orc_select(c, T, logits, bias, ids, w, NULL, NULL);
  for (size_t r = 0; rc == 0 && r < (size_t)T * k; ++r) {
    int e = ids[r];
    if (e < c->n_routed &&
        (!qg || !sg || !qu || !su || !qd || !sd || !qg[e] || !sg[e] || !qu[e] || !su[e] ||
         !qd[e] || !sd[e]))
      rc = -1;
  }
  if (rc == 0) {
#pragma omp parallel
    {
      const int Imax = I > Is ? I : Is;
      float* xf = (float*)malloc(sizeof(float) * H);
      float* hf = (float*)malloc(sizeof(float) * (Imax > 0 ? Imax : 1));
      int8_t* qh = (int8_t*)malloc(Imax > 0 ? Imax : 1);
      double* xt = (double*)malloc(sizeof(double) * H);
      double* y = (double*)malloc(sizeof(double) * H);
#pragma omp for schedule(dynamic, 1)
      for (int t = 0; t < T; ++t) {
        for (int i = 0; i < H; ++i) {
          xf[i] = bf16_to_f32(x[(size_t)t * H + i]);
          xt[i] = (double)xf[i];
        }
        orc_quantize_rows(1, H, xf, qx + (size_t)t * H, sx + t);
        const int8_t* q = qx + (size_t)t * H;
        double* o = out + (size_t)t * H;
        for (int i = 0; i < H; ++i) o[i] = 0.0;
        for (int j = 0; j < k; ++j) {
          int e = ids[(size_t)t * k + j];
          double wj = w[(size_t)t * k + j];
          if (e >= c->n_routed) {
            for (int i = 0; i < H; ++i) o[i] += wj * xt[i];
            continue;
          }
          w8a8_expert(H, I, q, sx[t], qg[e], sg[e], qu[e], su[e], qd[e], sd[e], y, hf, qh);
          for (int ch = 0; ch < H; ++ch) o[ch] += wj * y[ch];
        }
        if (Is > 0) {
          w8a8_expert(H, Is, q, sx[t], qsg, ssg, qsu, ssu, qsd, ssd, y, hf, qh);
          for (int ch = 0; ch < H; ++ch) o[ch] += y[ch];
        }
      }
      free(xf);
      free(hf);
      free(qh);
      free(xt);
      free(y);
    }
  }
  if (rc == 0 && ids_out) memcpy(ids_out, ids, sizeof(int32_t) * (size_t)T * k);
  if (rc == 0 && weights_out) memcpy(weights_out, w, sizeof(double) * (size_t)T * k);
  if (rc == 0 && q_x_out) memcpy(q_x_out, qx, (size_t)T * H);
  if (rc == 0 && s_x_out) memcpy(s_x_out, sx, sizeof(float) * (size_t)T);
  free(logits);
  free(ids);
  free(w);
  free(qx);
  free(sx);
  return rc;
}
