/*
 * moe_oracle.h -- plain, slow, fp64 CPU reference of the sparse MoE expert layer.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may include, link or
 * call this file: only the test-suite, the smoke check and the CPU-baseline leg
 * of the benchmark use it.  It shares no code, header, table or helper with the
 * CUDA library under sparse_expert_layer_gb300/.
 *
 * What it computes (the pages print no formula; each step below states the
 * plainest reading of the passages it cites):
 *   router logits -> scores (softmax over every expert, or sigmoid) ->
 *   optional group stage -> top-k -> weights -> stable sort of the picks by
 *   expert -> per-pick SwiGLU expert FFN -> weighted combine (+ zero-computation
 *   experts, + optional always-on shared expert).
 *
 * Sources (web pages; cited by title and section):
 *  [LC-A3]  "基于Atlas 900 A3 SuperPoD的LongCat-Flash模型推理性能优化实践",
 *           section 背景介绍 (zero-computation experts) and
 *           section 优化措施三：权重预取 (Router Matmul, QuantBatchMatmul).
 *  [LC-CANN] "LongCat-Flash与GLM-4.6V，昇腾CANN异构计算深水区突围详解",
 *           section 拆解MoE困局 (768 experts = 512 routed + 256 zero-computation;
 *           token dispatch and combine).
 *  [PANGU]  "华为技术披露集 VOL.12：昇腾×盘古" (Pangu Pro MoE inference system),
 *           opening section (grouped experts, MoGE), section 分层混合并行（H2P）
 *           (grouped routed experts, shared expert) and section SwiftGMM
 *           (grouped matmul switching GEMV/GEMM by load).
 *  [DS-ASC] DeepSeek-V3/R1 on Ascend (Huxiu article), deployment paragraph
 *           (routed experts plus one shared expert per card), section
 *           "2. 模型侧并发优化" (quantised activations travel with their scales)
 *           and section "2. MOE 算子优化" (InitialRouting sorts tokens by expert).
 */
#ifndef MOE_ORACLE_H
#define MOE_ORACLE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { ORC_SOFTMAX = 0, ORC_SIGMOID = 1 };
enum { ORC_BIAS_NONE = 0, ORC_BIAS_LOGIT = 1, ORC_BIAS_SELECT = 2 };

typedef struct {
  int hidden;        /* H */
  int inter;         /* I, routed-expert intermediate size */
  int n_routed;      /* E_r FFN experts, indices 0 .. E_r-1 */
  int n_zero;        /* E_z zero-computation experts, indices E_r .. E_r+E_z-1 */
  int top_k;         /* k */
  int n_group;       /* 1 = no group stage */
  int topk_group;    /* groups kept (group-limited mode, per_group_k == 0) */
  int per_group_k;   /* >0: exactly this many winners in every group (MoGE) */
  int score;         /* ORC_SOFTMAX / ORC_SIGMOID */
  int renormalize;   /* divide the k weights by their sum */
  double routed_scale;
  int bias_mode;     /* ORC_BIAS_* */
  int shared_inter;  /* 0 = no shared expert */
} orc_cfg;

/* Return codes: 0 ok, -1 bad argument. */

/* Router logits l[t,e] = sum_h x[t,h] * Wr[e,h] (+ b[e] when bias_mode is LOGIT).
 * x: bf16 bit patterns [T,H]; w_router: fp32 [E_tot,H]; bias: fp32 [E_tot] or NULL;
 * logits: fp64 [T,E_tot]. */
int orc_router_logits(const orc_cfg* c, int T, const uint16_t* x, const float* w_router,
                      const float* bias, double* logits);

/* Scores, group stage, top-k and weights from logits.
 * ids [T,k] int32 in slot order (descending key, ties to the lower index);
 * weights [T,k] fp64; scores [T,E_tot] fp64 (may be NULL); keys [T,E_tot] fp64
 * selection keys (may be NULL).  Masked experts keep their key in `keys`. */
int orc_select(const orc_cfg* c, int T, const double* logits, const float* bias,
               int32_t* ids, double* weights, double* scores, double* keys);

/* Stable sort of the T*k picks by (expert, token).  counts [E_tot], offsets
 * [E_tot+1], sorted_to_expanded [T*k], expanded_to_sorted [T*k]; expanded index
 * r = t*k + j.  Returns -1 on an out-of-range id. */
int orc_permute(int T, int k, int E_tot, const int32_t* ids, int32_t* counts, int32_t* offsets,
                int32_t* sorted_to_expanded, int32_t* expanded_to_sorted);

/* One SwiGLU expert on one token: g = Wg x, u = Wu x, h = silu(g) * u, y = Wd h.
 * x fp64 [H]; wg, wu bf16 [I,H]; wd bf16 [H,I]; y fp64 [H]; h fp64 [I] or NULL. */
void orc_swiglu_expert(int H, int I, const double* x, const uint16_t* wg, const uint16_t* wu,
                       const uint16_t* wd, double* y, double* h);

/* Whole bf16-weight layer for T tokens.
 * wg/wu/wd: arrays of E_r pointers, one per routed expert ([I,H], [I,H], [H,I]);
 * an entry may be NULL only if no token picks that expert (else -1).
 * sg/su/sd: shared expert ([I_s,H], [I_s,H], [H,I_s]) or NULL when shared_inter == 0.
 * out fp64 [T,H]; ids/weights as in orc_select (may be NULL). */
int orc_layer(const orc_cfg* c, int T, const uint16_t* x, const float* w_router, const float* bias,
              const uint16_t* const* wg, const uint16_t* const* wu, const uint16_t* const* wd,
              const uint16_t* sg, const uint16_t* su, const uint16_t* sd,
              double* out, int32_t* ids, double* weights);

/* ---- W8A8 (int8 weights with per-output-channel scales; per-token dynamic
 *      int8 activations; integer accumulation) ---- */

/* Symmetric per-row quantiser in IEEE fp32: s = amax/127 (fp32 division),
 * q = clamp(round_half_even(v/s), -127, 127); amax == 0 gives s = 0 and q = 0. */
void orc_quantize_rows(int R, int K, const float* v, int8_t* q, float* scale);

/* acc[r,n] = sum_k a[r,k] * w[n,k] in exact integer arithmetic.
 * a int8 [R,K], w int8 [N,K], acc int64 [R,N]. */
void orc_int8_matmul(int R, int N, int K, const int8_t* a, const int8_t* w, int64_t* acc);

/* Whole W8A8 layer.  qg/qu [I,H] int8 with scales sg/su [I]; qd [H,I] int8
 * with scale sd [H]; pointer arrays as in orc_layer.  Shared expert (when
 * shared_inter > 0, else NULL): qsg/qsu [I_s,H] with ssg/ssu [I_s], qsd [H,I_s]
 * with ssd [H]; it takes the token's int8 codes like the routed experts and adds
 * at weight 1.  Optional outputs (NULL to skip): q_x [T,H] int8, s_x [T]. */
int orc_layer_w8a8(const orc_cfg* c, int T, const uint16_t* x, const float* w_router,
                   const float* bias, const int8_t* const* qg, const float* const* sg,
                   const int8_t* const* qu, const float* const* su, const int8_t* const* qd,
                   const float* const* sd, const int8_t* qsg, const float* ssg,
                   const int8_t* qsu, const float* ssu, const int8_t* qsd, const float* ssd,
                   double* out, int32_t* ids, double* weights, int8_t* q_x, float* s_x);

#ifdef __cplusplus
}
#endif
#endif
