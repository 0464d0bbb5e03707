/*
 * moe_oracle.h -- plain CPU reference of one MoE FFN layer's inference forward.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or call
 * this code; it exists so tests, the smoke check and the CPU baseline of the
 * bench can compare the CUDA path against an obviously-correct definition.
 *
 * Sources (page title, section):
 *   [Mira]   "Mira: adaptive caching and predictive expert staging for MoE
 *            inference" (gsyq.cn/news/338825), sec. 2.1 (8 experts, 2 active),
 *            sec. 4.2 (Top-K gating).
 *   [CoInf]  "CPU-GPU co-inference for MoE models" (maplevalley.com.cn/news/2111104),
 *            sec. 2.1 (router on the GPU), sec. 5.1 (group quantisation; router
 *            kept at full precision).
 *   [Strata] "125B MoE on an RTX 3090 at 100+ tok/s: a full-stack inference
 *            optimisation log" (bjdmk.com.cn/news/6009460), sec. 1.1 (top-2 /
 *            top-1 routing), sec. 2.1 (shared expert always resident), sec. 3.1
 *            (per-expert int4 scale and zero-point), sec. 3.2 (expert FFN is a
 *            two-layer MLP; grouped GEMM), sec. 4.2 (regroup tokens by expert).
 *
 * Types: bf16 and fp16 values are passed as their raw 16-bit patterns (uint16_t).
 * All arithmetic is fp64 and nothing is rounded on the way: the results are the
 * exact layer math on the given bf16 inputs and weights (the routing weights
 * are returned as fp32, the type they are stored in).  The CUDA path's bf16
 * intermediates are approximations judged against these values.
 */
#ifndef MOE_ORACLE_H
#define MOE_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { ORACLE_W_BF16 = 0, ORACLE_W_INT4_G128 = 1, ORACLE_W_FP8_G128 = 2 };

/* One weight matrix [rows][cols], cols = K contiguous ("[out][in]"). */
typedef struct {
  int fmt;                 /* ORACLE_W_BF16, ORACLE_W_INT4_G128 or ORACLE_W_FP8_G128 */
  int rows, cols;
  const uint16_t* w;       /* bf16 [rows][cols]                          (fmt 0) */
  const uint8_t* q;        /* fmt 1: packed [rows][cols/2], low nibble = even col;
                              fmt 2: e4m3 codes [rows][cols] */
  const uint16_t* scale;   /* fp16 [rows][cols/128]                      (fmt 1, 2) */
  const uint16_t* zero;    /* fp16 [rows][cols/128], integer values 0..15 (fmt 1) */
} oracle_matrix;

/* One expert: gate, up [F][d]; down [d][F]. */
typedef struct {
  oracle_matrix gate, up, down;
} oracle_expert;

/* Number helpers (exposed so tests can pin them against independent code). */
double oracle_bf16_to_double(uint16_t b);
double oracle_fp16_to_double(uint16_t h);
double oracle_e4m3_to_double(uint8_t b);   /* OCP fp8 E4M3 (bias 7, no infinities; S.1111.111 = NaN) */
double oracle_weight(const oracle_matrix* m, int row, int col);   /* dequantised value */

/* Router logits ([CoInf] sec. 2.1 router resident on the GPU; sec. 5.1 router
 * kept at full precision): logits[t][e] = sum_i x[t][i] * w_router[e][i] for
 * bf16 x [T][d] and w_router [E][d] (both row-major, the input dim contiguous),
 * summed exactly in fp64.  Returns 0, or -1 on bad args. */
int oracle_router_logits(const uint16_t* x, const uint16_t* w_router, int T, int d, int E,
                         double* logits /* [T][E] */);

/* Top-k gating: idx [T][k] int32, w [T][k] fp32.  Returns 0, or -1 on bad args. */
int oracle_route_topk(const float* logits, int T, int E, int k, int32_t* idx, float* w);

/* Histogram, exclusive scan and stable scatter of the T*k assignments. */
int oracle_permute(const int32_t* idx, int T, int k, int E, int32_t* counts,
                   int32_t* offsets /* E+1 */, int32_t* row_of_assign /* T*k */,
                   int32_t* token_of_row /* T*k */);

/* SwiGLU expert FFN of one token row: h = silu(x Wg^T) * (x Wu^T) [F],
 * y = h Wd^T [d].  h_out may be NULL. */
int oracle_expert_ffn(const uint16_t* x_row, int d, int F, const oracle_expert* ex,
                      double* h_out, double* y_out);

/* Weighted combine of one token from bf16 expert outputs:
 * out = sum_j w[j] * y_j + y_shared. */
int oracle_combine_row(const uint16_t* const* y_rows, const float* w, int k, int d,
                       const uint16_t* y_shared /* nullable */, double* out);

/* Whole layer for the listed tokens (all T when token_list == NULL):
 * out [n][d], and per listed token its idx/w [n][k] (nullable). */
int oracle_layer_forward(const uint16_t* x, const float* logits, int T, int E, int k, int d,
                         int F, const oracle_expert* experts /* E */,
                         const oracle_expert* shared /* nullable, same d and F */,
                         const int32_t* token_list, int n_tokens, double* out,
                         int32_t* idx_out, float* w_out);

#ifdef __cplusplus
}
#endif
#endif
