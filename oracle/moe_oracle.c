/*
 * moe_oracle.c -- plain CPU reference of one MoE FFN layer's inference forward.
 *
 * TEST INFRASTRUCTURE ONLY (tests, the smoke check and the bench's CPU baseline).
 * Shares no code, header, table or helper with the CUDA library.  Deliberately
 * slow and literal: every loop is the definition, accumulation is in fp64.
 * Source passages are named in moe_oracle.h and beside each function.
 */
#include "moe_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------ numbers */

double oracle_bf16_to_double(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

double oracle_fp16_to_double(uint16_t h) {
  int s = (h >> 15) & 1, ex = (h >> 10) & 0x1F, man = h & 0x3FF;
  double v;
  if (ex == 0) v = ldexp((double)man, -24);                       /* subnormal */
  else if (ex == 31) v = man ? NAN : INFINITY;
  else v = ldexp(1.0 + (double)man / 1024.0, ex - 15);
  return s ? -v : v;
}

/* OCP 8-bit floating point E4M3: sign, 4 exponent bits (bias 7), 3 mantissa
 * bits; exponent 0 holds the subnormals m/8 * 2^-6; exponent 15 with mantissa 7
 * is NaN (the format has no infinities). */
double oracle_e4m3_to_double(uint8_t b) {
  int s = (b >> 7) & 1, ex = (b >> 3) & 0xF, man = b & 0x7;
  double v;
  if (ex == 15 && man == 7) v = NAN;
  else if (ex == 0) v = ldexp((double)man, -9);                    /* (m/8) * 2^-6 */
  else v = ldexp(1.0 + (double)man / 8.0, ex - 7);
  return s ? -v : v;
}

/* Dequantised weight [row][col].  int4 group-128 ([Strata] sec. 3.1 per-expert
 * scale and zero-point; [CoInf] sec. 5.1 group quantisation):
 *   w = (q - z) * s, q the nibble of element col (low nibble = even col),
 *   s and z the fp16 scale and zero of group col/128 of that row.
 * 8-bit experts ([CoInf] sec. 5.1: 8-bit quantisation of the expert layers
 * only, in groups): w = e4m3(q) * s, q the code byte of element col, s the
 * fp16 scale of group col/128 of that row. */
double oracle_weight(const oracle_matrix* m, int row, int col) {
  if (m->fmt == ORACLE_W_BF16) return oracle_bf16_to_double(m->w[(size_t)row * m->cols + col]);
  if (m->fmt == ORACLE_W_FP8_G128) {   /* 8-bit expert weights: w = e4m3(q) * s */
    double s = oracle_fp16_to_double(m->scale[(size_t)row * (m->cols / 128) + col / 128]);
    return oracle_e4m3_to_double(m->q[(size_t)row * m->cols + col]) * s;
  }
  uint8_t byte = m->q[(size_t)row * (m->cols / 2) + col / 2];
  int q = (col & 1) ? (byte >> 4) : (byte & 0xF);
  size_t g = (size_t)row * (m->cols / 128) + col / 128;
  double s = oracle_fp16_to_double(m->scale[g]);
  double z = oracle_fp16_to_double(m->zero[g]);
  return ((double)q - z) * s;
}

/* ------------------------------------------------------------------ router */

/* Router logits ([CoInf] sec. 2.1, sec. 5.1): the plain dot product of each
 * token row with each expert's router row, in fp64 (a product of two bf16
 * values is exact in fp64, and so is every partial sum up to d = 2^20). */
int oracle_router_logits(const uint16_t* x, const uint16_t* w_router, int T, int d, int E,
                         double* logits) {
  if (!x || !w_router || !logits || T < 0 || d < 1 || E < 1) return -1;
  for (int t = 0; t < T; ++t)
    for (int e = 0; e < E; ++e) {
      double acc = 0.0;
      for (int i = 0; i < d; ++i)
        acc += oracle_bf16_to_double(x[(size_t)t * d + i]) *
               oracle_bf16_to_double(w_router[(size_t)e * d + i]);
      logits[(size_t)t * E + e] = acc;
    }
  return 0;
}

/* ------------------------------------------------------------------ gating */

/* Top-k gating ([Mira] sec. 4.2; [Strata] sec. 1.1): the k largest fp32 logits
 * of each token, lower expert index first among equal logits, listed in
 * descending order; weights are the softmax over the k selected logits. */
int oracle_route_topk(const float* logits, int T, int E, int k, int32_t* idx, float* w) {
  if (!logits || !idx || !w || T < 0 || E < 1 || k < 1 || k > E) return -1;
  char* taken = (char*)malloc((size_t)E);
  if (!taken) return -1;
  for (int t = 0; t < T; ++t) {
    const float* l = logits + (size_t)t * E;
    memset(taken, 0, (size_t)E);
    for (int j = 0; j < k; ++j) {
      int best = -1;
      for (int e = 0; e < E; ++e) {
        if (taken[e]) continue;
        if (best < 0 || l[e] > l[best]) best = e;   /* strict '>' keeps the lower index on ties */
      }
      taken[best] = 1;
      idx[(size_t)t * k + j] = best;
    }
    double lmax = l[idx[(size_t)t * k]];
    double den = 0.0;
    for (int j = 0; j < k; ++j) den += exp((double)l[idx[(size_t)t * k + j]] - lmax);
    for (int j = 0; j < k; ++j)
      w[(size_t)t * k + j] = (float)(exp((double)l[idx[(size_t)t * k + j]] - lmax) / den);
  }
  free(taken);
  return 0;
}

/* ------------------------------------------------------------------ permute */

/* Regroup the assignments a = t*k + j by expert ([Strata] sec. 4.2): counts,
 * exclusive offsets, and the row r = offsets[e] + (number of earlier
 * assignments with the same expert) for every assignment. */
int oracle_permute(const int32_t* idx, int T, int k, int E, int32_t* counts, int32_t* offsets,
                   int32_t* row_of_assign, int32_t* token_of_row) {
  if (!idx || !counts || !offsets || !row_of_assign || !token_of_row || T < 0 || k < 1 || E < 1)
    return -1;
  int A = T * k;
  for (int e = 0; e < E; ++e) counts[e] = 0;
  for (int a = 0; a < A; ++a) {
    if (idx[a] < 0 || idx[a] >= E) return -1;
    counts[idx[a]] += 1;
  }
  offsets[0] = 0;
  for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
  int32_t* fill = (int32_t*)calloc((size_t)E, sizeof(int32_t));
  if (!fill) return -1;
  for (int a = 0; a < A; ++a) {
    int e = idx[a];
    int r = offsets[e] + fill[e];
    fill[e] += 1;
    row_of_assign[a] = r;
    token_of_row[r] = a / k;
  }
  free(fill);
  return 0;
}

/* ------------------------------------------------------------------ expert FFN */

static double silu(double g) { return g / (1.0 + exp(-g)); }

/* SwiGLU two-layer MLP ([Strata] sec. 3.2), no biases:
 *   g_f = sum_c x_c Wg[f][c],  u_f = sum_c x_c Wu[f][c],  h_f = silu(g_f) u_f
 *   y_c = sum_f h_f Wd[c][f] */
int oracle_expert_ffn(const uint16_t* x_row, int d, int F, const oracle_expert* ex,
                      double* h_out, double* y_out) {
  if (!x_row || !ex || !y_out || d < 1 || F < 1) return -1;
  if (ex->gate.rows != F || ex->gate.cols != d || ex->up.rows != F || ex->up.cols != d ||
      ex->down.rows != d || ex->down.cols != F)
    return -1;
  double* x = (double*)malloc(sizeof(double) * (size_t)d);
  double* h = (double*)malloc(sizeof(double) * (size_t)F);
  if (!x || !h) { free(x); free(h); return -1; }
  for (int c = 0; c < d; ++c) x[c] = oracle_bf16_to_double(x_row[c]);
  for (int f = 0; f < F; ++f) {
    double g = 0.0, u = 0.0;
    for (int c = 0; c < d; ++c) {
      g += x[c] * oracle_weight(&ex->gate, f, c);
      u += x[c] * oracle_weight(&ex->up, f, c);
    }
    h[f] = silu(g) * u;
    if (h_out) h_out[f] = h[f];
  }
  for (int c = 0; c < d; ++c) {
    double y = 0.0;
    for (int f = 0; f < F; ++f) y += h[f] * oracle_weight(&ex->down, c, f);
    y_out[c] = y;
  }
  free(x);
  free(h);
  return 0;
}

/* ------------------------------------------------------------------ combine */

/* out_c = sum_{j=0..k-1} w_j * y_j[c]  +  y_shared[c], summed in that order. */
int oracle_combine_row(const uint16_t* const* y_rows, const float* w, int k, int d,
                       const uint16_t* y_shared, double* out) {
  if (!y_rows || !w || !out || k < 1 || d < 1) return -1;
  for (int c = 0; c < d; ++c) {
    double acc = 0.0;
    for (int j = 0; j < k; ++j) acc += (double)w[j] * oracle_bf16_to_double(y_rows[j][c]);
    if (y_shared) acc += oracle_bf16_to_double(y_shared[c]);
    out[c] = acc;
  }
  return 0;
}

/* ------------------------------------------------------------------ layer */

/* out[t] = sum_j w_tj FFN_{e_tj}(x_t) (+ FFN_shared(x_t), weight 1.0; [Strata]
 * sec. 2.1).  Computed token by token from the definition: the regrouping of
 * [Strata] sec. 4.2 moves data but does not change any value. */
int oracle_layer_forward(const uint16_t* x, const float* logits, int T, int E, int k, int d,
                         int F, const oracle_expert* experts, const oracle_expert* shared,
                         const int32_t* token_list, int n_tokens, double* out,
                         int32_t* idx_out, float* w_out) {
  if (!x || !logits || !experts || !out || T < 0 || E < 1 || k < 1 || k > E) return -1;
  int n = token_list ? n_tokens : T;
  int32_t* idx = (int32_t*)malloc(sizeof(int32_t) * (size_t)k);
  float* w = (float*)malloc(sizeof(float) * (size_t)k);
  double* y = (double*)malloc(sizeof(double) * (size_t)d);
  int rc = 0;
  if (!idx || !w || !y) rc = -1;
  for (int i = 0; i < n && rc == 0; ++i) {
    int t = token_list ? token_list[i] : i;
    if (t < 0 || t >= T) { rc = -1; break; }
    double* o = out + (size_t)i * d;
    for (int c = 0; c < d; ++c) o[c] = 0.0;
    rc = oracle_route_topk(logits + (size_t)t * E, 1, E, k, idx, w);
    for (int j = 0; j < k && rc == 0; ++j) {           /* sum_j w_j FFN_{e_j}(x_t), j in order */
      rc = oracle_expert_ffn(x + (size_t)t * d, d, F, &experts[idx[j]], NULL, y);
      for (int c = 0; c < d && rc == 0; ++c) o[c] += (double)w[j] * y[c];
    }
    if (rc == 0 && shared) {                           /* + FFN_shared(x_t), weight 1 */
      rc = oracle_expert_ffn(x + (size_t)t * d, d, F, shared, NULL, y);
      for (int c = 0; c < d && rc == 0; ++c) o[c] += y[c];
    }
    if (rc == 0 && idx_out) memcpy(idx_out + (size_t)i * k, idx, sizeof(int32_t) * (size_t)k);
    if (rc == 0 && w_out) memcpy(w_out + (size_t)i * k, w, sizeof(float) * (size_t)k);
  }
  free(idx); free(w); free(y);
  return rc;
}
