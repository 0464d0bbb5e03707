// route_dev.cuh -- the per-token top-k gating step, shared by the routing
// kernel (route.cu) and the fused routing + permutation kernel for small
// batches (permute.cu).  "Mira: adaptive caching and predictive expert staging
// for MoE inference", sec. 4.2 Top-K gating.
//
// One warp routes one token: lane l holds logits l, l+32, ...; k rounds of a
// warp arg-max on the key (value desc, expert index asc) pick the experts in
// descending order (E <= 32: a shuffle butterfly on the (value, index) pair
// per round; E > 32: a warp max of an order-preserving integer key of the
// value, then a warp min of the expert indices that hold it -- fewer dependent
// steps, measured faster there and slower at E <= 32); the weights are the
// softmax over the k selected logits.
#pragma once
#include <math.h>

#include "kernels.cuh"

namespace moe {

// Order-preserving 32-bit key of a float (larger float -> larger key; -0.0
// is folded into +0.0 first so that equal values give equal keys) and back.
__device__ __forceinline__ uint32_t route_key(float x) {
  const uint32_t u = __float_as_uint(x == 0.f ? 0.f : x);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float route_key_value(uint32_t key) {
  return __uint_as_float((key & 0x80000000u) ? (key & 0x7FFFFFFFu) : ~key);
}

// Logit loads: through the read-only cache, or (COHERENT) from L2, for logits
// written earlier by the same kernel (the fused router, permute.cu).
template <bool COHERENT>
__device__ __forceinline__ float load_logit(const float* p) {
  if constexpr (COHERENT)
    return __ldcg(p);
  else
    return __ldg(p);
}

// E <= 32 (one logit per lane): a shuffle butterfly on (value, index).
template <int VPL, bool COHERENT>
__device__ __forceinline__ void route_one_token_small(const float* __restrict__ logits, int tok, int E,
                                                      int k, int32_t* __restrict__ idx, float* __restrict__ w,
                                                      int lane) {
  const float* row = logits + (size_t)tok * E;
  float v[VPL];
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
    const int e = lane + 32 * i;
    float x = e < E ? load_logit<COHERENT>(row + e) : -INFINITY;
    v[i] = (x != x) ? -INFINITY : x;   // NaN never outranks a number
  }
  uint32_t taken = 0;
  float sel[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    if (j < k) {
      float bv = -INFINITY;
      int bi = 0x7FFFFFFF;
#pragma unroll
      for (int i = 0; i < VPL; ++i) {
        const int e = lane + 32 * i;
        if (e < E && !((taken >> i) & 1u) && (v[i] > bv || (v[i] == bv && e < bi))) {
          bv = v[i];
          bi = e;
        }
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
        if (ov > bv || (ov == bv && oi < bi)) {
          bv = ov;
          bi = oi;
        }
      }
      if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
      sel[j] = bv;
      if (lane == 0) idx[(size_t)tok * k + j] = bi;
    }
  }
  // softmax over the selected logits, max-subtracted, summed in selection order
  const float m = sel[0];
  float den = 0.f;
#pragma unroll
  for (int j = 0; j < 16; ++j)
    if (j < k) den += expf(sel[j] - m);
#pragma unroll
  for (int j = 0; j < 16; ++j)
    if (j < k && lane == j) w[(size_t)tok * k + j] = expf(sel[j] - m) / den;
}

// E > 32: per round two warp reductions on an order-preserving integer key.
template <int VPL, bool COHERENT>
__device__ __forceinline__ void route_one_token_large(const float* __restrict__ logits, int tok, int E,
                                                      int k, int32_t* __restrict__ idx, float* __restrict__ w,
                                                      int lane) {
  const float* row = logits + (size_t)tok * E;
  uint32_t key[VPL];
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
    const int e = lane + 32 * i;
    float x = e < E ? load_logit<COHERENT>(row + e) : -INFINITY;
    key[i] = route_key((x != x) ? -INFINITY : x);   // NaN never outranks a number
  }
  uint32_t taken = 0;
  float sel[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    if (j < k) {
      // my best untaken logit (ties: my lower index, i.e. the first one seen);
      // experts past E have no candidate (key 0 and index INT_MAX never win)
      uint32_t bk = 0;
      int bi = 0x7FFFFFFF;
#pragma unroll
      for (int i = 0; i < VPL; ++i) {
        const int e = lane + 32 * i;
        if (e < E && !((taken >> i) & 1u) && (bi == 0x7FFFFFFF || key[i] > bk)) {
          bk = key[i];
          bi = e;
        }
      }
      // the warp's largest key, then the lowest expert index holding it
      const uint32_t mk = __reduce_max_sync(0xffffffffu, bk);
      const int mi = __reduce_min_sync(0xffffffffu, (bi != 0x7FFFFFFF && bk == mk) ? bi : 0x7FFFFFFF);
      if ((mi & 31) == lane) taken |= 1u << (mi >> 5);
      sel[j] = route_key_value(mk);
      if (lane == 0) idx[(size_t)tok * k + j] = mi;
    }
  }
  // softmax over the selected logits, max-subtracted, summed in selection order
  const float m = sel[0];
  float den = 0.f;
#pragma unroll
  for (int j = 0; j < 16; ++j)
    if (j < k) den += expf(sel[j] - m);
#pragma unroll
  for (int j = 0; j < 16; ++j)
    if (j < k && lane == j) w[(size_t)tok * k + j] = expf(sel[j] - m) / den;
}

template <int VPL, bool COHERENT = false>   // logits per lane = ceil(E / 32)
__device__ __forceinline__ void route_one_token(const float* __restrict__ logits, int tok, int E, int k,
                                                int32_t* __restrict__ idx, float* __restrict__ w, int lane) {
  if constexpr (VPL == 1)
    route_one_token_small<VPL, COHERENT>(logits, tok, E, k, idx, w, lane);
  else
    route_one_token_large<VPL, COHERENT>(logits, tok, E, k, idx, w, lane);
}

}  // namespace moe
