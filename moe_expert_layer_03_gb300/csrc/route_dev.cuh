// route_dev.cuh -- the per-token top-k gating step, shared by the routing
// kernel (route.cu) and the fused routing + permutation kernel for small
// batches (permute.cu).  "Mira: adaptive caching and predictive expert staging
// for MoE inference", sec. 4.2 Top-K gating.
//
// One warp routes one token: lane l holds logits l, l+32, ...; k rounds of a
// warp arg-max on the key (value desc, expert index asc) pick the experts in
// descending order; the weights are the softmax over the k selected logits.
#pragma once
#include <math.h>

#include "kernels.cuh"

namespace moe {

template <int VPL>   // logits per lane = ceil(E / 32)
__device__ __forceinline__ void route_one_token(const float* __restrict__ logits, int tok, int E, int k,
                                                int32_t* __restrict__ idx, float* __restrict__ w, int lane) {
  const float* row = logits + (size_t)tok * E;
  float v[VPL];
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
    const int e = lane + 32 * i;
    float x = e < E ? __ldg(row + e) : -INFINITY;
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

}  // namespace moe
