// route.cu -- top-k gating ("Mira: adaptive caching and predictive expert
// staging for MoE inference", sec. 4.2 Top-K gating; "125B MoE on an RTX 3090
// at 100+ tok/s", sec. 1.1: each token is sent to its top-2 or top-1 experts).
//
// One warp per token.  Lane l holds logits l, l+32, ...; k rounds of a warp
// arg-max on the key (value desc, expert index asc) pick the experts in
// descending order; the weights are the softmax over the k selected logits.
#include <math.h>

#include "kernels.cuh"
#include "ptx.cuh"

namespace moe {

template <int VPL>   // logits per lane = ceil(E / 32)
__global__ void __launch_bounds__(256) route_topk_kernel(const float* __restrict__ logits, int T,
                                                         int E, int k, int32_t* __restrict__ idx,
                                                         float* __restrict__ w, int* err_clear) {
  if (err_clear != nullptr && blockIdx.x == 0 && threadIdx.x == 0) *err_clear = 0;
  const int tok = (int)((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  if (tok >= T) return;
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

cudaError_t launch_route_topk(const float* logits, int T, int E, int k, int32_t* idx, float* w,
                              int* err_clear, cudaStream_t s) {
  const dim3 block(256);
  const dim3 grid((unsigned)((T + 7) / 8));
  if (E <= 32)
    route_topk_kernel<1><<<grid, block, 0, s>>>(logits, T, E, k, idx, w, err_clear);
  else if (E <= 64)
    route_topk_kernel<2><<<grid, block, 0, s>>>(logits, T, E, k, idx, w, err_clear);
  else if (E <= 128)
    route_topk_kernel<4><<<grid, block, 0, s>>>(logits, T, E, k, idx, w, err_clear);
  else
    route_topk_kernel<8><<<grid, block, 0, s>>>(logits, T, E, k, idx, w, err_clear);
  return cudaGetLastError();
}

}  // namespace moe
