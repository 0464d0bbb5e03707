// route.cu -- top-k gating ("Mira: adaptive caching and predictive expert
// staging for MoE inference", sec. 4.2 Top-K gating; "125B MoE on an RTX 3090
// at 100+ tok/s", sec. 1.1: each token is sent to its top-2 or top-1 experts).
// One warp per token (route_dev.cuh).
#include "kernels.cuh"
#include "ptx.cuh"
#include "route_dev.cuh"

namespace moe {

template <int VPL>   // logits per lane = ceil(E / 32)
__global__ void __launch_bounds__(256) route_topk_kernel(const float* __restrict__ logits, int T,
                                                         int E, int k, int32_t* __restrict__ idx,
                                                         float* __restrict__ w, int* err_clear) {
  griddep_wait();
  griddep_launch_dependents();
  if (err_clear != nullptr && blockIdx.x == 0 && threadIdx.x == 0) *err_clear = 0;
  const int tok = (int)((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
  if (tok >= T) return;
  route_one_token<VPL>(logits, tok, E, k, idx, w, threadIdx.x & 31);
}

cudaError_t launch_route_topk(const float* logits, int T, int E, int k, int32_t* idx, float* w,
                              int* err_clear, cudaStream_t s, bool pdl) {
  const dim3 block(256);
  const dim3 grid((unsigned)((T + 7) / 8));
  if (E <= 32)
    return launch_kernel(route_topk_kernel<1>, grid, block, 0, s, pdl, logits, T, E, k, idx, w, err_clear);
  if (E <= 64)
    return launch_kernel(route_topk_kernel<2>, grid, block, 0, s, pdl, logits, T, E, k, idx, w, err_clear);
  if (E <= 128)
    return launch_kernel(route_topk_kernel<4>, grid, block, 0, s, pdl, logits, T, E, k, idx, w, err_clear);
  return launch_kernel(route_topk_kernel<8>, grid, block, 0, s, pdl, logits, T, E, k, idx, w, err_clear);
}

}  // namespace moe
