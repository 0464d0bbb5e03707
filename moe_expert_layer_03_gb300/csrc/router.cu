// router.cu -- router logits in front of the top-k gating ("CPU-GPU co-inference
// for MoE models", sec. 2.1: the router runs on the GPU; sec. 5.1: the router
// keeps full precision):
//   logits[t][e] = sum_i x[t][i] * w_router[e][i]
// bf16 inputs, fp32 products and sums.
//
// E <= 256 outputs per token against a router matrix that stays in L2: far too
// narrow for the tensor pipe to pay, so CUDA-core FMAs.  One CTA of 256 threads
// per (tile of up to RT_TT tokens, block of RT_EB = 8 experts).  Thread i owns
// the 16-byte vectors i, i + 256, ... of the K dim: per vector it loads the
// block's 8 router vectors once and uses them for every token of the tile.
// The 32 (token, expert) sums of a thread are reduced across the warp by a
// butterfly that leaves lane l with sum l, then the 8 warps' sums are added in
// warp order from shared memory: a fixed order, so the result does not depend
// on scheduling.
#include "router_dev.cuh"

namespace moe {

__global__ void __launch_bounds__(RT_THREADS)
    router_logits_kernel(const uint16_t* __restrict__ x, const uint16_t* __restrict__ wr, int T,
                         int d, int E, int tt, float* __restrict__ logits) {
  griddep_wait();
  griddep_launch_dependents();
  __shared__ float red[RT_WARPS][32];
  router_tile(x, wr, T, d, E, blockIdx.x * tt, tt, blockIdx.y * RT_EB, logits, threadIdx.x, red, 1);
}

cudaError_t launch_router_logits(const uint16_t* x, const uint16_t* w_router, int T, int d, int E,
                                 float* logits, int n_sm, cudaStream_t s, bool pdl) {
  const int eb = (E + RT_EB - 1) / RT_EB;
  const int tt = router_token_tile(T, E, n_sm);
  const dim3 grid((unsigned)((T + tt - 1) / tt), (unsigned)eb);
  return launch_kernel(router_logits_kernel, grid, dim3(RT_THREADS), 0, s, pdl, x, w_router, T, d, E,
                       tt, logits);
}

}  // namespace moe
