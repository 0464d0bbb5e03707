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
#include "kernels.cuh"
#include "ptx.cuh"

namespace moe {

constexpr int RT_THREADS = 256;
constexpr int RT_WARPS = RT_THREADS / 32;
constexpr int RT_EB = 8;   // experts per CTA
constexpr int RT_TT = 4;   // tokens per CTA, at most
static_assert(RT_EB * RT_TT == 32, "one (token, expert) sum per lane after the warp reduction");

__device__ __forceinline__ void bf16x8_to_f32(const uint4 v, float* f) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

__global__ void __launch_bounds__(RT_THREADS)
    router_logits_kernel(const uint16_t* __restrict__ x, const uint16_t* __restrict__ wr, int T,
                         int d, int E, int tt, float* __restrict__ logits) {
  griddep_wait();
  griddep_launch_dependents();
  __shared__ float red[RT_WARPS][32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int t0 = blockIdx.x * tt, e0 = blockIdx.y * RT_EB;
  const int nt = min(tt, T - t0), ne = min(RT_EB, E - e0);
  const int nv = d / 8;

  float acc[RT_TT * RT_EB];
#pragma unroll
  for (int i = 0; i < RT_TT * RT_EB; ++i) acc[i] = 0.f;
  for (int v = threadIdx.x; v < nv; v += RT_THREADS) {
    float wf[RT_EB][8];
#pragma unroll
    for (int e = 0; e < RT_EB; ++e) {
      const uint4 u = e < ne ? __ldg(reinterpret_cast<const uint4*>(wr + (size_t)(e0 + e) * d) + v)
                             : make_uint4(0, 0, 0, 0);
      bf16x8_to_f32(u, wf[e]);
    }
#pragma unroll
    for (int j = 0; j < RT_TT; ++j) {
      if (j >= nt) break;
      float xf[8];
      bf16x8_to_f32(__ldg(reinterpret_cast<const uint4*>(x + (size_t)(t0 + j) * d) + v), xf);
#pragma unroll
      for (int e = 0; e < RT_EB; ++e)
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[j * RT_EB + e] = fmaf(xf[i], wf[e][i], acc[j * RT_EB + e]);
    }
  }

  // butterfly: at offset o a lane keeps the half of its remaining sums selected
  // by bit o of its lane index and adds its partner's copy of that half; after
  // offsets 16..1 lane l holds the warp's sum l (token l / 8, expert l % 8)
#pragma unroll
  for (int o = 16, n = 32; o > 0; o >>= 1, n >>= 1) {
    const bool up = (lane & o) != 0;
#pragma unroll
    for (int i = 0; i < n / 2; ++i) {
      const float send = up ? acc[i] : acc[i + n / 2];
      const float keep = up ? acc[i + n / 2] : acc[i];
      acc[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
    }
  }
  red[warp][lane] = acc[0];
  __syncthreads();
  if (warp == 0) {
    float s = 0.f;
#pragma unroll
    for (int w = 0; w < RT_WARPS; ++w) s += red[w][lane];
    const int j = lane / RT_EB, e = lane % RT_EB;
    if (j < nt && e < ne) logits[(size_t)(t0 + j) * E + e0 + e] = s;
  }
}

cudaError_t launch_router_logits(const uint16_t* x, const uint16_t* w_router, int T, int d, int E,
                                 float* logits, int n_sm, cudaStream_t s, bool pdl) {
  const int eb = (E + RT_EB - 1) / RT_EB;
  // widest token tile that still gives every SM a CTA (a wider tile reuses each
  // router vector for more tokens)
  int tt = RT_TT;
  while (tt > 1 && (long)((T + tt - 1) / tt) * eb < n_sm) tt >>= 1;
  const dim3 grid((unsigned)((T + tt - 1) / tt), (unsigned)eb);
  return launch_kernel(router_logits_kernel, grid, dim3(RT_THREADS), 0, s, pdl, x, w_router, T, d, E,
                       tt, logits);
}

}  // namespace moe
