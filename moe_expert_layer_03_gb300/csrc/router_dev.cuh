// router_dev.cuh -- the router-logit tile shared by the router GEMM kernel
// (router.cu) and the fused routing kernel for small batches (permute.cu):
//   logits[t][e] = sum_i x[t][i] * w_router[e][i], bf16 inputs, fp32 sums
// ("CPU-GPU co-inference for MoE models", sec. 2.1: the router runs on the GPU;
// sec. 5.1: the router keeps full precision).
#pragma once
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


// One (token tile, expert block) of logits by a team of RT_THREADS threads
// (tid = the thread's index in the team, red = the team's RT_WARPS x 32 floats
// of shared memory, bar_id = a named barrier the team alone uses).  The sum
// order of a logit depends only on d and on the token's position in its tile,
// so the standalone kernel and the fused routing kernel (permute.cu), which
// tile the tokens the same way, give the same bits.
__device__ __forceinline__ void router_tile(const uint16_t* __restrict__ x, const uint16_t* __restrict__ wr,
                                            int T, int d, int E, int t0, int tt, int e0,
                                            float* __restrict__ logits, int tid, float (*red)[32],
                                            uint32_t bar_id) {
  const int lane = tid & 31, warp = tid >> 5;
  const int nt = min(tt, T - t0), ne = min(RT_EB, E - e0);
  const int nv = d / 8;

  float acc[RT_TT * RT_EB];
#pragma unroll
  for (int i = 0; i < RT_TT * RT_EB; ++i) acc[i] = 0.f;
  for (int v = tid; v < nv; v += RT_THREADS) {
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
  named_barrier(bar_id, RT_THREADS);
  if (warp == 0) {
    float s = 0.f;
#pragma unroll
    for (int w = 0; w < RT_WARPS; ++w) s += red[w][lane];
    const int j = lane / RT_EB, e = lane % RT_EB;
    if (j < nt && e < ne) logits[(size_t)(t0 + j) * E + e0 + e] = s;
  }
  named_barrier(bar_id, RT_THREADS);   // red is reused by the team's next tile
}

inline int router_token_tile(int T, int E, int n_sm) {
  const int eb = (E + RT_EB - 1) / RT_EB;
  // widest token tile that still gives every SM a CTA (a wider tile reuses each
  // router vector for more tokens)
  int tt = RT_TT;
  while (tt > 1 && (long)((T + tt - 1) / tt) * eb < n_sm) tt >>= 1;
  return tt;
}

}  // namespace moe
