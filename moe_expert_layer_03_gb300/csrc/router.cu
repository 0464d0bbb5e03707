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
#include "router_tc.h"

namespace moe {

__global__ void __launch_bounds__(RT_THREADS)
    router_logits_kernel(const uint16_t* __restrict__ x, const uint16_t* __restrict__ wr, int T,
                         int d, int E, int tt, float* __restrict__ logits) {
  griddep_wait();
  griddep_launch_dependents();
  __shared__ float red[RT_WARPS][32];
  router_tile(x, wr, T, d, E, blockIdx.x * tt, tt, blockIdx.y * RT_EB, logits, threadIdx.x, red, 1);
}

// ------------------------------------------------------------------ tensor-core router (long batches)
// For long batches (T * max(E, 8) >= 8192) of at most 16 experts the router is
// a real (if thin) contraction: D[t][e] = sum_k x[t][k] w[e][k] with M = 128
// token rows per tile and N = 16 (the experts, the router tile's rows past E
// read as zeros by the TMA).  One thread-block cluster of RTC_SPLIT CTAs per
// 128-token tile, CTA r taking the r-th slice of K: TMA loads of the x tile (128 rows x 64
// K, 128-byte swizzle) and the router tile (16 rows x 64 K) through a ring of
// stages, tcgen05.mma kind::f16 (bf16 x bf16 -> fp32) into four accumulators
// of 16 TMEM columns (the 4 MMAs of one 64-wide K step go to different ones, so
// they do not wait on each other), added in a fixed order at the end.
// Then a reduce-scatter over distributed shared memory: CTA r owns the tile's
// token rows [16r, 16r + 16), every CTA sends its partial sums of those rows to
// CTA r with asynchronous remote stores that count their bytes on CTA r's
// mbarrier, and CTA r adds the eight slices in rank order (deterministic) and
// writes the logits of its rows.  Every CTA receives 7 x 16 rows, so no one
// SM's shared-memory port carries the whole tile.  Nothing is allocated.  Every
// wait is bounded; a CTA whose pipeline wait runs out contributes NaN, so the
// tile's logits come out NaN (and the error word, when given, gets
// MOE_DEVERR_TIMEOUT).  About 100 KB of shared memory, so two CTAs can share an
// SM (with ~210 KB per CTA a 2048-token launch, 16 clusters, ran in two waves;
// now its CTAs start within ~0.7 us of each other).
constexpr int RTC_M = 128;        // token rows per tile (the MMA's M)
constexpr int RTC_N = 16;         // experts per tile (the MMA's N)
constexpr int RTC_SPLIT = 8;      // CTAs per cluster = K slices per tile
constexpr int RTC_ST = 5;         // ring stages
constexpr int RTC_NACC = 4;       // accumulators: the 4 MMAs of a K step are independent
constexpr int RTC_ROWS = RTC_M / RTC_SPLIT;   // token rows each CTA reduces and writes
constexpr int RTC_LD = RTC_N + 4; // floats per row of the receive buffer (padded: conflict-free 16-byte reads)
constexpr uint32_t RTC_A_BYTES = RTC_M * 128;   // one 64-wide K step of the x tile
constexpr uint32_t RTC_B_BYTES = RTC_N * 128;   // one 64-wide K step of the router tile
constexpr uint32_t RTC_STAGE = RTC_A_BYTES + RTC_B_BYTES;
constexpr size_t RTC_SMEM = 1024 + (size_t)RTC_ST * RTC_STAGE + (size_t)RTC_SPLIT * RTC_ROWS * RTC_LD * 4 + 256;
static_assert(RTC_ST * 2 + 2 <= 30, "barriers and the TMEM slot fit the 256-byte tail");

__device__ __forceinline__ bool rtc_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait_sleep(bar, parity))
    if (global_timer_ns() - t0 > limit_ns) return false;
  return true;
}

__global__ void __cluster_dims__(1, RTC_SPLIT, 1) __launch_bounds__(128, 2)
    router_tc_kernel(const __grid_constant__ CUtensorMap tx, const __grid_constant__ CUtensorMap tw, int T, int d,
                     int E, float* __restrict__ logits, int k, int32_t* __restrict__ idx, float* __restrict__ w,
                     int* err, int stop_stage, uint64_t wait_ns) {
  extern __shared__ uint8_t smem_dyn[];
  const uint32_t pad = (1024u - (smem_u32(smem_dyn) & 1023u)) & 1023u;
  uint8_t* base = smem_dyn + pad;
  float* red = reinterpret_cast<float*>(base + (size_t)RTC_ST * RTC_STAGE);   // [RTC_SPLIT][RTC_ROWS][RTC_LD]
  uint64_t* full = reinterpret_cast<uint64_t*>(red + RTC_SPLIT * RTC_ROWS * RTC_LD);
  uint64_t* empty = full + RTC_ST;
  uint64_t* done = empty + RTC_ST;
  uint64_t* recv = done + 1;   // the slices' partial sums of this CTA's rows have landed
  uint32_t* tslot = reinterpret_cast<uint32_t*>(recv + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tile = blockIdx.x, rank = blockIdx.y;   // rank = this CTA's K slice (and its cluster rank)
  const int ksteps = d / 64;
  const int k0 = (int)((long long)rank * ksteps / RTC_SPLIT), k1 = (int)((long long)(rank + 1) * ksteps / RTC_SPLIT);
  const int nk = k1 - k0;

  // producer (thread 0): the slice's next K step into ring stage `issued % RTC_ST`
  int issued = 0;
  auto issue = [&]() {
    const int st = issued % RTC_ST;
    const uint32_t bar = smem_u32(&full[st]);
    mbar_arrive_expect_tx(bar, RTC_STAGE);
    const uint32_t a = smem_u32(base + (size_t)st * RTC_STAGE);
    tma_load_2d(a, &tx, (k0 + issued) * 64, tile * RTC_M, bar);
    tma_load_2d(a + RTC_A_BYTES, &tw, (k0 + issued) * 64, 0, bar);
    ++issued;
  };
  if (threadIdx.x == 0) {
    prefetch_tensormap(&tx);   // the descriptors' fetch overlaps the set-up
    prefetch_tensormap(&tw);
    for (int i = 0; i < RTC_ST; ++i) {
      mbar_init(smem_u32(&full[i]), 1);
      mbar_init(smem_u32(&empty[i]), 1);
    }
    mbar_init(smem_u32(done), 1);
    mbar_init(smem_u32(recv), 1);
    fence_mbar_init();
    // every slice sends its 16 rows x ceil(E / 4) 16-byte vectors
    mbar_arrive_expect_tx(smem_u32(recv), (uint32_t)(RTC_SPLIT * RTC_ROWS * ((min(E, RTC_N) + 3) / 4) * 16));
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tslot), RTC_NACC * RTC_N);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // every CTA of the cluster running before any writes into another's shared memory
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
  const uint32_t tmem = *tslot;
  bool ok = true;

  if (warp == 0 && lane == 0) {   // producer: the slice's K steps through the ring
    griddep_wait();
    while (issued < nk) {
      if (issued == stop_stage) break;   // fault-injection hook (off: -1): leave the pipeline starved
      if (issued >= RTC_ST &&
          !(ok = rtc_wait(smem_u32(&empty[issued % RTC_ST]), (uint32_t)(((issued / RTC_ST) - 1) & 1), wait_ns)))
        break;
      issue();
    }
    // every copy still in flight lands before the CTA may exit (bounded)
    for (int i = issued > RTC_ST ? issued - RTC_ST : 0; i < issued; ++i)
      rtc_wait(smem_u32(&full[i % RTC_ST]), (uint32_t)((i / RTC_ST) & 1), wait_ns);
  } else if (warp == 1) {   // MMA issuer (converged warp, one elected lane issues)
    const uint32_t idesc = idesc_f16kind_f32(RTC_M, RTC_N, 1u);
    for (int i = 0; i < nk && ok; ++i) {
      const int st = i % RTC_ST;
      if (!(ok = __all_sync(0xffffffffu, rtc_wait(smem_u32(&full[st]), (uint32_t)((i / RTC_ST) & 1), wait_ns))))
        break;
      tc_fence_after();
      const uint64_t ad = sdesc_kmajor_sw128(smem_u32(base + (size_t)st * RTC_STAGE));
      const uint64_t bd = sdesc_kmajor_sw128(smem_u32(base + (size_t)st * RTC_STAGE + RTC_A_BYTES));
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)   // K = 16 per MMA (+32 bytes inside the swizzle atom), accumulator kk
        mma_ss_elect(tmem + kk * RTC_N, ad + (uint64_t)((kk * 32) >> 4), bd + (uint64_t)((kk * 32) >> 4), idesc,
                     i > 0 ? 1u : 0u);
      mma_commit_elect(smem_u32(&empty[st]));
    }
    mma_commit_elect(smem_u32(done));   // after every MMA issued here (none: arrives at once)
  }
  // every thread: this CTA's partial sums of its token row (TMEM lane = row)
  __syncwarp();
  const bool got = rtc_wait(smem_u32(done), 0u, wait_ns);
  tc_fence_after();
  uint32_t v[16], v1[16], v2[16], v3[16];
  const uint32_t trow = tmem + ((uint32_t)(warp * 32) << 16);
  tmem_ld_16(trow, v);
  tmem_ld_16(trow + RTC_N, v1);
  tmem_ld_16(trow + 2 * RTC_N, v2);
  tmem_ld_16(trow + 3 * RTC_N, v3);
  tmem_ld_wait();
#pragma unroll
  for (int c = 0; c < 16; ++c)   // the four accumulators, in a fixed order
    v[c] = __float_as_uint(((__uint_as_float(v[c]) + __uint_as_float(v1[c])) + __uint_as_float(v2[c])) +
                           __uint_as_float(v3[c]));
  const bool good = __syncthreads_and(ok && got);
  asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
  // row m of the tile to CTA m / RTC_ROWS: red[rank][m % RTC_ROWS][0..E)
  {
    const int owner = (int)threadIdx.x / RTC_ROWS;
    const uint32_t local = smem_u32(red + ((size_t)rank * RTC_ROWS + (threadIdx.x % RTC_ROWS)) * RTC_LD);
    uint32_t remote, rbar;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local), "r"(owner));
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(rbar) : "r"(smem_u32(recv)), "r"(owner));
#pragma unroll
    for (int j = 0; j < RTC_N; j += 4) {
      if (j >= E) break;
      float f[4];
#pragma unroll
      for (int q = 0; q < 4; ++q)
        f[q] = (nk > 0 && good) ? __uint_as_float(v[j + q]) : (good ? 0.f : __int_as_float(0x7FC00000));
      asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(
                       remote + j * 4),
                   "f"(f[0]), "f"(f[1]), "f"(f[2]), "f"(f[3]), "r"(rbar)
                   : "memory");
    }
  }
  // no CTA leaves before every store into its shared memory has landed (second phase, waited for at the end)
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
  const bool in = rtc_wait(smem_u32(recv), 0u, wait_ns);
  if ((!good || !in) && err != nullptr && threadIdx.x == 0) atomicOr(err, MOE_DEVERR_TIMEOUT);
  griddep_launch_dependents();
  // this CTA's rows: thread (row, group of 4 experts) adds the slices in rank order
  if (threadIdx.x < RTC_ROWS * (RTC_N / 4)) {   // warps 0 and 1, whole: the top-k below shuffles
    const int jg = (int)threadIdx.x % (RTC_N / 4);
    const int row = (int)threadIdx.x / (RTC_N / 4), j = jg * 4;
    const int t = tile * RTC_M + rank * RTC_ROWS + row;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (j < E) {
#pragma unroll
      for (int r = 0; r < RTC_SPLIT; ++r) {
        const float4 q = *reinterpret_cast<const float4*>(red + ((size_t)r * RTC_ROWS + row) * RTC_LD + j);
        acc.x += q.x;
        acc.y += q.y;
        acc.z += q.z;
        acc.w += q.w;
      }
    }
    if (!in) acc = make_float4(__int_as_float(0x7FC00000), __int_as_float(0x7FC00000), __int_as_float(0x7FC00000),
                               __int_as_float(0x7FC00000));
    if (t < T && j < E) {
      float* out = logits + (size_t)t * E + j;
      if ((E & 3) == 0) {   // 16-byte aligned (the logits buffer is)
        *reinterpret_cast<float4*>(out) = acc;
      } else {
        const float q[4] = {acc.x, acc.y, acc.z, acc.w};
#pragma unroll
        for (int c = 0; c < 4; ++c)
          if (j + c < E) out[c] = q[c];
      }
    }
    if (idx != nullptr) {
      // top-k gating of the row (the same selection and softmax as the routing
      // kernels, so the same bits): the row's 4 threads hold experts j..j+3;
      // k rounds of an arg-max on (value desc, index asc) over the 4 lanes,
      // NaN ranked below every number; weights = softmax over the selected
      // logits, max-subtracted, summed in selection order
      float v[4] = {acc.x, acc.y, acc.z, acc.w};
#pragma unroll
      for (int q = 0; q < 4; ++q)
        if (v[q] != v[q]) v[q] = -INFINITY;
      uint32_t taken = 0;
      float sel[RTC_N];
#pragma unroll
      for (int sx = 0; sx < RTC_N; ++sx) {
        if (sx < k) {
          float bv = -INFINITY;
          int bi = 0x7FFFFFFF;
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int e = j + q;
            if (e < E && !((taken >> q) & 1u) && (v[q] > bv || (v[q] == bv && e < bi))) {
              bv = v[q];
              bi = e;
            }
          }
#pragma unroll
          for (int off = 1; off < 4; off <<= 1) {   // within the row's 4 lanes
            const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
            if (ov > bv || (ov == bv && oi < bi)) {
              bv = ov;
              bi = oi;
            }
          }
          if ((bi >> 2) == jg) taken |= 1u << (bi & 3);
          sel[sx] = bv;
          if (jg == 0 && t < T) idx[(size_t)t * k + sx] = bi;
        }
      }
      if (jg == 0 && t < T) {
        const float m = sel[0];
        float den = 0.f;
#pragma unroll
        for (int sx = 0; sx < RTC_N; ++sx)
          if (sx < k) den += expf(sel[sx] - m);
#pragma unroll
        for (int sx = 0; sx < RTC_N; ++sx)
          if (sx < k) w[(size_t)t * k + sx] = expf(sel[sx] - m) / den;
      }
    }
  }
  asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, RTC_NACC * RTC_N);
}

// Measured on GB300 (d = 4096, launches in a CUDA graph): the tensor-core
// kernel costs ~4.5 us at any T up to ~1000 tokens (its K slices are bound by
// shared-memory traffic: every x byte written by the TMA, then read by the
// MMA), the CUDA-core kernel grows with T * max(E, 8); they cross near
// T * max(E, 8) = 8192 (E = 8: 1024 tokens, 5.1 vs 4.6 us; E = 16: 512).
bool router_uses_tensor_cores(int T, int d, int E) {
  return E <= RTC_N && d % 64 == 0 && (long long)T * (E > 8 ? E : 8) >= 8192;
}

cudaError_t launch_router_topk_tc(const CUtensorMap& tx, const CUtensorMap& tw, int T, int d, int E, float* logits,
                                  int k, int32_t* idx, float* w, int* err, int stop_stage, uint64_t wait_ns,
                                  cudaStream_t s, bool pdl) {
  static bool attr_set = false;   // benign race: every caller sets the same value
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(router_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)RTC_SMEM);
    // the whole unified L1 as shared memory, so that two CTAs fit on an SM
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(router_tc_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                               (int)cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  return launch_kernel(router_tc_kernel, dim3((unsigned)((T + RTC_M - 1) / RTC_M), RTC_SPLIT), dim3(128), RTC_SMEM,
                       s, pdl, tx, tw, T, d, E, logits, k, idx, w, err, stop_stage, wait_ns);
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
