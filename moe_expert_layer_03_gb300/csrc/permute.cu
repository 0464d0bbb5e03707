// permute.cu -- regroup the token->expert assignments so every expert's rows are
// contiguous ("125B MoE on an RTX 3090 at 100+ tok/s", sec. 4.2: after routing,
// tokens are reordered by expert id so one grouped GEMM serves each expert).
//
// permute_index_kernel (one CTA of 1024 threads):
//   1. histogram of the A = T*k expert ids (shared-memory atomics),
//   2. exclusive scan -> offsets,
//   3. stable scatter: tiles of 1024 assignments in order; inside a warp the
//      lanes with the same expert find each other with __match_any_sync and
//      take their rank from the lanes below them; across warps a per-warp
//      count table gives each warp its base.  The row of assignment a is
//      offsets[e] + (number of earlier assignments with expert e) -- unique, so
//      the result is independent of scheduling.
// route_gather_kernel (batches of up to FUSED_ROUTE_MAX_T tokens): routing,
//   permutation and the row gather in one launch.  Every CTA routes all tokens
//   (a warp per token, route_dev.cuh) and runs the three steps above on its
//   own copy in shared memory -- a few hundred assignments, cheaper than any
//   hand-off between CTAs -- then gathers its share of the rows; CTA 0 also
//   publishes the routing results.
// gather_rows_kernel: x_perm[r] = x[token_of_row[r]], one warp per row, 16-byte
//   vector loads and stores.
// The gathers release their dependent kernel before their own dependency wait:
// the dependent (a GEMM) only reads their output after its own wait, and its
// large CTAs get their set-up done while the gather waits and runs.
#include "kernels.cuh"
#include "ptx.cuh"
#include "route_dev.cuh"
#include "router_dev.cuh"

namespace moe {

constexpr int PERM_THREADS = 1024;
constexpr int GATHER_UNROLL = 4;   // 16-byte row vectors a lane loads before storing any
constexpr int PERM_MAX_E = 256;

// histogram, scan and stable scatter of the A = T*k expert ids, by one CTA of
// NT threads (which all call it).  The arrays may be global or shared memory.
// err (nullable): the workspace's 1 KB error region, cleared first if `clear`
// (first kernel of the pipeline that reports device errors; the region also
// holds the decode GEMM's ready flags), then the error word ORed with
// MOE_DEVERR_EXPERT_RANGE for an id outside [0, E).
template <int NT>
__device__ __forceinline__ void permute_cta(const int32_t* idx, int T, int k, int E, int t_shared,
                                            int32_t* counts, int32_t* offsets, int32_t* row_of_assign,
                                            int32_t* token_of_row, int* err, bool clear = true) {
  constexpr int NW = NT / 32;
  __shared__ int s_cnt[PERM_MAX_E];
  __shared__ int s_base[PERM_MAX_E];
  __shared__ int s_wc[NW][PERM_MAX_E];
  __shared__ int s_total;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int A = T * k;

  if (err != nullptr && clear)   // the error word and the rest of its 1 KB region (the GEMMs' ready flags)
    for (int i = tid; i < 256; i += NT) err[i] = 0;
  for (int e = tid; e < E; e += NT) s_cnt[e] = 0;
  __syncthreads();
  bool bad = false;
  for (int a = tid; a < A; a += NT) {
    const int e = idx[a];
    if (e < 0 || e >= E)
      bad = true;
    else
      atomicAdd(&s_cnt[e], 1);
  }
  if (bad && err != nullptr) atomicOr(err, MOE_DEVERR_EXPERT_RANGE);
  __syncthreads();

  // exclusive scan by warp 0: lane l owns experts [8l, 8l+8)
  if (warp == 0) {
    int local[8];
    int sum = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int e = lane * 8 + i;
      local[i] = e < E ? s_cnt[e] : 0;
      sum += local[i];
    }
    int incl = sum;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += o;
    }
    int run = incl - sum;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int e = lane * 8 + i;
      if (e < E) {
        s_base[e] = run;
        counts[e] = local[i];
        offsets[e] = run;
      }
      run += local[i];
    }
    if (lane == 31) {
      s_total = incl;
      offsets[E] = incl;
      if (t_shared > 0) offsets[E + 1] = incl + t_shared;
    }
  }
  __syncthreads();

  const unsigned lt_mask = (1u << lane) - 1u;
  for (int base = 0; base < A; base += NT) {
    for (int i = tid; i < NW * E; i += NT) s_wc[i / E][i % E] = 0;
    __syncthreads();
    const int a = base + tid;
    int e = a < A ? idx[a] : -1;
    const bool valid = (e >= 0 && e < E);
    if (!valid) e = -1;
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    const int rank = __popc(peers & lt_mask);
    if (valid && rank == 0) s_wc[warp][e] = __popc(peers);
    __syncthreads();
    if (valid) {
      int r = s_base[e] + rank;
      for (int w = 0; w < warp; ++w) r += s_wc[w][e];
      row_of_assign[a] = r;
      token_of_row[r] = a / k;
    } else if (a < A) {
      row_of_assign[a] = -1;
    }
    __syncthreads();
    for (int ee = tid; ee < E; ee += NT) {
      int s = 0;
      for (int w = 0; w < NW; ++w) s += s_wc[w][ee];
      s_base[ee] += s;
    }
    __syncthreads();
  }
  // rows of the always-on shared expert follow the routed rows, in token order
  for (int t = tid; t < t_shared; t += NT) token_of_row[s_total + t] = t;
}

__global__ void __launch_bounds__(PERM_THREADS, 1)
    permute_index_kernel(const int32_t* __restrict__ idx, int T, int k, int E, int t_shared,
                         int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
                         int32_t* __restrict__ row_of_assign, int32_t* __restrict__ token_of_row,
                         int* __restrict__ err) {
  griddep_wait();
  griddep_launch_dependents();
  permute_cta<PERM_THREADS>(idx, T, k, E, t_shared, counts, offsets, row_of_assign, token_of_row, err);
}

__global__ void __launch_bounds__(256) gather_rows_kernel(const uint16_t* __restrict__ x,
                                                          const int32_t* __restrict__ token_of_row,
                                                          int rows, int T, int d,
                                                          uint16_t* __restrict__ x_perm) {
  griddep_launch_dependents();
  griddep_wait();
  const int lane = threadIdx.x & 31;
  const int nvec = d / 8;   // 16-byte vectors per row
  for (int r = (int)((blockIdx.x * blockDim.x + threadIdx.x) >> 5); r < rows;
       r += (int)((gridDim.x * blockDim.x) >> 5)) {
    const int t = token_of_row[r];
    uint4* dst = reinterpret_cast<uint4*>(x_perm + (size_t)r * d);
    if (t < 0 || t >= T) {   // only after an index error: keep the row defined
      for (int i = lane; i < nvec; i += 32) dst[i] = make_uint4(0, 0, 0, 0);
      continue;
    }
    const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)t * d);
    for (int i0 = lane; i0 < nvec; i0 += 32 * GATHER_UNROLL) {   // loads first: 4 vectors in flight
      uint4 v[GATHER_UNROLL];
#pragma unroll
      for (int u = 0; u < GATHER_UNROLL; ++u)
        if (i0 + 32 * u < nvec) v[u] = __ldg(src + i0 + 32 * u);
#pragma unroll
      for (int u = 0; u < GATHER_UNROLL; ++u)
        if (i0 + 32 * u < nvec) dst[i0 + 32 * u] = v[u];
    }
  }
}

// The quantised prefill GEMMs read fp16 rows scaled by a power of two: the
// row's largest magnitude m goes to [2^13, 2^14), so no element overflows fp16
// and every bf16 element of at least 2^-27 m (fp16's normal range) converts
// exactly (8 significant bits fit fp16's 11).  Returns 2^ex; *inv = 2^-ex.
__device__ __forceinline__ float f16_row_scale(float m, float* inv) {
  int ex = 0;
  if (m > 0.f) frexpf(m, &ex);               // m = f * 2^ex, f in [0.5, 1)
  int sc = m > 0.f ? 14 - ex : 0;            // m * 2^sc in [2^13, 2^14)
  sc = max(-126, min(126, sc));              // 2^sc and 2^-sc both normal fp32
  *inv = __int_as_float((127 - sc) << 23);
  return __int_as_float((127 + sc) << 23);
}
// bf16 pair * mul -> fp16 pair (mul a power of two, no overflow by the choice of mul)
__device__ __forceinline__ uint32_t bf16x2_scaled_f16x2(uint32_t u, float mul) {
  const __half2 h = __floats2half2_rn(__uint_as_float(u << 16) * mul, __uint_as_float(u & 0xFFFF0000u) * mul);
  return *reinterpret_cast<const uint32_t*>(&h);
}
__device__ __forceinline__ float bf16x2_absmax(uint32_t u) {
  return fmaxf(fabsf(__uint_as_float(u << 16)), fabsf(__uint_as_float(u & 0xFFFF0000u)));
}

// One warp per row: the row's largest magnitude, then the scaled fp16 copy.
__global__ void __launch_bounds__(256)
    gather_rows_f16_kernel(const uint16_t* __restrict__ x, const int32_t* __restrict__ token_of_row,
                           int rows, int T, int d, uint16_t* __restrict__ x16, float* __restrict__ xe) {
  griddep_launch_dependents();
  griddep_wait();
  const int lane = threadIdx.x & 31;
  const int nvec = d / 8;
  for (int r = (int)((blockIdx.x * blockDim.x + threadIdx.x) >> 5); r < rows;
       r += (int)((gridDim.x * blockDim.x) >> 5)) {
    const int t = token_of_row != nullptr ? token_of_row[r] : r;   // nullptr: rows in order
    const bool valid = (t >= 0 && t < T);
    uint4* dst = reinterpret_cast<uint4*>(x16 + (size_t)r * d);
    const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)(valid ? t : 0) * d);
    float m = 0.f;
    if (valid)
      for (int i = lane; i < nvec; i += 32) {
        const uint4 v = __ldg(src + i);
        m = fmaxf(m, fmaxf(fmaxf(bf16x2_absmax(v.x), bf16x2_absmax(v.y)),
                           fmaxf(bf16x2_absmax(v.z), bf16x2_absmax(v.w))));
      }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    float inv;
    const float mul = f16_row_scale(m, &inv);
    for (int i0 = lane; i0 < nvec; i0 += 32 * GATHER_UNROLL) {   // loads first: 4 vectors in flight
      uint4 v[GATHER_UNROLL];
#pragma unroll
      for (int u = 0; u < GATHER_UNROLL; ++u) {
        v[u] = make_uint4(0, 0, 0, 0);
        if (valid && i0 + 32 * u < nvec) v[u] = __ldg(src + i0 + 32 * u);
      }
#pragma unroll
      for (int u = 0; u < GATHER_UNROLL; ++u) {
        if (i0 + 32 * u >= nvec) continue;
        dst[i0 + 32 * u] = make_uint4(bf16x2_scaled_f16x2(v[u].x, mul), bf16x2_scaled_f16x2(v[u].y, mul),
                                      bf16x2_scaled_f16x2(v[u].z, mul), bf16x2_scaled_f16x2(v[u].w, mul));
      }
    }
    if (lane == 0) xe[r] = inv;
  }
}

// The quantised decode GEMMs' B operand is e4m3: each gathered row r is
// scaled by a power of two 2^e_r (its largest magnitude m lands in [128, 256))
// and split into hi = e4m3(x 2^e) and lo = e4m3(x 2^e - hi).  For a bf16 x with
// |x 2^e| >= 2^-2 (every element of at least m / 512) the residual x 2^e - hi
// is a multiple of x's bf16 ulp no larger than half an ulp of hi, so it has at
// most 4 significant bits on e4m3's grid and hi + lo == x 2^e exactly; a
// smaller element keeps an absolute error of at most 2^-10 (half the e4m3
// subnormal step), i.e. below 2^-17 m before scaling.  Within every 8-element
// block the elements are stored in the order {0,4,1,5,2,6,3,7}, the K order in
// which the GEMM unpacks the weight nibbles.  Writes xq [2*rows][d] (hi rows,
// then lo rows), xs [d/128][rows] (per-group sums of hi + lo) and xe [rows]
// (2^-e).
// fp8_row: one row by the NT threads of a CTA (src == nullptr: a zero row);
// a half-warp covers one 128-element group.  red: NT/32 floats of shared memory.
template <int NT>
__device__ __forceinline__ void fp8_row(const uint16_t* __restrict__ src, int r, int rows, int d,
                                        uint8_t* __restrict__ xq, float* __restrict__ xs,
                                        float* __restrict__ xe, float* red) {
  constexpr int NW = NT / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nvec = d / 8;   // 8-element blocks per row (a multiple of 16)
  const uint4* vsrc = reinterpret_cast<const uint4*>(src);
  uint4 first = make_uint4(0, 0, 0, 0);   // the thread's first block, kept for the second pass
  float m = 0.f;
  if (src != nullptr)
    for (int i = threadIdx.x; i < nvec; i += NT) {
      const uint4 v = __ldg(vsrc + i);
      if (i == (int)threadIdx.x) first = v;
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int j = 0; j < 4; ++j)
        m = fmaxf(m, fmaxf(fabsf(__uint_as_float(w[j] << 16)), fabsf(__uint_as_float(w[j] & 0xFFFF0000u))));
    }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
  if (lane == 0) red[warp] = m;
  __syncthreads();
  m = red[0];
#pragma unroll
  for (int i = 1; i < NW; ++i) m = fmaxf(m, red[i]);
  __syncthreads();   // red is rewritten for the next row
  int ex = 0;
  if (m > 0.f) frexpf(m, &ex);               // m = f * 2^ex, f in [0.5, 1)
  int sc = m > 0.f ? 8 - ex : 0;             // m * 2^sc in [128, 256)
  sc = max(-126, min(126, sc));              // 2^sc and 2^-sc both normal fp32
  const float mul = __int_as_float((127 + sc) << 23);
  const float inv = __int_as_float((127 - sc) << 23);
  uint8_t* hi_row = xq + (size_t)r * d;
  uint8_t* lo_row = xq + ((size_t)rows + r) * d;
  for (int base = 0; base < nvec; base += NT) {   // every thread runs every iteration
    const int i = base + threadIdx.x;
    const bool act = i < nvec;   // nvec % 16 == 0: whole half-warps
    float sum = 0.f;
    if (act) {
      float f[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      if (src != nullptr) {
        const uint4 v = base == 0 ? first : __ldg(vsrc + i);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          f[2 * j] = __uint_as_float(w[j] << 16) * mul;
          f[2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u) * mul;
        }
      }
      constexpr int PERM[8] = {0, 4, 1, 5, 2, 6, 3, 7};
      uint32_t hw[2] = {0u, 0u}, lw[2] = {0u, 0u};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float a = f[PERM[2 * q]], b = f[PERM[2 * q + 1]];
        const uint16_t h = f32x2_to_e4m3x2(a, b);
        const float2 hf = e4m3x2_to_f32x2(h);
        const uint16_t l = f32x2_to_e4m3x2(a - hf.x, b - hf.y);
        const float2 lf = e4m3x2_to_f32x2(l);
        sum += (hf.x + lf.x) + (hf.y + lf.y);
        hw[q >> 1] |= (uint32_t)h << (16 * (q & 1));
        lw[q >> 1] |= (uint32_t)l << (16 * (q & 1));
      }
      *reinterpret_cast<uint2*>(hi_row + (size_t)i * 8) = make_uint2(hw[0], hw[1]);
      *reinterpret_cast<uint2*>(lo_row + (size_t)i * 8) = make_uint2(lw[0], lw[1]);
    }
#pragma unroll
    for (int off = 8; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
    if (act && (lane & 15) == 0) xs[(size_t)(i >> 4) * rows + r] = sum;
  }
  if (threadIdx.x == 0) xe[r] = inv;
}

// One 128-thread block per row.
constexpr int FP8_GATHER_THREADS = 128;
__global__ void __launch_bounds__(FP8_GATHER_THREADS)
    gather_rows_fp8_kernel(const uint16_t* __restrict__ x, const int32_t* __restrict__ token_of_row,
                           int rows, int T, int d, uint8_t* __restrict__ xq, float* __restrict__ xs,
                           float* __restrict__ xe) {
  griddep_launch_dependents();
  griddep_wait();
  __shared__ float red[FP8_GATHER_THREADS / 32];
  for (int r = blockIdx.x; r < rows; r += gridDim.x) {
    const int t = token_of_row != nullptr ? token_of_row[r] : r;
    const bool valid = (t >= 0 && t < T);
    fp8_row<FP8_GATHER_THREADS>(valid ? x + (size_t)t * d : nullptr, r, rows, d, xq, xs, xe, red);
  }
}

// x_perm row = x row (bf16 copy), by the NT threads of a CTA; src == nullptr: a
// zero row.
template <int NT>
__device__ __forceinline__ void copy_row(const uint16_t* __restrict__ src, int d, uint16_t* __restrict__ dst) {
  const uint4* vs = reinterpret_cast<const uint4*>(src);
  uint4* vd = reinterpret_cast<uint4*>(dst);
  for (int i = threadIdx.x; i < d / 8; i += NT) vd[i] = src != nullptr ? __ldg(vs + i) : make_uint4(0, 0, 0, 0);
}

// The scaled fp16 row of gather_rows_f16_kernel, by the NT threads of a CTA
// (src == nullptr: a zero row); red: NT/32 floats of shared memory.
template <int NT>
__device__ __forceinline__ void f16_row(const uint16_t* __restrict__ src, int d, uint16_t* __restrict__ dst,
                                        float* __restrict__ xe_r, float* red) {
  constexpr int NW = NT / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint4* vs = reinterpret_cast<const uint4*>(src);
  uint4* vd = reinterpret_cast<uint4*>(dst);
  float m = 0.f;
  if (src != nullptr)
    for (int i = threadIdx.x; i < d / 8; i += NT) {
      const uint4 v = __ldg(vs + i);
      m = fmaxf(m, fmaxf(fmaxf(bf16x2_absmax(v.x), bf16x2_absmax(v.y)), fmaxf(bf16x2_absmax(v.z), bf16x2_absmax(v.w))));
    }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
  if (lane == 0) red[warp] = m;
  __syncthreads();
  m = red[0];
#pragma unroll
  for (int i = 1; i < NW; ++i) m = fmaxf(m, red[i]);
  __syncthreads();   // red is rewritten for the next row
  float inv;
  const float mul = f16_row_scale(m, &inv);
  for (int i = threadIdx.x; i < d / 8; i += NT) {
    uint4 o = make_uint4(0, 0, 0, 0);
    if (src != nullptr) {
      const uint4 v = __ldg(vs + i);
      o = make_uint4(bf16x2_scaled_f16x2(v.x, mul), bf16x2_scaled_f16x2(v.y, mul), bf16x2_scaled_f16x2(v.z, mul),
                     bf16x2_scaled_f16x2(v.w, mul));
    }
    vd[i] = o;
  }
  if (threadIdx.x == 0) *xe_r = inv;
}

// ------------------------------------------------------------------ fused
constexpr int RG_THREADS = 512;
constexpr int RG_MAX_A = FUSED_ROUTE_MAX_T * 16;            // T * k, k <= 16
constexpr int RG_MAX_ROWS = RG_MAX_A + FUSED_ROUTE_MAX_T;   // + the shared expert's rows

// Grid-wide barrier of a cooperative launch (every CTA resident): thread 0 of
// each CTA adds one to *ctr (zeroed before the launch, with the error word)
// and waits until all gridDim.x have arrived.  The wait is bounded: past MOE_WAIT_LIMIT_NS it sets
// MOE_DEVERR_TIMEOUT and lets the CTA go on (its results are then invalid, and
// the error word says so).
__device__ __forceinline__ void grid_barrier(int* ctr, int* err) {
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();   // this CTA's writes before its arrival
    atomicAdd(ctr, 1);
    const uint64_t t0 = global_timer_ns();
    while (ld_acquire_gpu(ctr) < (int)gridDim.x) {
      if (global_timer_ns() - t0 > MOE_WAIT_LIMIT_NS) {
        atomicOr(err, MOE_DEVERR_TIMEOUT);
        break;
      }
    }
  }
  __syncthreads();
}

// ROUTER: the router GEMM runs first, in the same launch (a cooperative
// launch: every CTA is resident).  The CTAs' two 256-thread teams compute the
// logit tiles (router_tile, the tiling of the standalone router kernel, so
// the logits are the same bits), write them to `logits`, and after a grid-wide
// barrier every CTA routes from them with L2-coherent loads.
template <int VPL, int OUT, bool ROUTER>
__global__ void __launch_bounds__(RG_THREADS, 1)
    route_gather_kernel(const float* logits, int T, int k, int E, int t_shared,
                        const uint16_t* __restrict__ x, int d, int32_t* __restrict__ idx,
                        float* __restrict__ w, int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
                        int32_t* __restrict__ row_of_assign, int32_t* __restrict__ token_of_row,
                        int* __restrict__ err, GatherDst dst, RouterSrc rsrc) {
  griddep_wait();
  if constexpr (ROUTER) {
    __shared__ float s_rred[2][RT_WARPS][32];
    const int team = threadIdx.x / RT_THREADS, tid = threadIdx.x % RT_THREADS;
    const int ntt = (T + rsrc.tt - 1) / rsrc.tt, eb = (E + RT_EB - 1) / RT_EB;
    for (int gt = (int)blockIdx.x * 2 + team; gt < ntt * eb; gt += (int)gridDim.x * 2)
      router_tile(x, rsrc.w_router, T, d, E, (gt % ntt) * rsrc.tt, rsrc.tt, (gt / ntt) * RT_EB,
                  const_cast<float*>(logits), tid, s_rred[team], 1 + team);
    grid_barrier(rsrc.sync, err);   // every logit written and visible
  }
  griddep_launch_dependents();
  __shared__ int32_t s_idx[RG_MAX_A];
  __shared__ float s_w[RG_MAX_A];
  __shared__ int32_t s_roa[RG_MAX_A];
  __shared__ int32_t s_tor[RG_MAX_ROWS];
  __shared__ int32_t s_counts[PERM_MAX_E];
  __shared__ int32_t s_offsets[PERM_MAX_E + 2];
  __shared__ float s_red[RG_THREADS / 32];
  const int A = T * k, rows = A + t_shared;
  const bool lead = blockIdx.x == 0;
  for (int i = threadIdx.x; i < rows; i += RG_THREADS) s_tor[i] = -1;   // rows of bad ids stay -1
  for (int tok = threadIdx.x >> 5; tok < T; tok += RG_THREADS / 32)
    route_one_token<VPL, ROUTER>(logits, tok, E, k, s_idx, s_w, threadIdx.x & 31);
  __syncthreads();
  // with the router, the error region was zeroed before the launch (the barrier
  // may already have reported into it)
  permute_cta<RG_THREADS>(s_idx, T, k, E, t_shared, s_counts, s_offsets, s_roa, s_tor,
                          lead ? err : nullptr, !ROUTER);
  __syncthreads();
  if (lead) {
    for (int i = threadIdx.x; i < A; i += RG_THREADS) {
      idx[i] = s_idx[i];
      w[i] = s_w[i];
      row_of_assign[i] = s_roa[i];
    }
    for (int i = threadIdx.x; i < rows; i += RG_THREADS) token_of_row[i] = s_tor[i];
    for (int i = threadIdx.x; i < E; i += RG_THREADS) counts[i] = s_counts[i];
    for (int i = threadIdx.x; i <= E + (t_shared > 0 ? 1 : 0); i += RG_THREADS) offsets[i] = s_offsets[i];
  }
  for (int r = blockIdx.x; r < rows; r += gridDim.x) {
    const int t = s_tor[r];
    const uint16_t* src = (t >= 0 && t < T) ? x + (size_t)t * d : nullptr;
    if (OUT == GATHER_FP8)
      fp8_row<RG_THREADS>(src, r, rows, d, dst.xq, dst.xs, dst.xe, s_red);
    else if (OUT == GATHER_F16)
      f16_row<RG_THREADS>(src, d, dst.x16 + (size_t)r * d, dst.xe + r, s_red);
    else
      copy_row<RG_THREADS>(src, d, dst.x16 + (size_t)r * d);
  }
}

cudaError_t launch_permute_index(const int32_t* idx, int T, int k, int E, int t_shared,
                                 int32_t* counts, int32_t* offsets, int32_t* row_of_assign,
                                 int32_t* token_of_row, int* err, cudaStream_t s, bool pdl) {
  return launch_kernel(permute_index_kernel, dim3(1), dim3(PERM_THREADS), 0, s, pdl, idx, T, k, E,
                       t_shared, counts, offsets, row_of_assign, token_of_row, err);
}

template <int VPL, int OUT>
static cudaError_t launch_route_gather_out(dim3 g, cudaStream_t s, bool pdl, const float* logits, int T, int k,
                                           int E, int t_shared, const uint16_t* x, int d, int32_t* idx, float* w,
                                           int32_t* counts, int32_t* offsets, int32_t* roa, int32_t* tor, int* err,
                                           const GatherDst& dst, const RouterSrc* router) {
  const dim3 b(RG_THREADS);
  if (router == nullptr)
    return launch_kernel(route_gather_kernel<VPL, OUT, false>, g, b, 0, s, pdl, logits, T, k, E, t_shared, x, d,
                         idx, w, counts, offsets, roa, tor, err, dst, RouterSrc{});
  // cooperative: the grid-wide barrier needs every CTA resident (grid <= SMs,
  // one 512-thread CTA per SM); the first kernel of its call, so no dependent
  // launch attribute
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = g;
  cfg.blockDim = b;
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, route_gather_kernel<VPL, OUT, true>, logits, T, k, E, t_shared, x, d, idx, w,
                            counts, offsets, roa, tor, err, dst, *router);
}

template <int VPL>
static cudaError_t launch_route_gather_vpl(int out, dim3 g, cudaStream_t s, bool pdl, const float* logits,
                                           int T, int k, int E, int t_shared, const uint16_t* x, int d,
                                           int32_t* idx, float* w, int32_t* counts, int32_t* offsets,
                                           int32_t* roa, int32_t* tor, int* err, const GatherDst& dst,
                                           const RouterSrc* router) {
  if (out == GATHER_FP8)
    return launch_route_gather_out<VPL, GATHER_FP8>(g, s, pdl, logits, T, k, E, t_shared, x, d, idx, w, counts,
                                                    offsets, roa, tor, err, dst, router);
  if (out == GATHER_F16)
    return launch_route_gather_out<VPL, GATHER_F16>(g, s, pdl, logits, T, k, E, t_shared, x, d, idx, w, counts,
                                                    offsets, roa, tor, err, dst, router);
  return launch_route_gather_out<VPL, GATHER_BF16>(g, s, pdl, logits, T, k, E, t_shared, x, d, idx, w, counts,
                                                   offsets, roa, tor, err, dst, router);
}

cudaError_t launch_route_gather(const float* logits, int T, int k, int E, int t_shared, const uint16_t* x,
                                int d, int32_t* idx, float* w, int32_t* counts, int32_t* offsets,
                                int32_t* row_of_assign, int32_t* token_of_row, int* err, int out,
                                const GatherDst& dst, int n_sm, cudaStream_t s, bool pdl, const RouterSrc* router) {
  if (T < 1 || T > FUSED_ROUTE_MAX_T || k < 1 || k > 16 || E < 1 || E > PERM_MAX_E) return cudaErrorInvalidValue;
  const int rows = T * k + t_shared;
  const dim3 g((unsigned)(rows < n_sm ? rows : n_sm));
  if (E <= 32)
    return launch_route_gather_vpl<1>(out, g, s, pdl, logits, T, k, E, t_shared, x, d, idx, w, counts,
                                      offsets, row_of_assign, token_of_row, err, dst, router);
  if (E <= 64)
    return launch_route_gather_vpl<2>(out, g, s, pdl, logits, T, k, E, t_shared, x, d, idx, w, counts,
                                      offsets, row_of_assign, token_of_row, err, dst, router);
  if (E <= 128)
    return launch_route_gather_vpl<4>(out, g, s, pdl, logits, T, k, E, t_shared, x, d, idx, w, counts,
                                      offsets, row_of_assign, token_of_row, err, dst, router);
  return launch_route_gather_vpl<8>(out, g, s, pdl, logits, T, k, E, t_shared, x, d, idx, w, counts,
                                    offsets, row_of_assign, token_of_row, err, dst, router);
}

cudaError_t launch_gather_rows(const uint16_t* x, const int32_t* token_of_row, int rows, int T,
                               int d, uint16_t* x_perm, int n_sm, cudaStream_t s, bool pdl) {
  if (rows <= 0) return cudaSuccess;
  int blocks = (rows + 7) / 8;   // 8 warps (rows) per block
  if (blocks > 4 * n_sm) blocks = 4 * n_sm;
  return launch_kernel(gather_rows_kernel, dim3(blocks), dim3(256), 0, s, pdl, x, token_of_row, rows,
                       T, d, x_perm);
}

cudaError_t launch_gather_rows_f16(const uint16_t* x, const int32_t* token_of_row, int rows, int T,
                                   int d, uint16_t* x16, float* xe, int n_sm, cudaStream_t s, bool pdl) {
  if (rows <= 0) return cudaSuccess;
  int blocks = (rows + 7) / 8;   // 8 warps (rows) per block
  if (blocks > 4 * n_sm) blocks = 4 * n_sm;
  return launch_kernel(gather_rows_f16_kernel, dim3(blocks), dim3(256), 0, s, pdl, x, token_of_row, rows,
                       T, d, x16, xe);
}

__global__ void clear_word_kernel(int* p) { p[threadIdx.x] = 0; }   // 256 words
cudaError_t launch_gather_rows_fp8(const uint16_t* x, const int32_t* token_of_row, int rows, int T,
                                   int d, uint8_t* xq, float* xs, float* xe, int n_sm, cudaStream_t s,
                                   bool pdl) {
  if (rows <= 0) return cudaSuccess;
  const int blocks = rows < 16 * n_sm ? rows : 16 * n_sm;   // one block per row
  return launch_kernel(gather_rows_fp8_kernel, dim3(blocks), dim3(FP8_GATHER_THREADS), 0, s, pdl, x,
                       token_of_row, rows, T, d, xq, xs, xe);
}

cudaError_t launch_clear_word(int* p, cudaStream_t s) {
  clear_word_kernel<<<1, 256, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace moe
