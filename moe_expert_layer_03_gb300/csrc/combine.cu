// combine.cu -- weighted un-permute back to token order:
//   out[t] = bf16( sum_{j<k} w[t][j] * y[row_of_assign[t*k+j]]  (+ y_shared[t]) )
// summed in fp32 in the order j = 0..k-1, the always-on shared expert last
// ("125B MoE on an RTX 3090 at 100+ tok/s": sec. 4.2 regroup and back, sec. 2.1
// shared expert).  The partial-sum variant (whole-layer path) adds the fp32
// K-split partial sums of each expert output and uses them unrounded; the bf16
// variant reads the bf16 y_perm of the standalone grouped-FFN entry point.
//
// One CTA per (token, column slab); each thread owns 4 consecutive columns
// (16-byte fp32 / 8-byte bf16 vectors) per vector: one vector (1024-column
// slabs) for batches up to 256 tokens, two (2048-column slabs, twice the loads
// in flight per thread) above.
#include "kernels.cuh"
#include "ptx.cuh"

namespace moe {

__device__ __forceinline__ float4 load_bf16x4(const uint16_t* p) {
  const uint2 u = *reinterpret_cast<const uint2*>(p);
  float4 r;
  r.x = __uint_as_float(u.x << 16);
  r.y = __uint_as_float(u.x & 0xFFFF0000u);
  r.z = __uint_as_float(u.y << 16);
  r.w = __uint_as_float(u.y & 0xFFFF0000u);
  return r;
}

__device__ __forceinline__ void store_bf16x4(uint16_t* p, float4 v) {
  __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y);
  __nv_bfloat162 b = __floats2bfloat162_rn(v.z, v.w);
  uint2 u;
  u.x = *reinterpret_cast<uint32_t*>(&a);
  u.y = *reinterpret_cast<uint32_t*>(&b);
  *reinterpret_cast<uint2*>(p) = u;
}

// sum over K splits of the fp32 partial sums of row r, columns [c, c+4), in
// split order.  OVERLAP (small batches, latency-bound): the loads of all
// splits are issued before the first add so their latencies overlap; else a
// plain loop (large batches are bandwidth-bound and keep more threads busy).
template <bool OVERLAP>
__device__ __forceinline__ float4 y_from_partials(const float* part, int n_split,
                                                  size_t split_stride, int r, int d, int c) {
  if (!OVERLAP) {
    float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int i = 0; i < n_split; ++i) {
      const float4 v = __ldg(reinterpret_cast<const float4*>(part + i * split_stride + (size_t)r * d + c));
      s.x += v.x;
      s.y += v.y;
      s.z += v.z;
      s.w += v.w;
    }
    return s;
  }
  constexpr int MAXS = 8;   // the largest K split (abi.cu)
  float4 v[MAXS];
#pragma unroll
  for (int i = 0; i < MAXS; ++i)
    if (i < n_split)
      v[i] = __ldg(reinterpret_cast<const float4*>(part + i * split_stride + (size_t)r * d + c));
  float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int i = 0; i < MAXS; ++i)
    if (i < n_split) {
      s.x += v[i].x;
      s.y += v[i].y;
      s.z += v[i].z;
      s.w += v[i].w;
    }
  return s;
}

// V: 4-column vectors per thread (the CTA covers 1024 V columns); all of a
// thread's loads for one expert row are issued before its adds.
template <bool OVERLAP, int V>
__global__ void __launch_bounds__(256)
    combine_partials_kernel(const float* __restrict__ part, int n_split, size_t split_stride,
                            const int32_t* __restrict__ row_of_assign,
                            const float* __restrict__ topk_w, int k, int d, int shared_row0,
                            uint16_t* __restrict__ out) {
  const int t = blockIdx.x;
  int cv[V];
#pragma unroll
  for (int v = 0; v < V; ++v) cv[v] = ((blockIdx.y * V + v) * 256 + threadIdx.x) * 4;
  // The token's rows and weights come from the routing kernels, which finished
  // before the GEMM that precedes this kernel passed its own dependency wait,
  // so they are read before this kernel's wait (only the partial sums come
  // from the preceding kernel).
  constexpr int PRE = 8;
  int rj[PRE];
  float wj[PRE];
#pragma unroll
  for (int j = 0; j < PRE; ++j)
    if (j < k) {
      rj[j] = row_of_assign[t * k + j];
      wj[j] = topk_w[t * k + j];
    }
  griddep_wait();
  griddep_launch_dependents();
  if (cv[0] >= d) return;
  float4 acc[V];
#pragma unroll
  for (int v = 0; v < V; ++v) acc[v] = make_float4(0.f, 0.f, 0.f, 0.f);
  auto add = [&](float4 (&y)[V], float w) {   // acc += w * y, this thread's columns
#pragma unroll
    for (int v = 0; v < V; ++v) {
      if (cv[v] >= d) continue;
      acc[v].x += w * y[v].x;
      acc[v].y += w * y[v].y;
      acc[v].z += w * y[v].z;
      acc[v].w += w * y[v].w;
    }
  };
  if (OVERLAP && n_split == 1 && k <= PRE) {
    // one split (decode with many experts per token): every row's load is in
    // flight before the first add (the rows are independent; the sum keeps its
    // order, so the result is the same bits as the loop below)
    float4 y[PRE + 1][V];
#pragma unroll
    for (int j = 0; j < PRE; ++j)
#pragma unroll
      for (int v = 0; v < V; ++v)
        if (j < k && rj[j] >= 0 && cv[v] < d)
          y[j][v] = __ldg(reinterpret_cast<const float4*>(part + (size_t)rj[j] * d + cv[v]));
#pragma unroll
    for (int v = 0; v < V; ++v)
      if (shared_row0 >= 0 && cv[v] < d)
        y[PRE][v] = __ldg(reinterpret_cast<const float4*>(part + (size_t)(shared_row0 + t) * d + cv[v]));
#pragma unroll
    for (int j = 0; j < PRE; ++j)
      if (j < k && rj[j] >= 0) add(y[j], wj[j]);   // r < 0 only after an index error
    if (shared_row0 >= 0) add(y[PRE], 1.f);
  } else if (OVERLAP && V == 1 && k <= 2 && n_split <= 8 && shared_row0 < 0) {
    // top-2 with K splits (decode of a few wide experts): both rows' split loads
    // in flight at once; each row's splits summed in split order, then the
    // weighted adds in j order -- the same bits as the loop below
    float4 y[2][8];
#pragma unroll
    for (int j = 0; j < 2; ++j)
#pragma unroll
      for (int i = 0; i < 8; ++i)
        if (j < k && i < n_split && rj[j] >= 0)
          y[j][i] = __ldg(reinterpret_cast<const float4*>(part + i * split_stride + (size_t)rj[j] * d + cv[0]));
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      if (j >= k || rj[j] < 0) continue;   // r < 0 only after an index error
      float4 sj[V] = {make_float4(0.f, 0.f, 0.f, 0.f)};
#pragma unroll
      for (int i = 0; i < 8; ++i)
        if (i < n_split) {
          sj[0].x += y[j][i].x;
          sj[0].y += y[j][i].y;
          sj[0].z += y[j][i].z;
          sj[0].w += y[j][i].w;
        }
      add(sj, wj[j]);
    }
  } else if (!OVERLAP && n_split == 1 && k <= 4) {
    // up to top-4, one split (the prefill chunks): every row's loads in flight
    // before the first add; the same adds in the same order as the loop below,
    // so the same bits (2048 x 4096 top-2: 27 -> 17 us)
    float4 y[4][V];
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int v = 0; v < V; ++v)
        if (j < k && rj[j] >= 0 && cv[v] < d)
          y[j][v] = __ldg(reinterpret_cast<const float4*>(part + (size_t)rj[j] * d + cv[v]));
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (j < k && rj[j] >= 0) add(y[j], wj[j]);   // r < 0 only after an index error
    if (shared_row0 >= 0) {
#pragma unroll
      for (int v = 0; v < V; ++v) {
        if (cv[v] >= d) continue;
        const float4 ys = __ldg(reinterpret_cast<const float4*>(part + (size_t)(shared_row0 + t) * d + cv[v]));
        acc[v].x += ys.x;
        acc[v].y += ys.y;
        acc[v].z += ys.z;
        acc[v].w += ys.w;
      }
    }
  } else {
    auto add_row = [&](int r, float w) {   // acc += w * y[r], this thread's columns
      if (r < 0) return;                    // r < 0 only after an index error
      float4 y[V];
#pragma unroll
      for (int v = 0; v < V; ++v)
        if (cv[v] < d) y[v] = y_from_partials<OVERLAP>(part, n_split, split_stride, r, d, cv[v]);
      add(y, w);
    };
#pragma unroll
    for (int j = 0; j < PRE; ++j)
      if (j < k) add_row(rj[j], wj[j]);
    for (int j = PRE; j < k; ++j) add_row(row_of_assign[t * k + j], topk_w[t * k + j]);
    if (shared_row0 >= 0) {
#pragma unroll
      for (int v = 0; v < V; ++v) {
        if (cv[v] >= d) continue;
        const float4 y = y_from_partials<OVERLAP>(part, n_split, split_stride, shared_row0 + t, d, cv[v]);
        acc[v].x += y.x;
        acc[v].y += y.y;
        acc[v].z += y.z;
        acc[v].w += y.w;
      }
    }
  }
#pragma unroll
  for (int v = 0; v < V; ++v)
    if (cv[v] < d) store_bf16x4(out + (size_t)t * d + cv[v], acc[v]);
}

__global__ void __launch_bounds__(256)
    combine_bf16_kernel(const uint16_t* __restrict__ y_perm, const int32_t* __restrict__ row_of_assign,
                        const float* __restrict__ topk_w, const uint16_t* __restrict__ shared_y,
                        int k, int d, uint16_t* __restrict__ out) {
  const int t = blockIdx.x;
  const int c = (blockIdx.y * 256 + threadIdx.x) * 4;
  if (c >= d) return;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int j = 0; j < k; ++j) {
    const int r = row_of_assign[t * k + j];
    if (r < 0) continue;
    const float w = topk_w[t * k + j];
    const float4 y = load_bf16x4(y_perm + (size_t)r * d + c);
    acc.x += w * y.x;
    acc.y += w * y.y;
    acc.z += w * y.z;
    acc.w += w * y.w;
  }
  if (shared_y != nullptr) {
    const float4 y = load_bf16x4(shared_y + (size_t)t * d + c);
    acc.x += y.x;
    acc.y += y.y;
    acc.z += y.z;
    acc.w += y.w;
  }
  store_bf16x4(out + (size_t)t * d + c, acc);
}

__global__ void __launch_bounds__(256) reduce_splits_kernel(const float* __restrict__ part,
                                                            int n_split, size_t split_stride,
                                                            int d, uint16_t* __restrict__ y) {
  griddep_wait();
  griddep_launch_dependents();
  const int r = blockIdx.x;
  const int c = (blockIdx.y * 256 + threadIdx.x) * 4;
  if (c >= d) return;
  store_bf16x4(y + (size_t)r * d + c, y_from_partials<false>(part, n_split, split_stride, r, d, c));
}

static dim3 grid_rows(int rows, int d) { return dim3((unsigned)rows, (unsigned)((d + 1023) / 1024)); }

cudaError_t launch_combine_partials(const float* part, int n_split, size_t split_stride,
                                    const int32_t* row_of_assign, const float* topk_w, int T,
                                    int k, int d, int shared_row0, uint16_t* out, cudaStream_t s,
                                    bool pdl) {
  if (T <= 0) return cudaSuccess;
  if (T <= 256)
    return launch_kernel(combine_partials_kernel<true, 1>, grid_rows(T, d), dim3(256), 0, s, pdl, part,
                         n_split, split_stride, row_of_assign, topk_w, k, d, shared_row0, out);
  return launch_kernel(combine_partials_kernel<false, 2>, dim3((unsigned)T, (unsigned)((d + 2047) / 2048)),
                       dim3(256), 0, s, pdl, part, n_split, split_stride, row_of_assign, topk_w, k, d,
                       shared_row0, out);
}

cudaError_t launch_combine_bf16(const uint16_t* y_perm, const int32_t* row_of_assign,
                                const float* topk_w, const uint16_t* shared_y, int T, int k, int d,
                                uint16_t* out, cudaStream_t s) {
  if (T <= 0) return cudaSuccess;
  combine_bf16_kernel<<<grid_rows(T, d), 256, 0, s>>>(y_perm, row_of_assign, topk_w, shared_y, k,
                                                      d, out);
  return cudaGetLastError();
}

cudaError_t launch_reduce_splits(const float* part, int n_split, size_t split_stride, int rows,
                                 int d, uint16_t* y, cudaStream_t s, bool pdl) {
  if (rows <= 0) return cudaSuccess;
  return launch_kernel(reduce_splits_kernel, grid_rows(rows, d), dim3(256), 0, s, pdl, part, n_split,
                       split_stride, d, y);
}

}  // namespace moe
