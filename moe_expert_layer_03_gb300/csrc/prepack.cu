// prepack.cu -- one-off rewrite of an expert's canonical weights into the slot
// layout streamed by the grouped GEMM (layout described in kernels.cuh).  Not on
// the hot path; one thread per 16-byte chunk of the destination.
#include "kernels.cuh"
#include "ptx.cuh"

namespace moe {

// bf16: destination block b = (mt * KS + ks) * NMAT + m; chunk (r, p) holds the
// source chunk j = p ^ (r % 8) of row mt*128 + r, K elements ks*64 + 8j .. +8.
__global__ void prepack_bf16_kernel(const uint16_t* __restrict__ w0, const uint16_t* __restrict__ w1,
                                    int nmat, int rows, int K, uint8_t* __restrict__ dst) {
  const int KS = K / KSTEP;
  const size_t n_chunks = (size_t)(rows / TILE_M) * KS * nmat * (BF16_TILE_BYTES / 16);
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n_chunks;
       i += (size_t)gridDim.x * blockDim.x) {
    const int within = (int)(i % (BF16_TILE_BYTES / 16));   // r * 8 + p
    const size_t blk = i / (BF16_TILE_BYTES / 16);
    const int m = (int)(blk % nmat);
    const size_t t2 = blk / nmat;
    const int ks = (int)(t2 % KS);
    const int mt = (int)(t2 / KS);
    const int r = within >> 3, p = within & 7, j = p ^ (r & 7);
    const uint16_t* src = (m == 0 ? w0 : w1) + (size_t)(mt * TILE_M + r) * K + ks * KSTEP + j * 8;
    *reinterpret_cast<uint4*>(dst + i * 16) = *reinterpret_cast<const uint4*>(src);
  }
}

// int4: gate/up (NMAT = 2) block b = (mt * G + g) * 2 + m of I4_MAT_BYTES; the
// down matrix (NMAT = 1) block at i4_down_block(mt, g).  Chunks
// 0..511 are the nibble quads (h, j, r) at ((h*2+j)*128 + r); chunks 512..543
// carry the (scale | zero << 16) words, 4 rows per chunk.
__global__ void prepack_int4_kernel(const uint8_t* __restrict__ q0, const uint16_t* __restrict__ s0,
                                    const uint16_t* __restrict__ z0, const uint8_t* __restrict__ q1,
                                    const uint16_t* __restrict__ s1, const uint16_t* __restrict__ z1,
                                    int nmat, int rows, int K, uint8_t* __restrict__ dst) {
  const int G = K / QGROUP;
  constexpr int CH = I4_MAT_BYTES / 16;   // 544
  const size_t n_chunks = (size_t)(rows / TILE_M) * G * nmat * CH;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n_chunks;
       i += (size_t)gridDim.x * blockDim.x) {
    const int c = (int)(i % CH);
    const size_t blk = i / CH;
    const int m = (int)(blk % nmat);
    const size_t t2 = blk / nmat;
    const int g = (int)(t2 % G);
    const int mt = (int)(t2 / G);
    const uint8_t* q = m == 0 ? q0 : q1;
    const uint16_t* sc = m == 0 ? s0 : s1;
    const uint16_t* zr = m == 0 ? z0 : z1;
    uint32_t out[4];
    if (c < 512) {
      const int r = c & 127, hj = c >> 7, h = hj >> 1, j = hj & 1;
      const int row = mt * TILE_M + r;
      const uint8_t* qrow = q + (size_t)row * (K / 2);
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        const int kb = g * QGROUP + h * 64 + j * 32 + w * 8;   // first K element of the word
        uint32_t word = 0;
#pragma unroll
        for (int i2 = 0; i2 < 4; ++i2) {
          const uint32_t byte = qrow[(kb >> 1) + i2];   // elements kb+2i2 (low), kb+2i2+1 (high)
          word |= (byte & 0xFu) << (4 * i2);
          word |= (byte >> 4) << (16 + 4 * i2);
        }
        out[w] = word;
      }
    } else {
      const int r0 = (c - 512) * 4;
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        const size_t gi = (size_t)(mt * TILE_M + r0 + w) * G + g;
        out[w] = (uint32_t)sc[gi] | ((uint32_t)zr[gi] << 16);
      }
    }
    const size_t blk_off = nmat == 2 ? blk * I4_MAT_BYTES : i4_down_block(mt, g, G, rows / TILE_M);
    *reinterpret_cast<uint4*>(dst + blk_off + (size_t)c * 16) = make_uint4(out[0], out[1], out[2], out[3]);
  }
}

// fp8: the block of (mt, g) holds NMAT code tiles then NMAT x 128 fp16 scales
// (layout in kernels.cuh).  Chunk (m, r, p) of a code tile holds the codes of
// row mt*128 + r for K elements g*128 + 16j .. +16, j = p ^ (r % 8), each
// 8-element block in the order {0,4,1,5,2,6,3,7}; the scale part is
// NMAT * 16 chunks of 8 scales.  down (NMAT = 1): the blocks of a tile pair
// share one 2-matrix block (fp8_down_block).
__global__ void prepack_fp8_kernel(const uint8_t* __restrict__ q0, const uint16_t* __restrict__ s0,
                                   const uint8_t* __restrict__ q1, const uint16_t* __restrict__ s1,
                                   int nmat, int rows, int K, uint8_t* __restrict__ dst) {
  const int G = K / QGROUP, n_mt = rows / TILE_M;
  constexpr int CODE_CH = F8_CODE_BYTES / 16;   // 1024 chunks per code tile
  constexpr int SC_CH = TILE_M * 2 / 16;        // 16 chunks of scales per matrix
  const size_t n_chunks = (size_t)n_mt * G * nmat * (CODE_CH + SC_CH);
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n_chunks;
       i += (size_t)gridDim.x * blockDim.x) {
    const int c = (int)(i % (CODE_CH + SC_CH));   // chunk within the matrix's share
    const size_t t2 = i / (CODE_CH + SC_CH);
    const int m = (int)(t2 % nmat);
    const size_t t3 = t2 / nmat;
    const int g = (int)(t3 % G);
    const int mt = (int)(t3 / G);
    // where the matrix sits: gate/up blocks hold both matrices of (mt, g);
    // the down section pairs output tiles
    size_t blk;
    int mpos, bmat;
    if (nmat == 2) {
      blk = ((size_t)mt * G + g) * (2 * F8_MAT_BYTES);
      mpos = m;
      bmat = 2;
    } else {
      blk = fp8_down_block(mt, g, G, n_mt, mpos, bmat);
    }
    const uint8_t* q = m == 0 ? q0 : q1;
    const uint16_t* sc = m == 0 ? s0 : s1;
    uint32_t out[4];
    size_t off;
    if (c < CODE_CH) {
      const int r = c >> 3, pch = c & 7, j = pch ^ (r & 7);
      const uint8_t* src = q + (size_t)(mt * TILE_M + r) * K + g * QGROUP + j * 16;
      uint8_t b[16];
#pragma unroll
      for (int blk8 = 0; blk8 < 2; ++blk8)
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int slot = e < 4 ? 2 * e : 2 * (e - 4) + 1;   // stored position of element e
          b[blk8 * 8 + slot] = src[blk8 * 8 + e];
        }
#pragma unroll
      for (int w = 0; w < 4; ++w)
        out[w] = (uint32_t)b[4 * w] | ((uint32_t)b[4 * w + 1] << 8) | ((uint32_t)b[4 * w + 2] << 16) |
                 ((uint32_t)b[4 * w + 3] << 24);
      off = blk + (size_t)mpos * F8_CODE_BYTES + (size_t)c * 16;
    } else {
      const int r0 = (c - CODE_CH) * 8;
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        const uint32_t lo = sc[(size_t)(mt * TILE_M + r0 + 2 * w) * G + g];
        const uint32_t hi = sc[(size_t)(mt * TILE_M + r0 + 2 * w + 1) * G + g];
        out[w] = lo | (hi << 16);
      }
      off = blk + (size_t)bmat * F8_CODE_BYTES + (size_t)mpos * TILE_M * 2 + (size_t)r0 * 2;
    }
    *reinterpret_cast<uint4*>(dst + off) = make_uint4(out[0], out[1], out[2], out[3]);
  }
}

// Slot trailer (kernels.cuh): largest row L1 norm of a quantised matrix [rows][K]
// in its canonical form, one warp per row, sum_k |w| in fp32 with w the
// dequantised value ((q - z) * s for int4, e4m3(q) * s for fp8); the row maxima
// meet in trailer float m by an integer atomicMax (non-negative floats order
// like their bit patterns).
__global__ void row_l1_max_kernel(int fmt, const uint8_t* __restrict__ q, const uint16_t* __restrict__ sc,
                                  const uint16_t* __restrict__ zr, int rows, int K, float* __restrict__ out) {
  const int lane = threadIdx.x & 31;
  const int G = K / QGROUP;
  for (int row = (int)((blockIdx.x * blockDim.x + threadIdx.x) >> 5); row < rows;
       row += (int)((gridDim.x * blockDim.x) >> 5)) {
    float acc = 0.f;
    for (int k = lane; k < K; k += 32) {
      const int g = k / QGROUP;
      const float s = __half2float(__ushort_as_half(sc[(size_t)row * G + g]));
      float w;
      if (fmt == MOE_W_INT4_G128) {
        const uint8_t b = q[(size_t)row * (K / 2) + (k >> 1)];
        const int code = (k & 1) ? (b >> 4) : (b & 15);
        w = ((float)code - __half2float(__ushort_as_half(zr[(size_t)row * G + g]))) * s;
      } else {
        const uint16_t pair = q[(size_t)row * K + k];
        w = e4m3x2_to_f32x2(pair).x * s;
      }
      acc += fabsf(w);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (lane == 0) atomicMax(reinterpret_cast<int*>(out), __float_as_int(acc));
  }
}

// trailer B[m] = ceil(log2(L[m] * (1 + 2^-7))) (the margin covers the fp16
// rounding of the GEMM's weights and the fp32 sums), clamped to [-126, 127].
__global__ void trailer_bounds_kernel(uint8_t* trailer) {
  const int m = threadIdx.x;
  if (m >= 2) return;
  const float L = reinterpret_cast<const float*>(trailer)[m] * (1.0f + 0.0078125f);
  int b = -126;
  if (L > 0.f) {
    int e;
    const float f = frexpf(L, &e);   // L = f * 2^e, f in [0.5, 1)
    b = f == 0.5f ? e - 1 : e;       // smallest b with L <= 2^b
  }
  reinterpret_cast<int*>(trailer + 8)[m] = max(-126, min(127, b));
}

cudaError_t launch_prepack(int fmt, int d, int F, const moe_expert_src& src, uint8_t* dst,
                           cudaStream_t s) {
  const int blocks = 1024, threads = 256;
  uint8_t* down_dst = dst + gateup_section_bytes(fmt, d, F);
  if (fmt == MOE_W_BF16) {
    prepack_bf16_kernel<<<blocks, threads, 0, s>>>((const uint16_t*)src.w[0],
                                                   (const uint16_t*)src.w[1], 2, F, d, dst);
    prepack_bf16_kernel<<<blocks, threads, 0, s>>>((const uint16_t*)src.w[2], nullptr, 1, d, F,
                                                   down_dst);
  } else if (fmt == MOE_W_FP8_G128) {
    prepack_fp8_kernel<<<blocks, threads, 0, s>>>((const uint8_t*)src.w[0], src.scale[0],
                                                  (const uint8_t*)src.w[1], src.scale[1], 2, F, d, dst);
    prepack_fp8_kernel<<<blocks, threads, 0, s>>>((const uint8_t*)src.w[2], src.scale[2], nullptr,
                                                  nullptr, 1, d, F, down_dst);
  } else {
    prepack_int4_kernel<<<blocks, threads, 0, s>>>(
        (const uint8_t*)src.w[0], src.scale[0], src.zero[0], (const uint8_t*)src.w[1],
        src.scale[1], src.zero[1], 2, F, d, dst);
    prepack_int4_kernel<<<blocks, threads, 0, s>>>((const uint8_t*)src.w[2], src.scale[2],
                                                   src.zero[2], nullptr, nullptr, nullptr, 1, d, F,
                                                   down_dst);
  }
  uint8_t* trailer = dst + slot_payload_bytes(fmt, d, F);
  cudaError_t e = cudaMemsetAsync(trailer, 0, SLOT_TRAILER_BYTES, s);
  if (e != cudaSuccess) return e;
  if (fmt_quantised(fmt)) {
    const int l1_blocks = (F + 7) / 8 < 1024 ? (F + 7) / 8 : 1024;   // 8 warps (rows) per block
    for (int m = 0; m < 2; ++m)
      row_l1_max_kernel<<<l1_blocks, 256, 0, s>>>(fmt, (const uint8_t*)src.w[m], src.scale[m],
                                                  fmt == MOE_W_INT4_G128 ? src.zero[m] : nullptr, F, d,
                                                  reinterpret_cast<float*>(trailer) + m);
    trailer_bounds_kernel<<<1, 32, 0, s>>>(trailer);
  }
  return cudaGetLastError();
}

}  // namespace moe
