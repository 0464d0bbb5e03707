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

cudaError_t launch_prepack(int fmt, int d, int F, const moe_expert_src& src, uint8_t* dst,
                           cudaStream_t s) {
  const int blocks = 1024, threads = 256;
  uint8_t* down_dst = dst + gateup_section_bytes(fmt, d, F);
  if (fmt == MOE_W_BF16) {
    prepack_bf16_kernel<<<blocks, threads, 0, s>>>((const uint16_t*)src.w[0],
                                                   (const uint16_t*)src.w[1], 2, F, d, dst);
    prepack_bf16_kernel<<<blocks, threads, 0, s>>>((const uint16_t*)src.w[2], nullptr, 1, d, F,
                                                   down_dst);
  } else {
    prepack_int4_kernel<<<blocks, threads, 0, s>>>(
        (const uint8_t*)src.w[0], src.scale[0], src.zero[0], (const uint8_t*)src.w[1],
        src.scale[1], src.zero[1], 2, F, d, dst);
    prepack_int4_kernel<<<blocks, threads, 0, s>>>((const uint8_t*)src.w[2], src.scale[2],
                                                   src.zero[2], nullptr, nullptr, nullptr, 1, d, F,
                                                   down_dst);
  }
  return cudaGetLastError();
}

}  // namespace moe
