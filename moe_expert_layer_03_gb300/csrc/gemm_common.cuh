// gemm_common.cuh -- pieces shared by the two grouped-GEMM kernels (gemm.cu:
// shared-memory A operand; gemm_group.cu: int4 group-scaled loop with the A
// operand in tensor memory): the device-built work list, item decoding, ring
// positions, nibble unpacking.
#pragma once
#include "kernels.cuh"
#include "ptx.cuh"

namespace moe {
namespace gemm {

struct Item {
  int g, mt, ks, r0, n_rows;
  const uint8_t* slot;
};

// Work list in shared memory: prefix[g] = first item of row group g, nch[g] =
// its row chunks, goff[g] = its first row.
struct WorkList {
  int* prefix;   // [n_groups + 1]
  int* nch;      // [n_groups + 1]
  int* goff;     // [n_groups + 1]
};

__host__ __device__ inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
__host__ __device__ inline size_t worklist_ints(int n_groups) { return 3 * (size_t)(n_groups + 1); }

// Built by one warp: items per group = row chunks * 128-row tiles * K splits.
// Returns the total item count (valid in lane 0's caller after the CTA barrier).
__device__ __forceinline__ int build_worklist(const GemmArgs& p, const WorkList& W, int lane) {
  int running = 0;
  bool bad = false;
  for (int g0 = 0; g0 < p.n_groups; g0 += 32) {
    const int g = g0 + lane;
    int items = 0, nch = 0;
    if (g < p.n_groups) {
      const int lo = p.offsets[g], hi = p.offsets[g + 1];
      int cnt = hi - lo;
      if (lo < 0 || cnt < 0 || hi > p.rows_total) { bad = true; cnt = 0; }
      nch = cnt > 0 ? (cnt + p.bn - 1) / p.bn : 0;
      items = nch * p.n_mt * p.ksplit;
      W.goff[g] = lo;
      if (g == p.n_groups - 1) W.goff[g + 1] = hi;
    }
    int incl = items;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += o;
    }
    if (g < p.n_groups) {
      W.prefix[g] = running + incl - items;
      W.nch[g] = nch;
    }
    running += __shfl_sync(0xffffffffu, incl, 31);
  }
  if (bad) atomicOr(p.err, MOE_DEVERR_OFFSETS);
  if (lane == 0) W.prefix[p.n_groups] = running;
  return running;
}

__device__ __forceinline__ bool decode_item(int item, const GemmArgs& p, const WorkList& W, Item& it) {
  int lo = 0, hi = p.n_groups - 1;
  while (lo < hi) {   // last group whose first item is <= item (empty groups are skipped)
    const int mid = (lo + hi + 1) >> 1;
    if (W.prefix[mid] <= item) lo = mid; else hi = mid - 1;
  }
  const int g = lo;
  const int local = item - W.prefix[g];
  const int nch = W.nch[g];
  const int nc = local % nch;
  const int t2 = local / nch;
  it.g = g;
  it.ks = t2 % p.ksplit;
  it.mt = t2 / p.ksplit;
  const int cnt = W.goff[g + 1] - W.goff[g];
  const int rpc = (((cnt + nch - 1) / nch) + 15) & ~15;   // rows per chunk, multiple of 16
  it.r0 = W.goff[g] + nc * rpc;
  it.n_rows = min(rpc, cnt - nc * rpc);
  int slot;
  if (g < p.n_routed) {
    slot = p.e2s_r[g];
    if (slot < 0 || slot >= p.n_slots_r) { atomicOr(p.err, MOE_DEVERR_SLOT_RANGE); return false; }
    it.slot = p.pool_r + (size_t)slot * p.slot_bytes_r;
  } else {
    slot = p.e2s_s[0];
    if (slot < 0 || slot >= p.n_slots_s) { atomicOr(p.err, MOE_DEVERR_SLOT_RANGE); return false; }
    it.slot = p.pool_s + (size_t)slot * p.slot_bytes_s;
  }
  return true;
}

// K range of split ks, in whole quantisation groups of 128.
__device__ __forceinline__ void kgroups(const GemmArgs& p, int ks, int& g0, int& g1) {
  const int G = p.K / QGROUP;
  g0 = (int)((long long)ks * G / p.ksplit);
  g1 = (int)((long long)(ks + 1) * G / p.ksplit);
}

struct Ring {
  int i;
  uint32_t ph;
  int n;
  __device__ __forceinline__ void next() {
    if (++i == n) { i = 0; ph ^= 1u; }
  }
};

// The 8 nibbles of a word -> 4 fp16 pairs (1024 + q): one LOP3 per pair.  In
// the prepacked layout element 2i sits in bits [4i, 4i+4) and 2i+1 in bits
// [16+4i, 20+4i), so pair i comes out in K order.
__device__ __forceinline__ void codes_of_word(uint32_t w, uint32_t* o) {
#pragma unroll
  for (int i = 0; i < 4; ++i) o[i] = lop3_and_or(w >> (4 * i), 0x000F000Fu, 0x64006400u);
}

// The 8 nibbles of a word -> 4 fp16 pairs holding q - z, exact for an integer
// zero point z.  Pair i is (element 2i at bits [4i, 4i+4), element 2i+1 at bits
// [16+4i, 20+4i)).  A nibble masked into the low mantissa bits of the fp16
// pattern of 1024 (0x6400) reads as 1024 + q (bits 0-3) or 1024 + 16q (bits
// 4-7); the upper two nibbles of each half are shifted down by 8 first.  One
// fp16 add (or FMA with 1/16) then removes the offset and the zero:
// nz_a = -(1024 + z), nz_b = -(64 + z).  Every intermediate is an integer
// below 2048, so no step rounds.
__device__ __forceinline__ uint32_t h2_add(uint32_t a, uint32_t b) {
  const __half2 r = __hadd2(*reinterpret_cast<const __half2*>(&a), *reinterpret_cast<const __half2*>(&b));
  return *reinterpret_cast<const uint32_t*>(&r);
}
__device__ __forceinline__ uint32_t h2_fma(uint32_t a, uint32_t b, uint32_t c) {
  const __half2 r = __hfma2(*reinterpret_cast<const __half2*>(&a), *reinterpret_cast<const __half2*>(&b),
                            *reinterpret_cast<const __half2*>(&c));
  return *reinterpret_cast<const uint32_t*>(&r);
}
__device__ __forceinline__ void codes_minus_zero(uint32_t w, uint32_t nz_a, uint32_t nz_b, uint32_t* o) {
  constexpr uint32_t SIXTEENTH = 0x2C002C00u;   // fp16 1/16 in both halves
  const uint32_t hi = w >> 8;
  o[0] = h2_add(lop3_and_or(w, 0x000F000Fu, 0x64006400u), nz_a);
  o[1] = h2_fma(lop3_and_or(w, 0x00F000F0u, 0x64006400u), SIXTEENTH, nz_b);
  o[2] = h2_add(lop3_and_or(hi, 0x000F000Fu, 0x64006400u), nz_a);
  o[3] = h2_fma(lop3_and_or(hi, 0x00F000F0u, 0x64006400u), SIXTEENTH, nz_b);
}

// silu(g) = g / (1 + e^-g) with the fast exponential and the approximate
// quotient: for g below about -87, e^-g overflows and the quotient is 0 (the
// limit); elsewhere a few ulp of fp32, far below the fp16/bf16 rounding of h.
__device__ __forceinline__ float silu_f(float g) { return __fdividef(g, 1.0f + __expf(-g)); }

// (a, b) -> fp16 pair (a in the low half), each saturated to the finite range
// and rounded to nearest even.
__device__ __forceinline__ uint32_t half2_bits_sat(float a, float b) {
  const __half2 t = __floats2half2_rn(fminf(fmaxf(a, -65504.f), 65504.f), fminf(fmaxf(b, -65504.f), 65504.f));
  return *reinterpret_cast<const uint32_t*>(&t);
}
// (a, b) -> bf16 pair (a in the low half), rounded to nearest even.
__device__ __forceinline__ uint32_t bf162_bits(float a, float b) {
  const __nv_bfloat162 t = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&t);
}

}  // namespace gemm
}  // namespace moe
