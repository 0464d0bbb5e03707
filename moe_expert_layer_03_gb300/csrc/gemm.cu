// gemm.cu -- grouped expert GEMM on the 5th-generation tensor cores (tcgen05),
// A operand in shared memory: bf16 experts, and int4 experts with row chunks of
// more than 32 rows (prefill).  Decode-sized int4 chunks use gemm_group.cu.
//
// "125B MoE on an RTX 3090 at 100+ tok/s": sec. 3.2 -- each expert FFN is a
// two-layer MLP; the tokens of each expert form one contiguous batch and the
// active experts run as one grouped GEMM instead of many small ones; sec. 3.1 --
// per-expert int4 weights with their own scale and zero-point, dequantised to
// fp16 for the tensor cores on the way in rather than in a separate pass.  The
// fp16 token rows and h are scaled per row by powers of two so that neither
// can leave fp16's range: x by its row maximum (the gather), h by a bound from
// x's row maximum and the expert's largest gate / up row L1 norms (the slot
// trailer, h_row_scale); the scales are undone in fp32.
//
// One persistent CTA per SM walks a list of work items
//   (expert group g, 128-row weight tile mt, K split ks, row chunk nc)
// built on the device from the group offsets, so experts without rows cost
// nothing.  The MMA is "swap-AB": weight rows are the M = 128 side and the
// expert's token rows the N side (16..256, a multiple of 16 set per item).
//
//   warp 0      producer: 1-D bulk copies of the prepacked weight blocks
//               (int4 nibbles + scales, or pre-swizzled bf16 tiles) and 2-D TMA
//               loads of the 64-wide K slices of the token rows (128-byte swizzle)
//   warp 1      TMEM owner and MMA issuer (tcgen05.mma kind::f16 from a
//               converged warp, fp32 accumulators in TMEM: gate/tile 0 at
//               column 0, up/tile 1 at column bn); bf16 operands for bf16
//               weights (A tiles in shared memory), fp16 for int4 weights
//   warps 2..   int4: write fp16((q - z) * s) ((q - z) exact, one rounding of
//               the product) for each 64-wide K slice into an A slot in TMEM
//               (beside the accumulators), so the A operand costs no shared-
//               memory bandwidth; then, per item, the epilogue: tcgen05.ld,
//               SwiGLU -> h, or fp32 K-split partials.
// int4 down GEMMs with an even number of output tiles take two adjacent tiles
// per item (like gate and up), so each token tile serves two weight tiles.
// Prefill-sized int4 items are at most 192 rows wide: 2 x 192 accumulator
// columns + 2 A slots of 64 columns fill the 512 TMEM columns.
//
// Every wait is bounded (ptx.cuh); on a timeout the CTA drains its in-flight
// copies and MMAs, frees TMEM and returns with MOE_DEVERR_TIMEOUT set.
#include "gemm_common.cuh"

namespace moe {

using namespace gemm;

namespace {

constexpr int MISC_INTS = 10;   // [0] tmem [1] abort [2] items; consumed raw/a/b [3..5];
                                // issued raw/a/b [6..8]; [9] stays 0
constexpr int A_SLOT_COLS = 32;   // TMEM columns of one matrix's 64-wide fp16 K slice

struct Shared {   // views into the dynamic shared-memory carve-out
  uint8_t* a_ring;   // bf16 only (int4 A slots live in TMEM)
  uint8_t* b_ring;
  uint8_t* raw_ring;
  uint64_t *a_full, *a_empty, *b_full, *b_empty, *raw_full, *raw_empty;
  uint64_t *tmem_full, *tmem_empty, *fin;
  int* misc;
  WorkList W;
};

// quant_bytes: bytes of one matrix's raw block (int4 or fp8), 0 for bf16.
size_t carve_bytes(int nmat, int quant_bytes, int bn, int n_a, int n_b, int n_raw, int n_groups) {
  const bool quant = quant_bytes > 0;
  size_t s = (quant ? 0 : (size_t)n_a * nmat * BF16_TILE_BYTES) + (size_t)n_b * bn * 128;
  if (quant) s += (size_t)n_raw * nmat * quant_bytes;
  s = align_up(s, 16);
  s += 8 * (size_t)(2 * (n_a + n_b + (quant ? n_raw : 0)) + 3);
  s += 4 * (MISC_INTS + worklist_ints(n_groups));
  return s;
}

// 8 words of one row (64 K elements) -> 32 fp16 pairs (q - z) * s, K order.
__device__ __forceinline__ void dequant_words(const uint4& w0, const uint4& w1, uint32_t nz_a, uint32_t nz_b,
                                              __half2 s2, uint32_t (&v)[32]) {
  const uint32_t words[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
  for (int w = 0; w < 8; ++w) codes_minus_zero(words[w], nz_a, nz_b, &v[w * 4]);
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    const __half2 b = __hmul2(*reinterpret_cast<const __half2*>(&v[i]), s2);   // one rounding
    v[i] = *reinterpret_cast<const uint32_t*>(&b);
  }
}
__device__ __forceinline__ void dequant_words16(const uint4& w0, uint32_t nz_a, uint32_t nz_b, __half2 s2,
                                                uint32_t (&v)[16]) {
  const uint32_t words[4] = {w0.x, w0.y, w0.z, w0.w};
#pragma unroll
  for (int w = 0; w < 4; ++w) codes_minus_zero(words[w], nz_a, nz_b, &v[w * 4]);
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const __half2 b = __hmul2(*reinterpret_cast<const __half2*>(&v[i]), s2);
    v[i] = *reinterpret_cast<const uint32_t*>(&b);
  }
}

// fp8: codes of row r for K chunks [c0, c0 + NC) of 16 (a 128-byte-swizzled
// row: chunk j at j ^ (r % 8); each 8-element block stored in the order
// {0,4,1,5,2,6,3,7}) -> fp16 pairs e4m3(q) * s in K order, 8 per chunk.
template <int NC>
__device__ __forceinline__ void dequant_fp8(const uint8_t* codes, int r, int c0, __half2 s2,
                                            uint32_t (&v)[8 * NC]) {
#pragma unroll
  for (int c = 0; c < NC; ++c) {
    const uint4 q = *reinterpret_cast<const uint4*>(codes + r * 128 + (((c0 + c) ^ (r & 7)) << 4));
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int b = 0; b < 2; ++b) {   // 8-element block b of the chunk: words w[2b] = (e0,e4,e1,e5), w[2b+1] = (e2,e6,e3,e7)
      const uint32_t lo = w[2 * b], hi = w[2 * b + 1];
      const uint16_t pr[4] = {(uint16_t)__byte_perm(lo, 0, 0x0020), (uint16_t)__byte_perm(hi, 0, 0x0020),
                              (uint16_t)__byte_perm(lo, 0, 0x0031), (uint16_t)__byte_perm(hi, 0, 0x0031)};
#pragma unroll
      for (int i = 0; i < 4; ++i) {   // pairs (e0,e1), (e2,e3), (e4,e5), (e6,e7)
        const uint32_t f = e4m3x2_to_f16x2(pr[i]);
        const __half2 h = __hmul2(*reinterpret_cast<const __half2*>(&f), s2);   // one rounding
        v[c * 8 + b * 4 + i] = *reinterpret_cast<const uint32_t*>(&h);
      }
    }
  }
}

// h's fp16 scale for one token row of a quantised prefill GEMM: x entered as
// fp16 x * 2^ex with max|x| * 2^ex < 2^14 (ux = 2^-ex), and every gate / up
// output of the row is at most max|x| * 2^Bg / * 2^Bu (bsum = Bg + Bu, the slot
// trailer's bound exponents), so |h| = |silu(g) u| <= |g| |u| <
// 2^(28 - 2 ex + bsum).  Returns 2^eh with eh = 2 ex - 13 - bsum, which keeps
// |h| 2^eh below 2^15 (fp16's largest finite value is 65504); *inv = 2^-eh.
__device__ __forceinline__ float h_row_scale(float ux, int bsum, float* inv) {
  const int ex = 127 - (int)(__float_as_uint(ux) >> 23);
  const int eh = max(-126, min(126, 2 * ex - 13 - bsum));
  *inv = __int_as_float((127 - eh) << 23);
  return __int_as_float((127 + eh) << 23);
}

}  // namespace

template <int FMT, bool GATEUP, int NDQ, bool PAIR>
__global__ void __launch_bounds__((2 + NDQ) * 32, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmap_b, const GemmArgs p) {
  constexpr bool F8 = (FMT == MOE_W_FP8_G128);
  constexpr bool INT4 = (FMT == MOE_W_INT4_G128) || F8;   // quantised: raw blocks, A dequantised into TMEM
  static_assert(!PAIR || (INT4 && !GATEUP), "paired output tiles: quantised down GEMM only");
  constexpr int NMAT = (GATEUP || PAIR) ? 2 : 1;
  static_assert(!INT4 || NDQ == 8, "dequantisation assumes 8 warps (2 per TMEM quadrant)");
  constexpr uint32_t AB_BF16 = INT4 ? 0u : 1u;   // operand type of the MMA
  constexpr uint32_t A_STAGE = NMAT * BF16_TILE_BYTES;   // bf16: shared-memory A stage
  constexpr uint32_t A_SLOT = NMAT * A_SLOT_COLS;        // quantised: TMEM columns of one A slot
  constexpr uint32_t MAT_RAW = F8 ? F8_MAT_BYTES : I4_MAT_BYTES;
  constexpr uint32_t RAW_STAGE = NMAT * MAT_RAW;
  constexpr int NDQ_THREADS = NDQ * 32;
  const uint32_t B_STAGE = (uint32_t)p.bn * 128u;

  extern __shared__ uint8_t smem_dyn[];
  const uint32_t pad = (1024u - (smem_u32(smem_dyn) & 1023u)) & 1023u;
  uint8_t* base = smem_dyn + pad;

  Shared S;
  S.a_ring = base;
  S.b_ring = S.a_ring + (INT4 ? 0 : (size_t)p.n_a * A_STAGE);
  S.raw_ring = S.b_ring + (size_t)p.n_b * B_STAGE;
  uint8_t* cur = S.raw_ring + (INT4 ? (size_t)p.n_raw * RAW_STAGE : 0);
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + align_up((size_t)(cur - base), 16));
  S.a_full = bars;
  S.a_empty = S.a_full + p.n_a;
  S.b_full = S.a_empty + p.n_a;
  S.b_empty = S.b_full + p.n_b;
  S.raw_full = S.b_empty + p.n_b;
  S.raw_empty = S.raw_full + (INT4 ? p.n_raw : 0);
  S.tmem_full = S.raw_empty + (INT4 ? p.n_raw : 0);
  S.tmem_empty = S.tmem_full + 1;
  S.fin = S.tmem_empty + 1;
  S.misc = reinterpret_cast<int*>(S.fin + 1);
  S.W.prefix = S.misc + MISC_INTS;
  S.W.nch = S.W.prefix + (p.n_groups + 1);
  S.W.goff = S.W.nch + (p.n_groups + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int* abort_flag = &S.misc[1];

  // ------------------------------------------------------------ set-up
  if (threadIdx.x == 0) {
    for (int i = 0; i < p.n_a; ++i) {
      mbar_init(smem_u32(&S.a_full[i]), INT4 ? NDQ_THREADS : 1);
      mbar_init(smem_u32(&S.a_empty[i]), 1);
    }
    for (int i = 0; i < p.n_b; ++i) {
      mbar_init(smem_u32(&S.b_full[i]), 1);
      mbar_init(smem_u32(&S.b_empty[i]), 1);
    }
    if (INT4)
      for (int i = 0; i < p.n_raw; ++i) {
        mbar_init(smem_u32(&S.raw_full[i]), 1);
        mbar_init(smem_u32(&S.raw_empty[i]), NDQ_THREADS);
      }
    mbar_init(smem_u32(S.tmem_full), 1);
    mbar_init(smem_u32(S.tmem_empty), NDQ_THREADS);
    mbar_init(smem_u32(S.fin), 1);
    for (int i = 1; i < MISC_INTS; ++i)
      if (i != 2) S.misc[i] = 0;   // [0] written by tcgen05.alloc, [2] by warp 2
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) prefetch_tensormap(&tmap_b);
  if (warp == 1) {
    tmem_alloc(smem_u32(&S.misc[0]), p.tmem_cols);
    tmem_relinquish();
  }
  // everything above overlaps the previous kernel's tail (dependent launch);
  // below, the offsets, token rows and outputs of earlier kernels are read
  griddep_wait();
  griddep_launch_dependents();
  if (warp == 2) {
    const int total = build_worklist(p, S.W, lane);
    if (lane == 0) S.misc[2] = total;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = (uint32_t)S.misc[0];
  const int total = S.misc[2];
  const uint32_t a_col0 = (uint32_t)(NMAT * p.bn);   // int4: A slots follow the accumulators

  // ------------------------------------------------------------ roles
  if (warp == 0) {
    if (lane == 0) {   // ---------------- producer
      Ring ra{0, 0, p.n_a}, rb{0, 0, p.n_b}, rr{0, 0, p.n_raw};
      int issued_a = 0, issued_b = 0, issued_raw = 0;
      const uint64_t pol = policy_evict_first();
      for (int item = blockIdx.x; item < total && !*abort_flag; item += gridDim.x) {
        Item it;
        if (!decode_item(item, p, S.W, it)) continue;
        int g0, g1;
        kgroups(p, it.ks, g0, g1);
        const uint8_t* sec = it.slot + p.sec_off;
        bool ok = true;
        for (int kg = g0; kg < g1 && ok; ++kg) {
          if (issued_b == p.stop_stage) {   // test hook: stop feeding the pipeline
            ok = false;
            break;
          }
          if (INT4) {
            if (!(ok = mbar_wait(smem_u32(&S.raw_empty[rr.i]), rr.ph ^ 1u, abort_flag, p.err, p.wait_ns))) break;
            const uint32_t bar = smem_u32(&S.raw_full[rr.i]);
            mbar_arrive_expect_tx(bar, RAW_STAGE);
            const uint32_t raw = smem_u32(S.raw_ring + (size_t)rr.i * RAW_STAGE);
            // gate/up: gate and up blocks of (mt, kg); down: tile mt's block, or
            // both blocks of the pair it.mt, contiguous in the down section
            if (!GATEUP && !PAIR && F8) {   // one tile of a pair block: its codes, then its scales
              int mp, bm;
              const size_t blk = fp8_down_block(it.mt, kg, p.K / QGROUP, p.n_mt, mp, bm);
              bulk_g2s_hint(raw, sec + blk + (size_t)mp * F8_CODE_BYTES, F8_CODE_BYTES, bar, pol);
              bulk_g2s_hint(raw + F8_CODE_BYTES, sec + blk + (size_t)bm * F8_CODE_BYTES + mp * TILE_M * 2,
                            TILE_M * 2, bar, pol);
            } else {
              const size_t off = (GATEUP || PAIR) ? ((size_t)it.mt * (p.K / QGROUP) + kg) * RAW_STAGE
                                                  : i4_down_block(it.mt, kg, p.K / QGROUP, p.n_mt);
              bulk_g2s_hint(raw, sec + off, RAW_STAGE, bar, pol);
            }
            rr.next();
            ++issued_raw;
          }
          for (int h = 0; h < 2 && ok; ++h) {
            const int kstep = 2 * kg + h;
            if (!INT4) {
              if (!(ok = mbar_wait(smem_u32(&S.a_empty[ra.i]), ra.ph ^ 1u, abort_flag, p.err, p.wait_ns))) break;
              const uint32_t bar = smem_u32(&S.a_full[ra.i]);
              mbar_arrive_expect_tx(bar, A_STAGE);
              bulk_g2s_hint(smem_u32(S.a_ring + (size_t)ra.i * A_STAGE),
                            sec + ((size_t)it.mt * (p.K / KSTEP) + kstep) * A_STAGE, A_STAGE, bar, pol);
              ra.next();
              ++issued_a;
            }
            if (!(ok = mbar_wait(smem_u32(&S.b_empty[rb.i]), rb.ph ^ 1u, abort_flag, p.err, p.wait_ns))) break;
            const uint32_t bar = smem_u32(&S.b_full[rb.i]);
            mbar_arrive_expect_tx(bar, B_STAGE);
            tma_load_2d(smem_u32(S.b_ring + (size_t)rb.i * B_STAGE), &tmap_b, kstep * KSTEP, it.r0, bar);
            rb.next();
            ++issued_b;
          }
        }
        if (!ok) break;
      }
      S.misc[6] = issued_raw;
      S.misc[7] = issued_a;
      S.misc[8] = issued_b;
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer: the whole warp runs the loop, one elected
    // lane issues.  Descriptors are built once and offset per stage / K step.
    Ring ra{0, 0, p.n_a}, rb{0, 0, p.n_b};
    int consumed_a = 0, consumed_b = 0;
    uint32_t it_count = 0;
    bool ok = true;
    const uint64_t bdesc0 = sdesc_kmajor_sw128(smem_u32(S.b_ring));
    const uint64_t adesc0 = sdesc_kmajor_sw128(smem_u32(S.a_ring));   // bf16 only
    for (int item = blockIdx.x; item < total && ok; item += gridDim.x) {
      Item it;
      if (!decode_item(item, p, S.W, it)) continue;
      int g0, g1;
      kgroups(p, it.ks, g0, g1);
      if (!(ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(S.tmem_empty), (it_count & 1u) ^ 1u,
                                                   abort_flag, p.err, p.wait_ns))))
        break;
      tc_fence_after();
      const uint32_t idesc = idesc_f16kind_f32(TILE_M, (uint32_t)((it.n_rows + 15) & ~15), AB_BF16);
      for (int kg = g0; kg < g1 && ok; ++kg) {
        for (int h = 0; h < 2; ++h) {
          if (!(ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&S.a_full[ra.i]), ra.ph, abort_flag, p.err, p.wait_ns))))
            break;
          if (!(ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&S.b_full[rb.i]), rb.ph, abort_flag, p.err, p.wait_ns))))
            break;
          tc_fence_after();
          const bool fresh = (kg == g0 && h == 0);
          const uint64_t bd = bdesc0 + (uint64_t)(((uint32_t)rb.i * B_STAGE) >> 4);
#pragma unroll
          for (int kk = 0; kk < KSTEP / 16; ++kk) {
            const uint64_t bq = bd + (uint64_t)((kk * 32) >> 4);
            const uint32_t acc = (fresh && kk == 0) ? 0u : 1u;
            if constexpr (INT4) {
              const uint32_t a0 = tmem_base + a_col0 + (uint32_t)ra.i * A_SLOT + (uint32_t)(kk * 8);
              if (NMAT == 2)
                mma2_ta_elect(tmem_base, tmem_base + (uint32_t)p.bn, a0, a0 + A_SLOT_COLS, bq, idesc, acc);
              else
                mma_ta_elect(tmem_base, a0, bq, idesc, acc);
            } else {
              const uint64_t aq = adesc0 + (uint64_t)(((uint32_t)ra.i * A_STAGE + kk * 32) >> 4);
#pragma unroll
              for (int m = 0; m < NMAT; ++m)
                mma_ss_elect(tmem_base + (uint32_t)(m * p.bn), aq + (uint64_t)((m * BF16_TILE_BYTES) >> 4), bq,
                             idesc, acc);
            }
          }
          mma_commit_elect(smem_u32(&S.a_empty[ra.i]));
          mma_commit_elect(smem_u32(&S.b_empty[rb.i]));
          ra.next();
          rb.next();
          ++consumed_a;
          ++consumed_b;
        }
      }
      if (!ok) break;
      mma_commit_elect(smem_u32(S.tmem_full));
      ++it_count;
    }
    if (lane == 0) {
      S.misc[4] = consumed_a;
      S.misc[5] = consumed_b;
    }
  } else {   // ---------------- dequant + epilogue warps
    const int wr = warp - 2;                  // 0 .. NDQ-1
    const int quad = warp & 3;                // TMEM lane quadrant this warp may access
    const int r = quad * 32 + lane;           // weight row of the tile = TMEM lane
    const uint32_t tl = tmem_base + ((uint32_t)(quad * 32) << 16);
    // int4 ownership: two matrices -> matrix m_own of row r; one matrix -> K quad j_own of row r
    const int m_own = NMAT == 2 ? (wr >> 2) : 0;
    const int j_own = NMAT == 2 ? 0 : (wr >> 2);
    constexpr int NHALF = NDQ / 4;            // epilogue: column interleave per quadrant
    Ring ra{0, 0, p.n_a}, rr{0, 0, p.n_raw};
    int consumed_raw = 0;
    uint32_t it_count = 0;
    bool ok = true;
    for (int item = blockIdx.x; item < total && ok; item += gridDim.x) {
      Item it;
      if (!decode_item(item, p, S.W, it)) continue;
      int g0, g1;
      kgroups(p, it.ks, g0, g1);
      if (INT4) {
        for (int kg = g0; kg < g1 && ok; ++kg) {
          ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&S.raw_full[rr.i]), rr.ph, abort_flag, p.err, p.wait_ns));
          if (!ok) break;
          const uint8_t* raw = S.raw_ring + (size_t)rr.i * RAW_STAGE;
          const uint8_t* mat = raw + m_own * (F8 ? F8_CODE_BYTES : I4_MAT_BYTES);
          // int4: scale | zero << 16 after the nibbles; fp8: the scales after all code tiles
          const uint32_t sz = F8 ? (uint32_t)*reinterpret_cast<const uint16_t*>(raw + NMAT * F8_CODE_BYTES +
                                                                               m_own * TILE_M * 2 + r * 2)
                                 : *reinterpret_cast<const uint32_t*>(mat + I4_PACKED_BYTES + r * 4);
          const __half sh = __ushort_as_half((unsigned short)(sz & 0xFFFFu));
          const float zf = __half2float(__ushort_as_half((unsigned short)(sz >> 16)));
          const __half2 s2 = __halves2half2(sh, sh);
          const __half2 za = __float2half2_rn(-(1024.f + zf)), zb = __float2half2_rn(-(64.f + zf));
          const uint32_t nz_a = *reinterpret_cast<const uint32_t*>(&za);
          const uint32_t nz_b = *reinterpret_cast<const uint32_t*>(&zb);
          for (int h = 0; h < 2; ++h) {   // K slices of the group: 64 codes of my row each
            ok = __all_sync(0xffffffffu,
                            mbar_wait(smem_u32(&S.a_empty[ra.i]), ra.ph ^ 1u, abort_flag, p.err, p.wait_ns));
            if (!ok) break;
            tc_fence_after();
            const uint32_t ta = tl + a_col0 + (uint32_t)ra.i * A_SLOT;
            if (NMAT == 2) {
              uint32_t v[32];
              if constexpr (F8) {
                dequant_fp8<4>(mat, r, 4 * h, s2, v);   // the 64 codes of K half h
              } else {
                const uint4 w0 = *reinterpret_cast<const uint4*>(mat + ((h * 2 + 0) * TILE_M + r) * 16);
                const uint4 w1 = *reinterpret_cast<const uint4*>(mat + ((h * 2 + 1) * TILE_M + r) * 16);
                dequant_words(w0, w1, nz_a, nz_b, s2, v);
              }
              tmem_st_32(ta + (uint32_t)(m_own * A_SLOT_COLS), v);
            } else {
              uint32_t v[16];
              if constexpr (F8) {
                dequant_fp8<2>(mat, r, 4 * h + 2 * j_own, s2, v);   // 32 codes: quarter j_own of the half
              } else {
                const uint4 w0 = *reinterpret_cast<const uint4*>(mat + ((h * 2 + j_own) * TILE_M + r) * 16);
                dequant_words16(w0, nz_a, nz_b, s2, v);
              }
              tmem_st_16(ta + (uint32_t)(j_own * 16), v);
            }
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(smem_u32(&S.a_full[ra.i]));
            ra.next();
          }
          if (!ok) break;
          mbar_arrive(smem_u32(&S.raw_empty[rr.i]));
          rr.next();
          ++consumed_raw;
        }
        if (!ok) break;
      }
      // ---- epilogue: one accumulator per item
      ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(S.tmem_full), it_count & 1u, abort_flag, p.err, p.wait_ns));
      if (!ok) break;
      tc_fence_after();
      const int half = wr >> 2;
      const int n_chunks = (it.n_rows + 15) >> 4;
      // quantised weights: token row n entered the MMA as fp16 x * 2^ex_n
      // (b_scale[n] = 2^-ex_n) and h is stored as fp16 h * 2^eh_n, eh_n from ex_n
      // and the expert's bound exponents in the slot trailer (h_row_scale)
      int bsum = 0;
      if constexpr (INT4) {
        const int2 bb = *reinterpret_cast<const int2*>(it.slot + p.trailer_off + 8);
        bsum = bb.x + bb.y;
      }
      for (int c = half; c < n_chunks; c += NHALF) {
        uint32_t acc0[16];
        tmem_ld_16(tl + (uint32_t)(c * 16), acc0);
        const int nv = it.n_rows - c * 16;   // valid token columns of the chunk (> 0)
        // quantised: lane i < 16 works out token i's factors once for the warp
        // (gate/up: x unscale fx = 2^-ex and fu = 2^-ex * 2^eh for up; down:
        // 2^-eh), handed to every lane by shuffles
        float fx = 1.f, fu = 1.f;
        if constexpr (INT4) {
          if (lane < 16 && lane < nv) {
            float inv;
            fx = __ldg(p.b_scale + it.r0 + c * 16 + lane);
            fu = fx * h_row_scale(fx, bsum, &inv);
            if (!GATEUP) fx = inv;
          }
        }
        if (GATEUP) {
          const int f = it.mt * TILE_M + r;   // output feature of this thread
          uint32_t acc1[16];
          tmem_ld_16(tl + (uint32_t)(p.bn + c * 16), acc1);
          tmem_ld_wait();
          const size_t o0 = (size_t)(it.r0 + c * 16) * p.out_ld + f;
          uint16_t* hout = reinterpret_cast<uint16_t*>(p.out);
          // Two tokens per conversion (one packed cvt instead of two scalar
          // ones, which share the quarter-rate unit with the exponentials).
#pragma unroll
          for (int i = 0; i < 16; i += 2) {
            float g0 = __uint_as_float(acc0[i]), u0 = __uint_as_float(acc1[i]);
            float g1 = __uint_as_float(acc0[i + 1]), u1 = __uint_as_float(acc1[i + 1]);
            if constexpr (INT4) {   // undo x's row scale (exact), apply h's (u * 2^-ex * 2^eh)
              g0 *= __shfl_sync(0xffffffffu, fx, i);
              u0 *= __shfl_sync(0xffffffffu, fu, i);
              g1 *= __shfl_sync(0xffffffffu, fx, i + 1);
              u1 *= __shfl_sync(0xffffffffu, fu, i + 1);
            }
            const float h0 = silu_f(g0) * u0, h1 = silu_f(g1) * u1;
            const uint32_t pk = INT4 ? half2_bits_sat(h0, h1) : bf162_bits(h0, h1);
            if (i < nv) hout[o0 + (size_t)i * p.out_ld] = (uint16_t)(pk & 0xFFFFu);
            if (i + 1 < nv) hout[o0 + (size_t)(i + 1) * p.out_ld] = (uint16_t)(pk >> 16);
          }
        } else {
          float* y = reinterpret_cast<float*>(p.out) + (size_t)it.ks * p.out_split_stride;
          uint32_t acc1[16];
          if (PAIR) tmem_ld_16(tl + (uint32_t)(p.bn + c * 16), acc1);
          float hu[16];   // quantised: 2^-eh of each token row (h's scale undone), else 1
#pragma unroll
          for (int i = 0; i < 16; ++i) hu[i] = INT4 ? __shfl_sync(0xffffffffu, fx, i) : 1.f;
          tmem_ld_wait();
#pragma unroll
          for (int m = 0; m < NMAT; ++m) {
            const int f = (PAIR ? 2 * it.mt + m : it.mt) * TILE_M + r;
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              if (i < nv)
                y[(size_t)(it.r0 + c * 16 + i) * p.out_ld + f] = __uint_as_float(m == 0 ? acc0[i] : acc1[i]) * hu[i];
            }
          }
        }
      }
      tc_fence_before();
      mbar_arrive(smem_u32(S.tmem_empty));
      ++it_count;
    }
    if (threadIdx.x == 64) S.misc[3] = consumed_raw;
  }

  // ------------------------------------------------------------ teardown
  __syncthreads();
  volatile int* no_abort = &S.misc[9];   // stays 0: drain waits are bounded by time only
  if (warp == 0 && lane == 0 && *abort_flag) {
    // wait (bounded) for copies that were issued but never consumed
    const int cons[3] = {S.misc[3], S.misc[4], S.misc[5]};
    const int iss[3] = {S.misc[6], S.misc[7], S.misc[8]};
    uint64_t* fulls[3] = {S.raw_full, S.a_full, S.b_full};
    const int ns[3] = {p.n_raw, p.n_a, p.n_b};
    for (int rg = 0; rg < 3; ++rg) {
      if (rg == 0 && !INT4) continue;
      if (rg == 1 && INT4) continue;
      for (int q = cons[rg]; q < iss[rg]; ++q)
        mbar_wait(smem_u32(&fulls[rg][q % ns[rg]]), (uint32_t)((q / ns[rg]) & 1), no_abort, p.err, p.wait_ns);
    }
  }
  if (warp == 1) {   // every MMA this CTA issued has finished
    mma_commit_elect(smem_u32(S.fin));
    mbar_wait(smem_u32(S.fin), 0, no_abort, p.err, p.wait_ns);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, p.tmem_cols);
}

// ------------------------------------------------------------------ host side
GemmPlan plan_gemm_group(int fmt, bool gateup, int bn, int n_groups, int n_mt);
cudaError_t launch_grouped_gemm_group(int fmt, bool gateup, const CUtensorMap& tmap_b, GemmArgs args,
                                      const GemmPlan& plan, int grid, cudaStream_t stream, bool pdl);

GemmPlan plan_gemm(int fmt, bool gateup, int bn, int n_groups, int n_mt) {
  const bool int4 = fmt_quantised(fmt);   // raw blocks dequantised into TMEM
  const int qbytes = int4 ? quant_mat_bytes(fmt) : 0;
  if (gemm_is_group(fmt, bn)) return plan_gemm_group(fmt, gateup, bn, n_groups, n_mt);
  GemmPlan pl{};
  pl.group = false;
  pl.pair = !gateup && down_paired(fmt, n_mt);
  const int nmat = (gateup || pl.pair) ? 2 : 1;
  pl.ndq = int4 ? 8 : 4;
  const size_t budget = 227 * 1024 - 1024;   // opt-in maximum minus the alignment pad
  pl.n_b = bn >= 128 ? 3 : (bn >= 64 ? 4 : 8);
  uint32_t cols = 32;
  if (int4) {
    // A slots in TMEM after the accumulators (nmat * bn columns), 2..4 of them
    const int acc_cols = nmat * bn;
    pl.n_a = (512 - acc_cols) / (nmat * A_SLOT_COLS);
    if (pl.n_a > 4) pl.n_a = 4;
    if (bn >= 128 && pl.n_b < 4) pl.n_b = 4;
    pl.n_raw = 2;
    while (pl.n_raw < 12 &&
           carve_bytes(nmat, qbytes, bn, pl.n_a, pl.n_b, pl.n_raw + 1, n_groups) <= budget)
      ++pl.n_raw;
    while (cols < (uint32_t)(acc_cols + pl.n_a * nmat * A_SLOT_COLS)) cols <<= 1;
  } else {
    pl.n_raw = 0;
    pl.n_a = 2;
    while (pl.n_a < 8 && carve_bytes(nmat, 0, bn, pl.n_a + 1, pl.n_b, 0, n_groups) <= budget)
      ++pl.n_a;
    while (cols < (uint32_t)(nmat * bn)) cols <<= 1;
  }
  pl.smem_bytes = carve_bytes(nmat, qbytes, bn, pl.n_a, pl.n_b, pl.n_raw, n_groups) + 1024;
  pl.tmem_cols = cols;
  return pl;
}

template <int FMT, bool GATEUP, int NDQ, bool PAIR>
static cudaError_t launch_one(const CUtensorMap& tmap, const GemmArgs& a, const GemmPlan& pl,
                              int grid, cudaStream_t s, bool pdl) {
  auto kern = grouped_gemm_kernel<FMT, GATEUP, NDQ, PAIR>;
  static bool attr_set = false;   // per instantiation; the maximum is requested once
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  return launch_kernel(kern, dim3(grid), dim3((2 + NDQ) * 32), pl.smem_bytes, s, pdl, tmap, a);
}

cudaError_t launch_grouped_gemm(int fmt, bool gateup, const CUtensorMap& tmap_b, GemmArgs args,
                                const GemmPlan& plan, int grid, cudaStream_t stream, bool pdl) {
  if (plan.group) return launch_grouped_gemm_group(fmt, gateup, tmap_b, args, plan, grid, stream, pdl);
  args.n_a = plan.n_a;
  args.n_b = plan.n_b;
  args.n_raw = plan.n_raw;
  args.tmem_cols = plan.tmem_cols;
  constexpr int I4 = MOE_W_INT4_G128, F8 = MOE_W_FP8_G128, B16 = MOE_W_BF16;
  if (fmt == I4) {
    if (gateup) return launch_one<I4, true, 8, false>(tmap_b, args, plan, grid, stream, pdl);
    if (plan.pair) {
      args.n_mt /= 2;   // work items name pairs of output tiles
      return launch_one<I4, false, 8, true>(tmap_b, args, plan, grid, stream, pdl);
    }
    return launch_one<I4, false, 8, false>(tmap_b, args, plan, grid, stream, pdl);
  }
  if (fmt == F8) {
    if (gateup) return launch_one<F8, true, 8, false>(tmap_b, args, plan, grid, stream, pdl);
    if (plan.pair) {
      args.n_mt /= 2;
      return launch_one<F8, false, 8, true>(tmap_b, args, plan, grid, stream, pdl);
    }
    return launch_one<F8, false, 8, false>(tmap_b, args, plan, grid, stream, pdl);
  }
  return gateup ? launch_one<B16, true, 4, false>(tmap_b, args, plan, grid, stream, pdl)
                : launch_one<B16, false, 4, false>(tmap_b, args, plan, grid, stream, pdl);
}

}  // namespace moe
