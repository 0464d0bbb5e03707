// gemm_group.cu -- grouped expert GEMM for int4 experts and small row chunks
// (decode-sized batches, <= 32 rows of one expert per work item).
//
// "125B MoE on an RTX 3090 at 100+ tok/s": sec. 3.2 (grouped GEMM over the
// active experts, each a two-layer MLP), sec. 3.1 (per-expert int4 weights with
// their own scale and zero-point, turned into fp16 for the tensor cores without
// a separate pass over memory).
//
// At decode the layer streams int4 weights from HBM; the tensor-core work per
// weight is tiny, so the kernel is built to keep per-byte overheads low:
//   * one pipeline stage = one quantisation group (128 K): one bulk copy of
//     nibbles + scales, one TMA pair for the token rows, 16 MMAs (M = 128 weight
//     rows, N = 16/32 token rows, K = 16) per stage;
//   * the A operand lives in tensor memory: each dequant thread owns one weight
//     row (one TMEM lane) and writes the group's 128 codes with tcgen05.st,
//     so shared memory carries only the nibbles and the small token tiles;
//   * the codes are the biased integers 1024 + q (one LOP3 per pair, exact in
//     fp16); each group accumulates into its own TMEM slice and the dequant
//     warps fold it in two groups later with the group's scale and zero:
//         acc += s * (D_g - (1024 + z) * sum_{k in g} b_k),
//     where sum b_k is the group sum of the token row's fp16 values (computed by
//     the gather kernel for x, by the gate/up epilogue for h);
//   * two MMA warps take alternate groups (each group has its own A stage
//     and accumulator slice, so they never touch the same TMEM), and each
//     prepares its next group's operands while the current MMAs issue: the
//     issue rate of one warp, not the tensor core, bounds small-N MMAs.
//
//   warp 0   producer (bulk copy + TMA), warps 1-2 MMA issuers (warp 1 owns
//   TMEM), warps 3-10 unpack + fold + epilogue (two warps per TMEM lane
//   quadrant: gate/up -> one warp per (matrix, quadrant); down -> the two
//   warps of a quadrant split each row's K quads and the accumulator columns).
//
// Every wait is bounded; on a timeout the CTA drains its copies and MMAs,
// frees TMEM and returns with MOE_DEVERR_TIMEOUT set.
#include "gemm_common.cuh"

namespace moe {

using namespace gemm;

namespace {

constexpr int G_NBUF = 4;     // accumulator slices
constexpr int G_LAG = 2;      // groups between a slice's MMA and its fold
constexpr int G_NA = 2;       // A stages in tensor memory
constexpr int G_MISC = 10;    // [0] tmem [1] abort [2] items [6] raw issued [8] b issued
                              // [9] stays 0
constexpr int G_NMMA = 2;     // MMA-issuing warps (alternate groups)
constexpr int G_NDQ = 8;
constexpr int G_DQ0 = 1 + G_NMMA;                  // first dequant warp
constexpr int G_THREADS = (1 + G_NMMA + G_NDQ) * 32;

struct GShared {
  uint8_t* b_ring;
  uint8_t* raw_ring;
  float* xch;   // gate/up: up accumulators handed to the gate threads [bn][128]
  float* red;   // gate/up: per-quadrant partial sums of h [4][32]
  uint64_t *raw_full, *raw_empty, *a_full, *a_empty, *b_full, *b_empty;
  uint64_t *acc_full, *acc_empty, *xch_bar, *fin;
  int* misc;
  WorkList W;
};

size_t group_carve_bytes(int nmat, int bn, int n_b, int n_raw, int n_groups) {
  size_t s = (size_t)n_b * bn * 256 + (size_t)n_raw * nmat * I4_MAT_BYTES;
  s += (nmat == 2 ? (size_t)TILE_M * bn * 4 : 0) + 4 * 32 * 4;
  s = align_up(s, 16);
  s += 8 * (size_t)(2 * n_raw + 2 * G_NA + 2 * n_b + 2 * G_NBUF + 2 + 1);
  s += 4 * (G_MISC + worklist_ints(n_groups));
  return s;
}

}  // namespace

template <bool GATEUP, int GBN>
__global__ void __launch_bounds__(G_THREADS, 1)
    grouped_gemm_group_kernel(const __grid_constant__ CUtensorMap tmap_b, const GemmArgs p) {
  constexpr int NMAT = GATEUP ? 2 : 1;
  constexpr int CW = GATEUP ? GBN : GBN / 2;           // accumulator columns per dequant thread
  constexpr uint32_t RAW_STAGE = NMAT * I4_MAT_BYTES;
  constexpr uint32_t A_COLS = NMAT * (QGROUP / 2);     // TMEM columns of one A stage
  const uint32_t B_HALF = (uint32_t)GBN * 128u;        // one 64-wide K slice of the token rows
  const uint32_t B_STAGE = 2u * B_HALF;

  extern __shared__ uint8_t smem_dyn[];
  const uint32_t pad = (1024u - (smem_u32(smem_dyn) & 1023u)) & 1023u;
  uint8_t* base = smem_dyn + pad;
  GShared S;
  S.b_ring = base;
  S.raw_ring = S.b_ring + (size_t)p.n_b * B_STAGE;
  uint8_t* cur = S.raw_ring + (size_t)p.n_raw * RAW_STAGE;
  S.xch = reinterpret_cast<float*>(cur);
  cur += (NMAT == 2 ? (size_t)TILE_M * GBN * 4 : 0);
  S.red = reinterpret_cast<float*>(cur);
  cur += 4 * 32 * 4;
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + align_up((size_t)(cur - base), 16));
  S.raw_full = bars;
  S.raw_empty = S.raw_full + p.n_raw;
  S.a_full = S.raw_empty + p.n_raw;
  S.a_empty = S.a_full + G_NA;
  S.b_full = S.a_empty + G_NA;
  S.b_empty = S.b_full + p.n_b;
  S.acc_full = S.b_empty + p.n_b;
  S.acc_empty = S.acc_full + G_NBUF;
  S.xch_bar = S.acc_empty + G_NBUF;
  S.fin = S.xch_bar + 2;
  S.misc = reinterpret_cast<int*>(S.fin + 1);
  S.W.prefix = S.misc + G_MISC;
  S.W.nch = S.W.prefix + (p.n_groups + 1);
  S.W.goff = S.W.nch + (p.n_groups + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int* abort_flag = &S.misc[1];

  // ------------------------------------------------------------ set-up
  if (threadIdx.x == 0) {
    for (int i = 0; i < p.n_raw; ++i) {
      mbar_init(smem_u32(&S.raw_full[i]), 1);
      mbar_init(smem_u32(&S.raw_empty[i]), G_NDQ * 32);
    }
    for (int i = 0; i < G_NA; ++i) {
      mbar_init(smem_u32(&S.a_full[i]), G_NDQ * 32);
      mbar_init(smem_u32(&S.a_empty[i]), 1);
    }
    for (int i = 0; i < p.n_b; ++i) {
      mbar_init(smem_u32(&S.b_full[i]), 1);
      mbar_init(smem_u32(&S.b_empty[i]), 1);
    }
    for (int i = 0; i < G_NBUF; ++i) {
      mbar_init(smem_u32(&S.acc_full[i]), 1);
      mbar_init(smem_u32(&S.acc_empty[i]), G_NDQ * 32);
    }
    for (int i = 0; i < 2; ++i) mbar_init(smem_u32(&S.xch_bar[i]), G_NDQ * 32);
    mbar_init(smem_u32(S.fin), G_NMMA);
    for (int i = 1; i < G_MISC; ++i)
      if (i != 2) S.misc[i] = 0;   // [0] written by tcgen05.alloc, [2] by warp 2
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) prefetch_tensormap(&tmap_b);
  if (warp == 1) {
    tmem_alloc(smem_u32(&S.misc[0]), p.tmem_cols);
    tmem_relinquish();
  }
  if (warp == G_DQ0) {
    const int total = build_worklist(p, S.W, lane);
    if (lane == 0) S.misc[2] = total;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = (uint32_t)S.misc[0];
  const int total = S.misc[2];
  const uint32_t acc0 = (uint32_t)G_NA * A_COLS;   // accumulator slices follow the A stages

  if (warp == 0) {
    // ================================================================ producer
    if (lane == 0) {
      Ring rr{0, 0, p.n_raw}, rb{0, 0, p.n_b};
      int issued_raw = 0, issued_b = 0;
      const uint64_t pol = policy_evict_first();
      bool ok = true;
      for (int item = blockIdx.x; item < total && ok && !*abort_flag; item += gridDim.x) {
        Item it;
        if (!decode_item(item, p, S.W, it)) continue;
        int g0, g1;
        kgroups(p, it.ks, g0, g1);
        const uint8_t* sec = it.slot + p.sec_off;
        for (int kg = g0; kg < g1; ++kg) {
          if (!(ok = mbar_wait(smem_u32(&S.raw_empty[rr.i]), rr.ph ^ 1u, abort_flag, p.err))) break;
          uint32_t bar = smem_u32(&S.raw_full[rr.i]);
          mbar_arrive_expect_tx(bar, RAW_STAGE);
          bulk_g2s_hint(smem_u32(S.raw_ring + (size_t)rr.i * RAW_STAGE),
                        sec + ((size_t)it.mt * (p.K / QGROUP) + kg) * RAW_STAGE, RAW_STAGE, bar, pol);
          rr.next();
          ++issued_raw;
          if (!(ok = mbar_wait(smem_u32(&S.b_empty[rb.i]), rb.ph ^ 1u, abort_flag, p.err))) break;
          bar = smem_u32(&S.b_full[rb.i]);
          mbar_arrive_expect_tx(bar, B_STAGE);
          const uint32_t dst = smem_u32(S.b_ring + (size_t)rb.i * B_STAGE);
          tma_load_2d(dst, &tmap_b, (2 * kg) * KSTEP, it.r0, bar);
          tma_load_2d(dst + B_HALF, &tmap_b, (2 * kg + 1) * KSTEP, it.r0, bar);
          rb.next();
          ++issued_b;
        }
      }
      S.misc[6] = issued_raw;
      S.misc[8] = issued_b;
    }
  } else if (warp < G_DQ0) {
    // ================================================================ MMA issuers
    // Warp 1 + mw issues the groups with (group counter % 2) == mw; their A
    // stage is always mw.  Every ring position and phase follows from the
    // group counter gc, which both warps advance identically.  The whole warp
    // runs the loop; lane 0 issues.
    const int mw = warp - 1;
    uint32_t gc = 0;
    bool ok = true;
    struct Ops {
      uint32_t a[NMAT][8];
      uint64_t b[8];
      uint32_t d[NMAT];
    };
    const uint32_t b_ring0 = smem_u32(S.b_ring);
    auto prep = [&](uint32_t g) -> Ops {
      Ops o;
      const uint32_t bst = b_ring0 + (g % (uint32_t)p.n_b) * B_STAGE;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        o.b[q] = sdesc_kmajor_sw128(bst + (uint32_t)(q >> 2) * B_HALF + (uint32_t)(q & 3) * 32u);
#pragma unroll
        for (int m = 0; m < NMAT; ++m)
          o.a[m][q] = tmem_base + (uint32_t)mw * A_COLS + (uint32_t)(m * (QGROUP / 2) + q * 8);
      }
#pragma unroll
      for (int m = 0; m < NMAT; ++m)
        o.d[m] = tmem_base + acc0 + (g % G_NBUF) * (uint32_t)(NMAT * GBN) + (uint32_t)(m * GBN);
      return o;
    };
    Ops curo = prep((uint32_t)mw);
    for (int item = blockIdx.x; item < total && ok; item += gridDim.x) {
      Item it;
      if (!decode_item(item, p, S.W, it)) continue;
      int g0, g1;
      kgroups(p, it.ks, g0, g1);
      const uint32_t idesc = idesc_f16kind_f32(TILE_M, (uint32_t)((it.n_rows + 15) & ~15), 0u);
      for (int kg = g0; kg < g1; ++kg, ++gc) {
        if ((int)(gc & 1u) != mw) continue;
        const uint32_t bi = gc % (uint32_t)p.n_b;
        if (!(ok = mbar_wait(smem_u32(&S.acc_empty[gc % G_NBUF]), ((gc / G_NBUF) & 1u) ^ 1u,
                             abort_flag, p.err)))
          break;
        if (!(ok = mbar_wait(smem_u32(&S.a_full[mw]), (gc / G_NA) & 1u, abort_flag, p.err))) break;
        if (!(ok = mbar_wait(smem_u32(&S.b_full[bi]), (gc / (uint32_t)p.n_b) & 1u, abort_flag, p.err)))
          break;
        tc_fence_after();
        const Ops nxt = prep(gc + G_NMMA);
        if (lane == 0) {
#pragma unroll
          for (int q = 0; q < 8; ++q)
#pragma unroll
            for (int m = 0; m < NMAT; ++m)
              mma_f16kind_ta(curo.d[m], curo.a[m][q], curo.b[q], idesc, q > 0 ? 1u : 0u);
          mma_commit(smem_u32(&S.a_empty[mw]));
          mma_commit(smem_u32(&S.b_empty[bi]));
          mma_commit(smem_u32(&S.acc_full[gc % G_NBUF]));
        }
        __syncwarp();
        curo = nxt;
      }
    }
  } else {
    // ================================================================ dequant + fold + epilogue
    const int wr = warp - G_DQ0;
    const int quad = warp & 3;               // TMEM lane quadrant of this warp
    const int r = quad * 32 + lane;          // weight row of the tile = TMEM lane
    const int m_own = GATEUP ? (wr >> 2) : 0;
    const int j_own = GATEUP ? 0 : (wr >> 2);
    const uint32_t lane_base = tmem_base + ((uint32_t)(quad * 32) << 16);
    Ring ra{0, 0, G_NA}, rr{0, 0, p.n_raw};
    uint32_t it_count = 0, gc = 0;
    bool ok = true;
    for (int item = blockIdx.x; item < total && ok; item += gridDim.x) {
      Item it;
      if (!decode_item(item, p, S.W, it)) continue;
      int g0, g1;
      kgroups(p, it.ks, g0, g1);
      const int cbeg = GATEUP ? 0 : j_own * (GBN / 2);
      const int nc = max(0, min(CW, it.n_rows - cbeg));
      float acc[CW];
#pragma unroll
      for (int i = 0; i < CW; ++i) acc[i] = 0.f;
      float bpre[CW];
      auto prefetch_sums = [&](int kg) {
        const float* bs = p.bsum + (size_t)kg * p.rows_total + it.r0 + cbeg;
#pragma unroll
        for (int i = 0; i < CW; ++i) bpre[i] = (i < nc) ? __ldg(bs + i) : 0.f;
      };
      auto fold = [&](float s, float c) -> bool {
        const uint32_t buf = gc % G_NBUF;
        const uint32_t ta = lane_base + acc0 + buf * (uint32_t)(NMAT * GBN) + (uint32_t)(m_own * GBN + cbeg);
        if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&S.acc_full[buf]), (gc / G_NBUF) & 1u,
                                               abort_flag, p.err)))
          return false;
        tc_fence_after();
        uint32_t d[CW];
#pragma unroll
        for (int ch = 0; ch < CW / 8; ++ch)
          if (ch * 8 < nc) tmem_ld_8(ta + ch * 8, *reinterpret_cast<uint32_t(*)[8]>(&d[ch * 8]));
        tmem_ld_wait();
        tc_fence_before();
        mbar_arrive(smem_u32(&S.acc_empty[buf]));
#pragma unroll
        for (int i = 0; i < CW; ++i)
          if (i < nc) acc[i] = fmaf(s, fmaf(-c, bpre[i], __uint_as_float(d[i])), acc[i]);
        ++gc;
        return true;
      };
      int np = 0, pk0 = 0, pk1 = 0;
      float ps0 = 0.f, pc0 = 0.f, ps1 = 0.f, pc1 = 0.f;

      for (int kg = g0; kg < g1 && ok; ++kg) {
        if (np == G_LAG) prefetch_sums(pk0);
        if (!(ok = __all_sync(0xffffffffu,
                              mbar_wait(smem_u32(&S.raw_full[rr.i]), rr.ph, abort_flag, p.err))))
          break;
        const uint8_t* mat = S.raw_ring + (size_t)rr.i * RAW_STAGE + m_own * I4_MAT_BYTES;
        const uint32_t sz = *reinterpret_cast<const uint32_t*>(mat + I4_PACKED_BYTES + r * 4);
        const float s = __half2float(__ushort_as_half((unsigned short)(sz & 0xFFFFu)));
        const float c = 1024.f + __half2float(__ushort_as_half((unsigned short)(sz >> 16)));
        const uint32_t ta = lane_base + (uint32_t)ra.i * A_COLS + (uint32_t)(m_own * (QGROUP / 2));
        if (!(ok = __all_sync(0xffffffffu,
                              mbar_wait(smem_u32(&S.a_empty[ra.i]), ra.ph ^ 1u, abort_flag, p.err))))
          break;
        tc_fence_after();
#pragma unroll
        for (int h = 0; h < 2; ++h) {   // K halves of the group: 64 codes of my row each
          if (GATEUP) {
            uint32_t v[32];
#pragma unroll
            for (int j = 0; j < 2; ++j) {
              const uint4 wq = *reinterpret_cast<const uint4*>(mat + ((h * 2 + j) * TILE_M + r) * 16);
              codes_of_word(wq.x, &v[j * 16 + 0]);
              codes_of_word(wq.y, &v[j * 16 + 4]);
              codes_of_word(wq.z, &v[j * 16 + 8]);
              codes_of_word(wq.w, &v[j * 16 + 12]);
            }
            tmem_st_32(ta + (uint32_t)(h * 32), v);
          } else {
            uint32_t v[16];
            const uint4 wq = *reinterpret_cast<const uint4*>(mat + ((h * 2 + j_own) * TILE_M + r) * 16);
            codes_of_word(wq.x, &v[0]);
            codes_of_word(wq.y, &v[4]);
            codes_of_word(wq.z, &v[8]);
            codes_of_word(wq.w, &v[12]);
            tmem_st_16(ta + (uint32_t)(h * 32 + j_own * 16), v);
          }
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(smem_u32(&S.a_full[ra.i]));
        ra.next();
        mbar_arrive(smem_u32(&S.raw_empty[rr.i]));
        rr.next();
        // fold the group G_LAG behind this one, then queue this one
        if (np == G_LAG) {
          if (!(ok = fold(ps0, pc0))) break;
          pk0 = pk1; ps0 = ps1; pc0 = pc1;
          np = G_LAG - 1;
        }
        if (np == 0) { pk0 = kg; ps0 = s; pc0 = c; } else { pk1 = kg; ps1 = s; pc1 = c; }
        ++np;
      }
      while (ok && np > 0) {
        prefetch_sums(pk0);
        if (!(ok = fold(ps0, pc0))) break;
        pk0 = pk1; ps0 = ps1; pc0 = pc1;
        --np;
      }
      if (!ok) break;

      // ---- item epilogue from the register accumulators
      if (GATEUP) {
        // hand-offs among the dequant warps use bounded mbarrier waits (not
        // bar.sync), so a warp that aborted cannot leave the others blocked
        const uint32_t xpar = it_count & 1u;
        if (m_own == 1) {
#pragma unroll
          for (int i = 0; i < CW; ++i)
            if (i < nc) S.xch[i * TILE_M + r] = acc[i];
        }
        mbar_arrive(smem_u32(&S.xch_bar[0]));
        if (!(ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&S.xch_bar[0]), xpar, abort_flag, p.err))))
          break;
        if (m_own == 0) {
          __half* hout = reinterpret_cast<__half*>(p.out);
          const int f = it.mt * TILE_M + r;
#pragma unroll
          for (int i = 0; i < CW; ++i) {
            if (i < nc) {
              const __half hv = to_half_sat(silu_f(acc[i]) * S.xch[i * TILE_M + r]);
              hout[(size_t)(it.r0 + i) * p.out_ld + f] = hv;
              float v = __half2float(hv);   // sum of the rounded values the down GEMM reads
#pragma unroll
              for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
              if (lane == 0) S.red[quad * 32 + i] = v;
            }
          }
        }
        mbar_arrive(smem_u32(&S.xch_bar[1]));
        if (!(ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&S.xch_bar[1]), xpar, abort_flag, p.err))))
          break;
        if (m_own == 0 && quad == 0 && lane < nc)
          p.hsum_out[(size_t)it.mt * p.rows_total + it.r0 + lane] =
              S.red[lane] + S.red[32 + lane] + S.red[64 + lane] + S.red[96 + lane];
      } else {
        float* y = reinterpret_cast<float*>(p.out) + (size_t)it.ks * p.out_split_stride;
        const int f = it.mt * TILE_M + r;
#pragma unroll
        for (int i = 0; i < CW; ++i)
          if (i < nc) y[(size_t)(it.r0 + cbeg + i) * p.out_ld + f] = acc[i];
      }
      ++it_count;
    }
  }

  // ------------------------------------------------------------ teardown
  __syncthreads();
  volatile int* no_abort = &S.misc[9];   // stays 0: drain waits are bounded by time only
  if (warp == 0 && lane == 0 && *abort_flag) {
    // for each ring slot, wait (bounded) for the last copy issued into it; an
    // earlier copy into the same slot had landed before the slot was reused
    const int iss_raw = S.misc[6], iss_b = S.misc[8];
    for (int sl = 0; sl < p.n_raw && sl < iss_raw; ++sl) {
      const int q = sl + ((iss_raw - 1 - sl) / p.n_raw) * p.n_raw;
      mbar_wait(smem_u32(&S.raw_full[sl]), (uint32_t)((q / p.n_raw) & 1), no_abort, p.err);
    }
    for (int sl = 0; sl < p.n_b && sl < iss_b; ++sl) {
      const int q = sl + ((iss_b - 1 - sl) / p.n_b) * p.n_b;
      mbar_wait(smem_u32(&S.b_full[sl]), (uint32_t)((q / p.n_b) & 1), no_abort, p.err);
    }
  }
  if (warp >= 1 && warp < G_DQ0 && lane == 0) {   // every MMA this CTA issued has finished
    mma_commit(smem_u32(S.fin));
    mbar_wait(smem_u32(S.fin), 0, no_abort, p.err);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, p.tmem_cols);
}

// ------------------------------------------------------------------ host side
GemmPlan plan_gemm_group(bool gateup, int bn, int n_groups) {
  GemmPlan pl{};
  const int nmat = gateup ? 2 : 1;
  pl.group = true;
  pl.ndq = G_NDQ;
  pl.n_a = G_NA;
  pl.n_b = 8;
  const size_t budget = 227 * 1024 - 1024;
  pl.n_raw = 2;
  while (pl.n_raw < 16 && group_carve_bytes(nmat, bn, pl.n_b, pl.n_raw + 1, n_groups) <= budget)
    ++pl.n_raw;
  pl.smem_bytes = group_carve_bytes(nmat, bn, pl.n_b, pl.n_raw, n_groups) + 1024;
  const uint32_t need = (uint32_t)(G_NA * nmat * (QGROUP / 2) + G_NBUF * nmat * bn);
  uint32_t cols = 32;
  while (cols < need) cols <<= 1;
  pl.tmem_cols = cols;
  return pl;
}

template <bool GATEUP, int GBN>
static cudaError_t launch_group_one(const CUtensorMap& tmap, const GemmArgs& a, const GemmPlan& pl,
                                    int grid, cudaStream_t s) {
  auto kern = grouped_gemm_group_kernel<GATEUP, GBN>;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  kern<<<grid, G_THREADS, pl.smem_bytes, s>>>(tmap, a);
  return cudaGetLastError();
}

cudaError_t launch_grouped_gemm_group(bool gateup, const CUtensorMap& tmap_b, GemmArgs args,
                                      const GemmPlan& plan, int grid, cudaStream_t stream) {
  args.n_a = plan.n_a;
  args.n_b = plan.n_b;
  args.n_raw = plan.n_raw;
  args.tmem_cols = plan.tmem_cols;
  if (args.bn == 16)
    return gateup ? launch_group_one<true, 16>(tmap_b, args, plan, grid, stream)
                  : launch_group_one<false, 16>(tmap_b, args, plan, grid, stream);
  return gateup ? launch_group_one<true, 32>(tmap_b, args, plan, grid, stream)
                : launch_group_one<false, 32>(tmap_b, args, plan, grid, stream);
}

}  // namespace moe
