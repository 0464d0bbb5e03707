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
//     nibbles + scales and one TMA pair for the token rows, all on one
//     barrier; 8 K16 steps of M = 128 weight rows x N = 16/32 token rows;
//   * the A operand lives in tensor memory: each unpack thread owns one weight
//     row (one TMEM lane) and writes the group's codes with tcgen05.st, so
//     shared memory carries only the nibbles and the small token tiles;
//   * the codes are q - z, exact in fp16 (a LOP3 into the fp16 pattern of
//     1024, then one fp16 add or FMA); each group accumulates into its own
//     TMEM slice, folded into fp32 registers with the group's scale:
//     acc += s * D_g;
//   * the warps that feed the MMAs (unpack) and the warps that consume them
//     (fold + epilogue) are separate, each running a short per-group chain:
//     unpack waits for the stage and a free A slot, fold waits for the
//     group's accumulator; item epilogues never stall the unpacking;
//   * two MMA warps take alternate groups and issue from a converged warp
//     (elect.sync): their issue rate, not the tensor core, bounds small-N
//     MMAs; 3 A slots where tensor memory allows (2 otherwise).
//
//   warp 0       producer (bulk copy + TMA)
//   warps 1-2    MMA issuers (warp 1 owns TMEM)
//   warps 3-10   unpack, two per TMEM lane quadrant: in the two-matrix modes
//                each writes one matrix's codes for its quadrant's rows, in
//                single down each writes one K quad of each half
//   warps 11-14  fold + epilogue, one per quadrant: every matrix and token
//                column of its 32 rows
// Modes: gate/up (a stage holds the gate and up rows of one output tile;
// SwiGLU epilogue), paired down (two adjacent 128-row output tiles sharing the
// token tile), single down (one tile).
//
// Every wait is bounded; on a timeout the CTA drains its copies and MMAs,
// frees TMEM and returns with MOE_DEVERR_TIMEOUT set.
#include "gemm_common.cuh"

namespace moe {

using namespace gemm;

namespace {

constexpr int G_NBUF = 4;     // accumulator slices: group g uses slice g % 4
constexpr int G_MAX_NA = 3;   // A slots in tensor memory (3 where the columns allow)
constexpr int G_MISC = 8;     // [0] tmem [1] abort [2] items [3] stages issued [4] stays 0
constexpr int G_NMMA = 2;     // MMA-issuing warps (alternate groups)
constexpr int G_NUP = 8;      // unpack warps
constexpr int G_NFOLD = 4;    // fold + epilogue warps
constexpr int G_UP0 = 1 + G_NMMA;                  // first unpack warp
constexpr int G_FOLD0 = G_UP0 + G_NUP;             // first fold warp
constexpr int G_THREADS = (G_FOLD0 + G_NFOLD) * 32;

enum GroupMode { G_GATEUP = 0, G_DOWN_PAIR = 1, G_DOWN = 2 };

// A work item decoded once per CTA (the decode needs integer divisions by
// run-time values, which every warp would otherwise repeat).
struct ItemDesc {
  const uint8_t* slot;   // nullptr: the item is skipped (bad expert slot)
  int g0, g1;            // quantisation groups [g0, g1) of its K split
  int r0, n_rows;        // token rows
  int mt, ks;            // output tile (pair) and K split
};
constexpr int G_ITEM_TAB = 64;   // items per CTA kept in the table; later ones are decoded on the fly

struct GShared {
  ItemDesc* items;     // [G_ITEM_TAB]
  uint8_t* b_ring;     // [n_st][2 * bn * 128]  token rows, SW128 K-major (1024-aligned stages)
  uint8_t* raw_ring;   // [n_st][nmat * I4_MAT_BYTES]  nibbles + scale/zero words
  uint64_t *full, *empty;          // stages: producer -> consumers, consumers -> producer
  uint64_t *a_full, *a_empty;      // A slots: unpack -> MMA, MMA (commit) -> unpack
  uint64_t *acc_full, *acc_empty;  // accumulator slices: MMA (commit) -> fold, fold -> MMA
  uint64_t* fin;
  int* misc;
  WorkList W;
};

size_t group_carve_bytes(int nmat, int bn, int n_st, int n_groups) {
  size_t s = (size_t)n_st * ((size_t)bn * 256 + (size_t)nmat * I4_MAT_BYTES);
  s += sizeof(ItemDesc) * G_ITEM_TAB;
  s = align_up(s, 16);
  s += 8 * (size_t)(2 * n_st + 2 * G_MAX_NA + 2 * G_NBUF + 1);
  s += 4 * (G_MISC + worklist_ints(n_groups));
  return s;
}

__device__ __forceinline__ ItemDesc make_item_desc(int item, const GemmArgs& p, const WorkList& W) {
  ItemDesc d;
  Item it;
  d.slot = decode_item(item, p, W, it) ? it.slot : nullptr;
  kgroups(p, it.ks, d.g0, d.g1);
  d.r0 = it.r0;
  d.n_rows = it.n_rows;
  d.mt = it.mt;
  d.ks = it.ks;
  return d;
}

// The CTA's i-th item (item index blockIdx.x + i * gridDim.x).
__device__ __forceinline__ ItemDesc get_item(int i, const GemmArgs& p, const GShared& S) {
  if (i < G_ITEM_TAB) return S.items[i];
  return make_item_desc(blockIdx.x + i * gridDim.x, p, S.W);
}

__device__ __forceinline__ bool wait_all(uint32_t bar, uint32_t parity, volatile int* abort_flag, int* err) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort_flag, err));
}

}  // namespace

template <int MODE, int GBN>
__global__ void __launch_bounds__(G_THREADS, 1)
    grouped_gemm_group_kernel(const __grid_constant__ CUtensorMap tmap_b, const GemmArgs p) {
  constexpr bool GATEUP = MODE == G_GATEUP;
  constexpr bool PAIR = MODE != G_DOWN;                // two 128-row matrices per stage
  constexpr int NMAT = PAIR ? 2 : 1;
  constexpr uint32_t RAW_STAGE = NMAT * I4_MAT_BYTES;
  constexpr uint32_t A_COLS = NMAT * (QGROUP / 2);     // TMEM columns of one A slot
  constexpr uint32_t B_HALF = (uint32_t)GBN * 128u;    // one 64-wide K slice of the token rows
  constexpr uint32_t B_STAGE = 2u * B_HALF;
  // A slots: 3 where they fit beside the 4 accumulator slices in 512 columns
  constexpr int NA = (3 * A_COLS + G_NBUF * NMAT * GBN <= 512) ? 3 : 2;
  const int n_st = p.n_raw;

  extern __shared__ uint8_t smem_dyn[];
  const uint32_t pad = (1024u - (smem_u32(smem_dyn) & 1023u)) & 1023u;
  uint8_t* base = smem_dyn + pad;
  GShared S;
  S.b_ring = base;
  S.raw_ring = S.b_ring + (size_t)n_st * B_STAGE;
  uint8_t* cur = S.raw_ring + (size_t)n_st * RAW_STAGE;
  S.items = reinterpret_cast<ItemDesc*>(cur);
  cur += sizeof(ItemDesc) * G_ITEM_TAB;
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + align_up((size_t)(cur - base), 16));
  S.full = bars;
  S.empty = S.full + n_st;
  S.a_full = S.empty + n_st;
  S.a_empty = S.a_full + G_MAX_NA;
  S.acc_full = S.a_empty + G_MAX_NA;
  S.acc_empty = S.acc_full + G_NBUF;
  S.fin = S.acc_empty + G_NBUF;
  S.misc = reinterpret_cast<int*>(S.fin + 1);
  S.W.prefix = S.misc + G_MISC;
  S.W.nch = S.W.prefix + (p.n_groups + 1);
  S.W.goff = S.W.nch + (p.n_groups + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int* abort_flag = &S.misc[1];

  // ------------------------------------------------------------ set-up
  if (threadIdx.x == 0) {
    for (int i = 0; i < n_st; ++i) {
      mbar_init(smem_u32(&S.full[i]), 1);
      mbar_init(smem_u32(&S.empty[i]), (G_NUP + G_NFOLD) * 32);
    }
    for (int i = 0; i < G_MAX_NA; ++i) {
      mbar_init(smem_u32(&S.a_full[i]), G_NUP * 32);
      mbar_init(smem_u32(&S.a_empty[i]), 1);
    }
    for (int i = 0; i < G_NBUF; ++i) {
      mbar_init(smem_u32(&S.acc_full[i]), 1);
      mbar_init(smem_u32(&S.acc_empty[i]), G_NFOLD * 32);
    }
    mbar_init(smem_u32(S.fin), G_NMMA);
    for (int i = 1; i < G_MISC; ++i)
      if (i != 2) S.misc[i] = 0;   // [0] written by tcgen05.alloc, [2] by the first unpack warp
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
  if (warp == G_UP0) {
    const int total = build_worklist(p, S.W, lane);
    __syncwarp();
    const int n_mine = total > (int)blockIdx.x ? (total - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x : 0;
    for (int i = lane; i < n_mine && i < G_ITEM_TAB; i += 32)
      S.items[i] = make_item_desc(blockIdx.x + i * gridDim.x, p, S.W);
    if (lane == 0) S.misc[2] = n_mine;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = (uint32_t)S.misc[0];
  const int n_mine = S.misc[2];   // items of this CTA
  const uint32_t acc0 = NA * A_COLS;   // accumulator slices follow the A slots

  if (warp == 0) {
    // ================================================================ producer
    // Per group one stage: the NMAT nibble blocks and the two 64-wide K
    // slices of the token rows, on one barrier.  In the paired down mode the
    // item's tile index mt names the output tiles 2mt and 2mt + 1.
    if (lane == 0) {
      Ring rs{0, 0, n_st};
      int issued = 0;
      const uint64_t pol = policy_evict_first();
      bool ok = true;
      for (int ii = 0; ii < n_mine && ok && !*abort_flag; ++ii) {
        const ItemDesc it = get_item(ii, p, S);
        if (!it.slot) continue;
        const int g0 = it.g0, g1 = it.g1;
        const uint8_t* sec = it.slot + p.sec_off;
        for (int kg = g0; kg < g1; ++kg) {
          if (!(ok = mbar_wait(smem_u32(&S.empty[rs.i]), rs.ph ^ 1u, abort_flag, p.err))) break;
          const uint32_t bar = smem_u32(&S.full[rs.i]);
          mbar_arrive_expect_tx(bar, RAW_STAGE + B_STAGE);
          const uint32_t raw = smem_u32(S.raw_ring + (size_t)rs.i * RAW_STAGE);
          if (MODE == G_DOWN_PAIR) {
#pragma unroll
            for (int m = 0; m < 2; ++m)
              bulk_g2s_hint(raw + m * I4_MAT_BYTES,
                            sec + ((size_t)(2 * it.mt + m) * (p.K / QGROUP) + kg) * I4_MAT_BYTES,
                            I4_MAT_BYTES, bar, pol);
          } else {
            bulk_g2s_hint(raw, sec + ((size_t)it.mt * (p.K / QGROUP) + kg) * RAW_STAGE, RAW_STAGE, bar,
                          pol);
          }
          const uint32_t dst = smem_u32(S.b_ring + (size_t)rs.i * B_STAGE);
          tma_load_2d(dst, &tmap_b, (2 * kg) * KSTEP, it.r0, bar);
          tma_load_2d(dst + B_HALF, &tmap_b, (2 * kg + 1) * KSTEP, it.r0, bar);
          rs.next();
          ++issued;
        }
      }
      S.misc[3] = issued;
    }
  } else if (warp < G_UP0) {
    // ================================================================ MMA issuers
    // Warp 1 + mw issues the groups with (group counter % 2) == mw.  Group gc
    // uses A slot gc % NA and accumulator slice gc % 4.  a_full(gc) also
    // implies that the group's stage (token tile) has landed: the unpack
    // threads arrive only after seeing it.  The whole warp runs the loop;
    // ring positions advance by one per group, owned or not.
    const int mw = warp - 1;
    uint32_t gc = 0;
    bool ok = true;
    Ring rs{0, 0, n_st}, ra{0, 0, NA};
    const uint64_t bdesc0 = sdesc_kmajor_sw128(smem_u32(S.b_ring));   // stage 0, K step 0
    for (int ii = 0; ii < n_mine && ok; ++ii) {
      const ItemDesc it = get_item(ii, p, S);
      if (!it.slot) continue;
      const int g0 = it.g0, g1 = it.g1;
      const uint32_t idesc = idesc_f16kind_f32(TILE_M, (uint32_t)((it.n_rows + 15) & ~15), 0u);
      for (int kg = g0; kg < g1; ++kg, ++gc, rs.next(), ra.next()) {
        if ((int)(gc & 1u) != mw) continue;
        const uint32_t bi = gc % G_NBUF;
        if (!(ok = wait_all(smem_u32(&S.a_full[ra.i]), ra.ph, abort_flag, p.err))) break;
        if (!(ok = wait_all(smem_u32(&S.acc_empty[bi]), ((gc / G_NBUF) & 1u) ^ 1u, abort_flag, p.err)))
          break;
        tc_fence_after();
        // the descriptor's start-address field counts 16-byte units
        const uint64_t bd = bdesc0 + (uint64_t)(((uint32_t)rs.i * B_STAGE) >> 4);
        const uint32_t a_base = tmem_base + (uint32_t)ra.i * A_COLS;
        const uint32_t d0 = tmem_base + acc0 + bi * (uint32_t)(NMAT * GBN);
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const uint64_t bq = bd + (uint64_t)(((q >> 2) * B_HALF + (q & 3) * 32) >> 4);
          if (NMAT == 2)
            mma2_ta_elect(d0, d0 + GBN, a_base + q * 8, a_base + (QGROUP / 2) + q * 8, bq, idesc,
                          q > 0 ? 1u : 0u);
          else
            mma_ta_elect(d0, a_base + q * 8, bq, idesc, q > 0 ? 1u : 0u);
        }
        mma_commit_elect(smem_u32(&S.a_empty[ra.i]));
        mma_commit_elect(smem_u32(&S.acc_full[bi]));
      }
    }
  } else if (warp < G_FOLD0) {
    // ================================================================ unpack
    // Group gc: wait for its stage and for A slot gc % NA to be free (the
    // MMAs of group gc - NA are done), both tested one group ahead; write
    // the codes; hand the slot to the MMA warp; release my reads of the stage.
    const int wr = warp - G_UP0;
    const int quad = warp & 3;               // TMEM lane quadrant of this warp
    const int r = quad * 32 + lane;          // weight row of the tile = TMEM lane
    const int hw = wr >> 2;                  // which of the quadrant's two unpack warps
    const int m_own = PAIR ? hw : 0;         // matrix ...
    const int j_own = PAIR ? 0 : hw;         // ... and K quad of each half (single down)
    const uint32_t lane_base = tmem_base + ((uint32_t)(quad * 32) << 16);
    Ring rs{0, 0, n_st}, ra{0, 0, NA};
    bool ok = true, full_ready = false, a_ready = false;
    for (int ii = 0; ii < n_mine && ok; ++ii) {
      const ItemDesc it = get_item(ii, p, S);
      if (!it.slot) continue;
      const int g0 = it.g0, g1 = it.g1;
      for (int kg = g0; kg < g1 && ok; ++kg) {
        if (!full_ready && !(ok = wait_all(smem_u32(&S.full[rs.i]), rs.ph, abort_flag, p.err))) break;
        if (!a_ready && !(ok = wait_all(smem_u32(&S.a_empty[ra.i]), ra.ph ^ 1u, abort_flag, p.err))) break;
        tc_fence_after();
        const uint8_t* mat = S.raw_ring + (size_t)rs.i * RAW_STAGE + m_own * I4_MAT_BYTES;
        const uint32_t sz = *reinterpret_cast<const uint32_t*>(mat + I4_PACKED_BYTES + r * 4);
        const float zf = __half2float(__ushort_as_half((unsigned short)(sz >> 16)));
        const __half2 za = __float2half2_rn(-(1024.f + zf)), zb = __float2half2_rn(-(64.f + zf));
        const uint32_t nz_a = *reinterpret_cast<const uint32_t*>(&za);
        const uint32_t nz_b = *reinterpret_cast<const uint32_t*>(&zb);
        const uint32_t ta = lane_base + (uint32_t)ra.i * A_COLS + (uint32_t)(m_own * (QGROUP / 2));
#pragma unroll
        for (int h = 0; h < 2; ++h) {   // K halves of the group: 64 codes of my row each
          if (PAIR) {
            uint32_t v[32];
#pragma unroll
            for (int jj = 0; jj < 2; ++jj) {
              const uint4 wq = *reinterpret_cast<const uint4*>(mat + ((h * 2 + jj) * TILE_M + r) * 16);
              codes_minus_zero(wq.x, nz_a, nz_b, &v[jj * 16 + 0]);
              codes_minus_zero(wq.y, nz_a, nz_b, &v[jj * 16 + 4]);
              codes_minus_zero(wq.z, nz_a, nz_b, &v[jj * 16 + 8]);
              codes_minus_zero(wq.w, nz_a, nz_b, &v[jj * 16 + 12]);
            }
            tmem_st_32(ta + (uint32_t)(h * 32), v);
          } else {
            uint32_t v[16];
            const uint4 wq = *reinterpret_cast<const uint4*>(mat + ((h * 2 + j_own) * TILE_M + r) * 16);
            codes_minus_zero(wq.x, nz_a, nz_b, &v[0]);
            codes_minus_zero(wq.y, nz_a, nz_b, &v[4]);
            codes_minus_zero(wq.z, nz_a, nz_b, &v[8]);
            codes_minus_zero(wq.w, nz_a, nz_b, &v[12]);
            tmem_st_16(ta + (uint32_t)(h * 32 + j_own * 16), v);
          }
        }
        mbar_arrive(smem_u32(&S.empty[rs.i]));   // my reads of the stage are done
        {   // while the stores drain, test what the next group waits for
          Ring ns = rs, na = ra;
          ns.next();
          na.next();
          const uint32_t t = __reduce_and_sync(
              0xffffffffu, mbar_test_wait2(smem_u32(&S.full[ns.i]), ns.ph, smem_u32(&S.a_empty[na.i]),
                                           na.ph ^ 1u));
          full_ready = (t & 1u) != 0;
          a_ready = (t & 2u) != 0;
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(smem_u32(&S.a_full[ra.i]));
        rs.next();
        ra.next();
      }
    }
  } else {
    // ================================================================ fold + epilogue
    // One warp per TMEM lane quadrant; each thread owns weight row r of every
    // matrix and all the item's token columns.  Group gc: wait for its
    // accumulator slice, fold it with the group's scales (read from the
    // stage, which this warp releases afterwards), free the slice.
    const int quad = warp & 3;
    const int r = quad * 32 + lane;
    const uint32_t lane_base = tmem_base + ((uint32_t)(quad * 32) << 16);
    constexpr int CH = 16;   // columns per tcgen05.ld
    Ring rs{0, 0, n_st};
    uint32_t gc = 0;
    bool ok = true;
    for (int ii = 0; ii < n_mine && ok; ++ii) {
      const ItemDesc it = get_item(ii, p, S);
      if (!it.slot) continue;
      const int g0 = it.g0, g1 = it.g1;
      const int nc = it.n_rows;   // token columns of this item (<= GBN)
      float acc[NMAT][GBN];
#pragma unroll
      for (int m = 0; m < NMAT; ++m)
#pragma unroll
        for (int i = 0; i < GBN; ++i) acc[m][i] = 0.f;
      for (int kg = g0; kg < g1 && ok; ++kg, ++gc) {
        const uint32_t bi = gc % G_NBUF;
        if (!(ok = wait_all(smem_u32(&S.full[rs.i]), rs.ph, abort_flag, p.err))) break;
        const uint8_t* raw = S.raw_ring + (size_t)rs.i * RAW_STAGE;
        float sc[NMAT];
#pragma unroll
        for (int m = 0; m < NMAT; ++m)
          sc[m] = __half2float(__ushort_as_half(
              *reinterpret_cast<const unsigned short*>(raw + m * I4_MAT_BYTES + I4_PACKED_BYTES + r * 4)));
        if (!(ok = wait_all(smem_u32(&S.acc_full[bi]), (gc / G_NBUF) & 1u, abort_flag, p.err))) break;
        tc_fence_after();
        const uint32_t ta = lane_base + acc0 + bi * (uint32_t)(NMAT * GBN);
#pragma unroll
        for (int m = 0; m < NMAT; ++m) {
#pragma unroll
          for (int ch = 0; ch < GBN / CH; ++ch) {
            if (ch * CH < nc) {
              uint32_t d[CH];
              tmem_ld_16(ta + (uint32_t)(m * GBN + ch * CH), d);
              tmem_ld_wait_regs(d);
#pragma unroll
              for (int i = 0; i < CH; ++i)
                acc[m][ch * CH + i] = fmaf(sc[m], __uint_as_float(d[i]), acc[m][ch * CH + i]);
            }
          }
        }
        tc_fence_before();
        mbar_arrive(smem_u32(&S.acc_empty[bi]));
        mbar_arrive(smem_u32(&S.empty[rs.i]));
        rs.next();
      }
      if (!ok) break;

      // ---- item epilogue from the register accumulators
      if (GATEUP) {
        __half* hout = reinterpret_cast<__half*>(p.out);
        const int f = it.mt * TILE_M + r;
#pragma unroll
        for (int i = 0; i < GBN; ++i)
          if (i < nc) hout[(size_t)(it.r0 + i) * p.out_ld + f] = to_half_sat(silu_f(acc[0][i]) * acc[1][i]);
      } else {
        float* y = reinterpret_cast<float*>(p.out) + (size_t)it.ks * p.out_split_stride;
#pragma unroll
        for (int m = 0; m < NMAT; ++m) {
          const int f = (MODE == G_DOWN_PAIR ? 2 * it.mt + m : it.mt) * TILE_M + r;
#pragma unroll
          for (int i = 0; i < GBN; ++i)
            if (i < nc) y[(size_t)(it.r0 + i) * p.out_ld + f] = acc[m][i];
        }
      }
    }
  }

  // ------------------------------------------------------------ teardown
  __syncthreads();
  volatile int* no_abort = &S.misc[4];   // stays 0: drain waits are bounded by time only
  if (warp == 0 && lane == 0 && *abort_flag) {
    // for each stage, wait (bounded) for the last copies issued into it; an
    // earlier fill of the same stage had landed before the stage was reused
    const int iss = S.misc[3];
    for (int sl = 0; sl < n_st && sl < iss; ++sl) {
      const int q = sl + ((iss - 1 - sl) / n_st) * n_st;
      mbar_wait(smem_u32(&S.full[sl]), (uint32_t)((q / n_st) & 1), no_abort, p.err);
    }
  }
  if (warp >= 1 && warp < G_UP0) {   // every MMA this CTA issued has finished
    mma_commit_elect(smem_u32(S.fin));
    mbar_wait(smem_u32(S.fin), 0, no_abort, p.err);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, p.tmem_cols);
}

// ------------------------------------------------------------------ host side
GemmPlan plan_gemm_group(bool gateup, int bn, int n_groups, int n_mt) {
  GemmPlan pl{};
  pl.group = true;
  pl.pair = !gateup && down_paired(MOE_W_INT4_G128, n_mt);
  const int nmat = (gateup || pl.pair) ? 2 : 1;
  pl.ndq = G_NUP + G_NFOLD;
  const size_t budget = 227 * 1024 - 1024;
  int n_st = 3;
  while (n_st < 16 && group_carve_bytes(nmat, bn, n_st + 1, n_groups) <= budget) ++n_st;
  pl.n_raw = n_st;   // stages (nibbles + token rows)
  pl.n_b = n_st;
  pl.smem_bytes = group_carve_bytes(nmat, bn, n_st, n_groups) + 1024;
  // A slots: 3 where they fit beside the 4 accumulator slices in 512 columns
  // (the kernel derives the same number from its template arguments)
  const uint32_t acc_cols = (uint32_t)(G_NBUF * nmat * bn);
  pl.n_a = (uint32_t)(3 * nmat * (QGROUP / 2)) + acc_cols <= 512u ? 3 : 2;
  const uint32_t need = (uint32_t)(pl.n_a * nmat * (QGROUP / 2)) + acc_cols;
  uint32_t cols = 32;
  while (cols < need) cols <<= 1;
  pl.tmem_cols = cols;
  return pl;
}

template <int MODE, int GBN>
static cudaError_t launch_group_one(const CUtensorMap& tmap, const GemmArgs& a, const GemmPlan& pl,
                                    int grid, cudaStream_t s, bool pdl) {
  auto kern = grouped_gemm_group_kernel<MODE, GBN>;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  return launch_kernel(kern, dim3(grid), dim3(G_THREADS), pl.smem_bytes, s, pdl, tmap, a);
}

template <int MODE>
static cudaError_t launch_group_mode(const CUtensorMap& tmap, const GemmArgs& a, const GemmPlan& pl,
                                     int grid, cudaStream_t s, bool pdl) {
  return a.bn == 16 ? launch_group_one<MODE, 16>(tmap, a, pl, grid, s, pdl)
                    : launch_group_one<MODE, 32>(tmap, a, pl, grid, s, pdl);
}

cudaError_t launch_grouped_gemm_group(bool gateup, const CUtensorMap& tmap_b, GemmArgs args,
                                      const GemmPlan& plan, int grid, cudaStream_t stream, bool pdl) {
  args.n_a = plan.n_a;
  args.n_b = plan.n_b;
  args.n_raw = plan.n_raw;
  args.tmem_cols = plan.tmem_cols;
  if (gateup) return launch_group_mode<G_GATEUP>(tmap_b, args, plan, grid, stream, pdl);
  if (plan.pair) {
    args.n_mt /= 2;   // work items name pairs of output tiles
    return launch_group_mode<G_DOWN_PAIR>(tmap_b, args, plan, grid, stream, pdl);
  }
  return launch_group_mode<G_DOWN>(tmap_b, args, plan, grid, stream, pdl);
}

}  // namespace moe
