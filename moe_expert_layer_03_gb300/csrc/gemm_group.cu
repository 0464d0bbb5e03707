// gemm_group.cu -- grouped expert GEMM for int4 experts and small row chunks
// (decode-sized batches, <= 32 rows of one expert per work item).
//
// "125B MoE on an RTX 3090 at 100+ tok/s": sec. 3.2 (grouped GEMM over the
// active experts, each a two-layer MLP), sec. 3.1 (per-expert int4 weights with
// their own scale and zero-point, turned into tensor-core operands without a
// separate pass over memory).
//
// At decode the layer streams int4 weights from HBM and the tensor-core work
// per weight is tiny, so the kernel is built around the per-byte cost of
// turning nibbles into MMA operands:
//   * the A operand is e4m3: a nibble q zero-extended to a byte is exactly the
//     e4m3 number q * 2^-9, so one AND (and one shift per 8 codes) makes the
//     operand; it lives in tensor memory (tcgen05.st), one TMEM lane per
//     weight row;
//   * the B operand is the token rows in e4m3 too, each row (h: each row's
//     128-feature block) scaled by a power of two that puts its largest
//     magnitude m in [128, 256), then split into hi = e4m3(v) and
//     lo = e4m3(v - hi) (the gather kernel and this kernel's gate/up epilogue
//     write them): hi + lo is the bf16 value exactly for every element of at
//     least m / 512, and within 2^-17 m for the smaller ones; the hi tile and
//     the lo tile below it form one B operand of 2 x bn rows, so one MMA per K
//     step and matrix covers both, and the fold adds the hi and lo columns of
//     the accumulator;
//   * the MMA is tcgen05.mma kind::f8f6f4 (K = 32), A from TMEM;
//   * each quantisation group (K = 128) accumulates into its own TMEM slice,
//     folded into fp32 registers with the group's scale s and zero z:
//         acc += s * (2^9 * (D_hi + D_lo) - z * S),
//     S the group's sum of the (scaled) token row; the token row's scale is
//     undone at the end (gate/up) or per group (down, where h is scaled per
//     128-feature block);
//   * within every 8-element K block the MMA sees the order {0,4,1,5,2,6,3,7}
//     (the order the nibbles come out of a word); the token rows are stored
//     in that order;
//   * one pipeline stage = one quantisation group: the int4 blocks of two
//     128-row matrices (gate and up of one output tile, or two adjacent down
//     tiles when d/128 is even), the token tile and the token rows' group
//     sums (for down: (sum, unscale factor) pairs), on one barrier;
//   * the warps that feed the MMAs (unpack) and the warps that consume them
//     (fold + epilogue) are separate; two MMA warps take alternate groups and
//     issue from a converged warp (elect.sync).
//
//   warps 0, 19  producers (bulk copy + TMA), one lane each, alternate groups:
//                an async-copy instruction costs its thread ~100 cycles of
//                issue, and one thread issuing every stage paced the
//                pipeline (Mixtral-shaped step 149.7 -> 148.0 us, 125B-class
//                143.0 -> 139.7 us)
//   warps 1-2    MMA issuers (warp 1 owns TMEM)
//   warps 3-10   unpack: two teams of four (one warp per TMEM lane quadrant)
//                taking alternate groups; a warp writes all codes of its
//                quadrant's rows (both matrices in the two-matrix modes)
//   warps 11-18  fold + epilogue, two per quadrant: every matrix and half the
//                token columns of its 32 rows
// Modes: gate/up (SwiGLU epilogue, h written in the e4m3 form the down GEMM
// reads), paired down (two output tiles), single down (one tile).
// fp8 experts (E4M3 codes, one fp16 scale per row and group): the codes are
// already the MMA's A operand, stored in the tensor core's 128-byte-swizzled
// image, so the MMAs read A straight from the stage in shared memory; the
// unpack warps stay idle and the fold drops the zero-point term
// (acc += s * (D_hi + D_lo)).
//
// Every wait is bounded; on a timeout the CTA drains its copies and MMAs,
// frees TMEM and returns with MOE_DEVERR_TIMEOUT set.
#include "gemm_common.cuh"

namespace moe {

using namespace gemm;

namespace {

constexpr int G_MAX_NBUF = 4;   // accumulator slices (fewer where TMEM is short)
constexpr int G_MAX_NA = 4;     // A slots in tensor memory
constexpr int G_MISC = 8;       // [0] tmem [1] abort [2] items [3] and [5] the producers' last group + 1
                                // [4] stays 0
constexpr int G_NMMA = 2;       // MMA-issuing warps (alternate groups)
constexpr int G_NUP = 8;        // unpack warps
constexpr int G_NFOLD = 8;      // fold + epilogue warps
constexpr int G_UP0 = 1 + G_NMMA;                  // first unpack warp
constexpr int G_FOLD0 = G_UP0 + G_NUP;             // first fold warp
constexpr int G_PROD1 = G_FOLD0 + G_NFOLD;          // the second producer warp
constexpr int G_THREADS = (G_PROD1 + 1) * 32;

enum GroupMode { G_GATEUP = 0, G_DOWN_PAIR = 1, G_DOWN = 2 };

// Where element e (0..7) of an 8-element K block is stored: the MMA sees the
// block in the order {0,4,1,5,2,6,3,7}.
__host__ __device__ constexpr int k_slot(int e) { return e < 4 ? 2 * e : 2 * (e - 4) + 1; }

// A work item (or, under the stream-K split, a segment of one) decoded once
// per CTA (the decode needs integer divisions by run-time values, which every
// warp would otherwise repeat).
struct ItemDesc {
  const uint8_t* slot;   // nullptr: the item is skipped (bad expert slot)
  int g0, g1;            // quantisation groups [g0, g1) of its K split (or segment)
  int r0, n_rows;        // token rows
  int mt, ks;            // output tile (pair) and K split
  int kind;              // 0 whole item; 1 its trailing groups, handed to the CTA before;
                         // 2 its leading groups, finished here with the next CTA's part
};
constexpr int G_PREFETCH_STAGES = 8;   // weight stages a CTA prefetches into L2 before its dependency wait
constexpr int G_ITEM_TAB = 64;   // items per CTA kept in the table; later ones are decoded on the fly

// Per stage the producer also copies the item rows' entries of the token
// rows' per-group array: floats (the group sums of x, [groups][rows_total])
// for gate/up, (sum, unscale factor) pairs ([groups][rows_total][2], for h)
// for down; a 16-byte-aligned superset of the row range, so the arrays need
// SUMS_PAD_BYTES of readable slack.
__host__ __device__ constexpr uint32_t sums_bytes(int bn, bool pairs) {
  return pairs ? (uint32_t)(bn + 2) * 8u : (uint32_t)(bn + 4) * 4u;
}

// Where the entries [r0, r0 + bn) of row `kg` of a [groups][rows_total] array
// of `esz`-byte entries start: a 16-byte-aligned address at or below them, and
// r0's entry offset from that address.
__device__ __forceinline__ const void* sums_src(const float* arr, int esz, int rows_total, int kg, int r0,
                                                int& off) {
  const uintptr_t u = reinterpret_cast<uintptr_t>(arr) + ((size_t)kg * rows_total + r0) * esz;
  off = (int)((u & 15u) / (uintptr_t)esz);
  return reinterpret_cast<const void*>(u & ~(uintptr_t)15);
}

struct GShared {
  ItemDesc* items;     // [G_ITEM_TAB]
  uint8_t* b_ring;     // [n_st][2 * bn * 128]  token rows (hi, then lo), SW128 K-major
  uint8_t* raw_ring;   // [n_st][nmat * I4_MAT_BYTES + sums_bytes]  nibbles + scale/zero
                       // words, then the token rows' group sums (and unscale factors)
  float* red;          // gate/up epilogue: [2][4][32] per-quadrant partial max / sum
  uint64_t *full, *empty;          // stages: producer -> consumers, consumers -> producer
  uint64_t *a_full, *a_empty;      // A slots: unpack -> MMA, MMA (commit) -> unpack
  uint64_t *acc_full, *acc_empty;  // accumulator slices: MMA (commit) -> fold, fold -> MMA
  uint64_t* epi;                   // [2] gate/up epilogue hand-offs among the fold warps
  uint64_t* fin;
  uint64_t* sk;                    // stream-K: the fold warps' partial sums are written
  int* misc;
  WorkList W;
};

// Bytes of one stage's weights + token-row entries (fp8: rounded up to 1 KB so
// every stage's code tiles keep the 1 KB alignment of the swizzled image).
__host__ __device__ constexpr uint32_t group_raw_stage(bool f8w, int nmat, int bn, bool gateup) {
  return f8w ? (((uint32_t)(nmat * F8_MAT_BYTES) + (gateup ? 0u : sums_bytes(bn, true)) + 1023u) & ~1023u)
             : (uint32_t)(nmat * I4_MAT_BYTES) + sums_bytes(bn, !gateup);
}

size_t group_carve_bytes(bool f8w, int nmat, int bn, bool gateup, int n_st, int n_groups) {
  size_t s = (size_t)n_st * ((size_t)bn * 256 + group_raw_stage(f8w, nmat, bn, gateup));
  s += sizeof(ItemDesc) * G_ITEM_TAB + 2 * 4 * 32 * sizeof(float);
  s = align_up(s, 16);
  s += 8 * (size_t)(2 * n_st + 2 * G_MAX_NA + 2 * G_MAX_NBUF + 2 + 1 + 1);
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
  d.kind = 0;
  return d;
}

// The stream-K sequence takes the items output tile by output tile, each tile
// over all experts' row chunks, instead of expert by expert: a share then holds
// tiles of several experts, so the few experts with many token rows (whose
// groups cost more to fold) do not all fall to a few neighbouring CTAs.
// Position q -> item index (items of group g: its row chunks x tiles, chunk
// fastest, one K split).
__device__ __forceinline__ int tile_major_item(int q, int total, const GemmArgs& p, const WorkList& W) {
  const int chunks = total / p.n_mt;   // row chunks over all groups
  const int mt = q / chunks, j = q - mt * chunks;
  int lo = 0, hi = p.n_groups - 1;   // last group whose first chunk is <= j
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (W.prefix[mid] / p.n_mt <= j) lo = mid; else hi = mid - 1;
  }
  return W.prefix[lo] + mt * W.nch[lo] + (j - W.prefix[lo] / p.n_mt);
}

// The CTA's i-th item (item index blockIdx.x + i * gridDim.x).
__device__ __forceinline__ ItemDesc get_item(int i, const GemmArgs& p, const GShared& S) {
  if (i < G_ITEM_TAB) return S.items[i];
  return make_item_desc(blockIdx.x + i * gridDim.x, p, S.W);
}

__device__ __forceinline__ bool wait_all(uint32_t bar, uint32_t parity, volatile int* abort_flag, int* err,
                                         uint64_t limit_ns) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort_flag, err, limit_ns));
}

// The 8 nibbles of a word as two registers of e4m3 codes q * 2^-9 (a nibble
// zero-extended to a byte): K positions {0,4,1,5} and {2,6,3,7} of the word's
// 8 elements (element 2i sits in bits [4i, 4i+4), 2i+1 in [16+4i, 20+4i)).
__device__ __forceinline__ void e4m3_codes(uint32_t w, uint32_t& a, uint32_t& b) {
  a = w & 0x0F0F0F0Fu;
  b = (w >> 4) & 0x0F0F0F0Fu;
}

}  // namespace

template <int MODE, int GBN, bool F8W>
__global__ void __launch_bounds__(G_THREADS, 1)
    grouped_gemm_group_kernel(const __grid_constant__ CUtensorMap tmap_b, const GemmArgs p) {
  constexpr bool GATEUP = MODE == G_GATEUP;
  constexpr bool PAIR = MODE != G_DOWN;                // two 128-row matrices per stage
  constexpr int NMAT = PAIR ? 2 : 1;
  constexpr int ESZ = GATEUP ? 4 : 8;                  // bytes per token entry of the per-group array
  // int4: gate/up needs the token rows' group sums (zero-point term), down the
  // (sum, unscale) pairs of h; fp8: only down's unscale factors
  constexpr uint32_t SUMS = (F8W && GATEUP) ? 0u : sums_bytes(GBN, !GATEUP);
  constexpr uint32_t W_BYTES = NMAT * (F8W ? F8_MAT_BYTES : I4_MAT_BYTES);   // weights of a stage
  constexpr uint32_t SUMS_OFF = W_BYTES;               // the token rows' per-group entries
  constexpr uint32_t RAW_STAGE = group_raw_stage(F8W, NMAT, GBN, GATEUP);
  constexpr uint32_t LOADED = W_BYTES + SUMS;          // bytes the copies of a stage bring
  constexpr uint32_t A_COLS = NMAT * 32;               // TMEM columns of one A slot (128 e4m3 per row)
  constexpr uint32_t B_BOX = (uint32_t)GBN * 128u;     // one TMA box: GBN rows x 128 bytes
  constexpr uint32_t B_STAGE = 2u * B_BOX;             // hi rows, then lo rows
  constexpr int NA = F8W ? 0 : G_MAX_NA;               // A slots (fp8: A is read from the stage)
  constexpr uint32_t SLICE = NMAT * 2 * GBN;           // TMEM columns of one accumulator slice (hi, lo)
  constexpr int NBUF = (512 - NA * (int)A_COLS) / (int)SLICE < G_MAX_NBUF
                           ? (512 - NA * (int)A_COLS) / (int)SLICE
                           : G_MAX_NBUF;               // accumulator slices
  static_assert(NA * (int)A_COLS + NBUF * (int)SLICE <= 512, "tensor memory columns");
  // The two MMA warps and the two unpack teams take alternate groups, and a
  // barrier polled by parity must never run two phases ahead of a waiter: so
  // every A slot and every accumulator slice belongs to one MMA warp (and one
  // unpack team) only, i.e. both counts are multiples of 2.  (With 3 A slots
  // and 5 slices a warp saw the phase before its own as complete and the
  // pipeline stalled until the wait limit.)
  static_assert(G_NMMA == 2 && G_NUP / 4 == 2 && NA % 2 == 0 && NBUF % 2 == 0, "slots per MMA warp");
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
  S.red = reinterpret_cast<float*>(cur);
  cur += 2 * 4 * 32 * sizeof(float);
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + align_up((size_t)(cur - base), 16));
  S.full = bars;
  S.empty = S.full + n_st;
  S.a_full = S.empty + n_st;
  S.a_empty = S.a_full + G_MAX_NA;
  S.acc_full = S.a_empty + G_MAX_NA;
  S.acc_empty = S.acc_full + G_MAX_NBUF;
  S.epi = S.acc_empty + G_MAX_NBUF;
  S.fin = S.epi + 2;
  S.sk = S.fin + 1;
  S.misc = reinterpret_cast<int*>(S.sk + 1);
  S.W.prefix = S.misc + G_MISC;
  S.W.nch = S.W.prefix + (p.n_groups + 1);
  S.W.goff = S.W.nch + (p.n_groups + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int* abort_flag = &S.misc[1];

  // ------------------------------------------------------------ set-up
  if (threadIdx.x == 0) {
    for (int i = 0; i < n_st; ++i) {
      mbar_init(smem_u32(&S.full[i]), 1);
      mbar_init(smem_u32(&S.empty[i]), ((F8W ? 0 : G_NUP / 2) + G_NFOLD) * 32);   // one unpack team per group
    }
    for (int i = 0; i < G_MAX_NA; ++i) {
      mbar_init(smem_u32(&S.a_full[i]), G_NUP / 2 * 32);
      mbar_init(smem_u32(&S.a_empty[i]), 1);
    }
    for (int i = 0; i < G_MAX_NBUF; ++i) {
      mbar_init(smem_u32(&S.acc_full[i]), 1);
      mbar_init(smem_u32(&S.acc_empty[i]), G_NFOLD * 32);
    }
    for (int i = 0; i < 2; ++i) mbar_init(smem_u32(&S.epi[i]), G_NFOLD * 32);
    mbar_init(smem_u32(S.fin), G_NMMA);
    mbar_init(smem_u32(S.sk), G_NFOLD * 32);
    for (int i = 1; i < G_MISC; ++i)
      if (i != 2) S.misc[i] = 0;   // [0] written by tcgen05.alloc, [2] by the first unpack warp
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) prefetch_tensormap(&tmap_b);
  if (warp == 1) {
    tmem_alloc(smem_u32(&S.misc[0]), p.tmem_cols);
    tmem_relinquish();
  }
  // Before the dependency wait, prefetch into L2 the first weight stages of
  // the item this CTA gets if every group is active with one row chunk
  // (likely when the batch holds at least two rows per routed expert), so the
  // weight stream starts while the previous kernel finishes (Mixtral-shaped
  // decode step: 8-bit 232 -> 224 us; int4, once its two producers kept the
  // ring full, 148.7 -> 143.1 us, 125B-class 139.5 -> 137.7 us; 16 stages
  // instead of 8 measured slower).  Only the expert-to-slot table is read (an
  // input, not an earlier kernel's output); a wrong guess costs the
  // prefetched bytes.
  if constexpr (MODE != G_DOWN) {
    if (warp == 0 && lane == 0 && p.rows_total >= 2 * p.n_routed) {
      const int per_g = p.n_mt * p.ksplit;
      const int g = (int)blockIdx.x / per_g;
      if (g < p.n_groups) {
        const int t2 = (int)blockIdx.x - g * per_g, ks = t2 % p.ksplit, mt = t2 / p.ksplit;
        int g0, g1;
        kgroups(p, ks, g0, g1);
        const uint8_t* slot = nullptr;
        if (g < p.n_routed) {
          const int sl = p.e2s_r[g];
          if (sl >= 0 && sl < p.n_slots_r) slot = p.pool_r + (size_t)sl * p.slot_bytes_r;
        } else if (p.pool_s != nullptr) {
          const int sl = p.e2s_s[0];
          if (sl >= 0 && sl < p.n_slots_s) slot = p.pool_s + (size_t)sl * p.slot_bytes_s;
        }
        if (slot != nullptr)
          for (int kg = g0; kg < g1 && kg < g0 + G_PREFETCH_STAGES; ++kg) {
            prefetch_l2_bulk(slot + p.sec_off + ((size_t)mt * (p.K / QGROUP) + kg) * W_BYTES, W_BYTES);
          }
      }
    }
  }
  // everything above overlaps the previous kernel's tail (dependent launch);
  // below, the offsets, token rows and outputs of earlier kernels are read
  griddep_wait();
  griddep_launch_dependents();
  if (warp == G_UP0) {
    const int total = build_worklist(p, S.W, lane);
    __syncwarp();
    // Stream-K (gate/up): the items' quantisation groups in one sequence
    // (items in tile-major order), an equal share of it per CTA, so the last
    // wave is never a partial one.  An
    // item cut between CTAs c and c + 1 is finished by c (its leading groups
    // come last in c's share) with the partial sums c + 1 hands over (its
    // trailing groups come first in c + 1's share).  Only when every share
    // holds at least one whole item (an item spans at most two CTAs), and only
    // when whole items would leave the last wave well short of full: the
    // shares scatter the CTAs over the whole pool at once, which measured a
    // few percent slower than whole items taken in step (a last wave 89% full,
    // 896 items on 152 CTAs, is better left alone; one 34% full, 660 items, is
    // not).
    const int G = p.K / QGROUP;
    const long long units = (long long)total * G;
    const long long u0 = units * blockIdx.x / gridDim.x, u1 = units * (blockIdx.x + 1) / gridDim.x;
    const long long whole_waves = ((long long)total + gridDim.x - 1) / gridDim.x;
    const bool sk = GATEUP && p.sk_part != nullptr && p.ksplit == 1 && units >= (long long)gridDim.x * G &&
                    (u1 - u0) / G + 2 <= G_ITEM_TAB && whole_waves * gridDim.x * 100 > (long long)total * 108;
    int n_mine;
    if (sk) {
      const int first = (int)(u0 / G), last = (int)((u1 - 1) / G);
      n_mine = last - first + 1;
      for (int i = lane; i < n_mine; i += 32) {
        const int q = first + i;   // position in the sequence
        ItemDesc dsc = make_item_desc(tile_major_item(q, total, p, S.W), p, S.W);
        const long long ib = (long long)q * G;
        dsc.g0 = (int)((u0 > ib ? u0 : ib) - ib);
        dsc.g1 = (int)((u1 < ib + G ? u1 : ib + G) - ib);
        dsc.kind = dsc.g0 > 0 ? 1 : (dsc.g1 < G ? 2 : 0);
        S.items[i] = dsc;
      }
    } else {
      n_mine = total > (int)blockIdx.x ? (total - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x : 0;
      for (int i = lane; i < n_mine && i < G_ITEM_TAB; i += 32)
        S.items[i] = make_item_desc(blockIdx.x + i * gridDim.x, p, S.W);
    }
    if (lane == 0) S.misc[2] = n_mine;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = (uint32_t)S.misc[0];
  const int n_mine = S.misc[2];   // items of this CTA
  const uint32_t acc0 = NA * A_COLS;   // accumulator slices follow the A slots

  if (warp == 0 || warp == G_PROD1) {
    // ================================================================ producers
    // Per group one stage: the NMAT nibble blocks and the token tile (hi rows
    // at y = r0, lo rows at y = rows_total + r0), on one barrier.  In the
    // paired down mode the item's tile index mt names the output tiles 2mt
    // and 2mt + 1.  Two producers take alternate groups; the stage count is
    // even, so every stage belongs to one of them and each waits only for its
    // own stages' earlier fills (the consumers take the groups in order, so
    // neither can wait on a group the other has not issued yet).
    if (lane == 0) {
      const int pid = warp == 0 ? 0 : 1;   // producer pid feeds the groups gc with gc % 2 == pid
      Ring rs{0, 0, n_st};
      int last = 0;
      uint32_t gc = 0;
      const uint64_t pol = policy_evict_first();
      bool ok = true;
      for (int ii = 0; ii < n_mine && ok && !*abort_flag; ++ii) {
        const ItemDesc it = get_item(ii, p, S);
        if (!it.slot) continue;
        const int g0 = it.g0, g1 = it.g1;
        const uint8_t* sec = it.slot + p.sec_off;
        for (int kg = g0; kg < g1; ++kg, ++gc, rs.next()) {
          if ((int)(gc & 1u) != pid) continue;
          if ((int)gc == p.stop_stage) {   // test hook: stop feeding the pipeline
            ok = false;
            break;
          }
          if (!(ok = mbar_wait(smem_u32(&S.empty[rs.i]), rs.ph ^ 1u, abort_flag, p.err, p.wait_ns))) break;
          const uint32_t bar = smem_u32(&S.full[rs.i]);
          mbar_arrive_expect_tx(bar, LOADED + B_STAGE);
          const uint32_t raw = smem_u32(S.raw_ring + (size_t)rs.i * RAW_STAGE);
          int off;
          if (SUMS > 0)
            bulk_g2s(raw + SUMS_OFF, sums_src(p.b_sum, ESZ, p.rows_total, kg, it.r0, off), SUMS, bar);
          // gate/up: gate and up blocks of (mt, kg); down: tile mt's block, or
          // both blocks of the pair it.mt, contiguous in the down section
          if (F8W && MODE == G_DOWN) {   // one tile of an fp8 pair block: its codes, then its scales
            int mp, bm;
            const size_t blk = fp8_down_block(it.mt, kg, p.K / QGROUP, p.n_mt, mp, bm);
            bulk_g2s_hint(raw, sec + blk + (size_t)mp * F8_CODE_BYTES, F8_CODE_BYTES, bar, pol);
            bulk_g2s_hint(raw + F8_CODE_BYTES, sec + blk + (size_t)bm * F8_CODE_BYTES + mp * TILE_M * 2,
                          TILE_M * 2, bar, pol);
          } else {
            const size_t woff = MODE == G_DOWN ? i4_down_block(it.mt, kg, p.K / QGROUP, p.n_mt)
                                               : ((size_t)it.mt * (p.K / QGROUP) + kg) * W_BYTES;
            bulk_g2s_hint(raw, sec + woff, W_BYTES, bar, pol);
          }
          const uint32_t dst = smem_u32(S.b_ring + (size_t)rs.i * B_STAGE);
          tma_load_2d(dst, &tmap_b, kg * QGROUP, it.r0, bar);
          tma_load_2d(dst + B_BOX, &tmap_b, kg * QGROUP, p.rows_total + it.r0, bar);
          last = (int)gc + 1;
        }
      }
      S.misc[pid ? 5 : 3] = last;
    }
  } else if (warp < G_UP0) {
    // ================================================================ MMA issuers
    // Warp 1 + mw issues the groups with (group counter % 2) == mw.  Group gc
    // uses A slot gc % NA and accumulator slice gc % NBUF.  a_full(gc) also
    // implies that the group's stage (token tile) has landed: the unpack
    // threads arrive only after seeing it.  The whole warp runs the loop;
    // ring positions advance by one per group, owned or not.
    const int mw = warp - 1;
    bool ok = true;
    Ring rs{0, 0, n_st}, ra{0, 0, NA > 0 ? NA : 1}, rc{0, 0, NBUF};
    const uint64_t bdesc0 = sdesc_kmajor_sw128(smem_u32(S.b_ring));   // stage 0, K step 0
    const uint64_t adesc0 = sdesc_kmajor_sw128(smem_u32(S.raw_ring));   // fp8: stage 0's first code tile
    const uint32_t idesc = idesc_f16kind_f32(TILE_M, (uint32_t)(2 * GBN), 0u);   // e4m3 x e4m3 -> f32
    uint32_t gc = 0;
    for (int ii = 0; ii < n_mine && ok; ++ii) {
      const ItemDesc it = get_item(ii, p, S);
      if (!it.slot) continue;
      const int g0 = it.g0, g1 = it.g1;
      for (int kg = g0; kg < g1; ++kg, ++gc, rs.next(), ra.next(), rc.next()) {
        if ((int)(gc & 1u) != mw) continue;
        // int4: the unpacked A slot (which implies its stage has landed); fp8:
        // the stage itself, whose code tiles are the A operand
        if (!(ok = wait_all(F8W ? smem_u32(&S.full[rs.i]) : smem_u32(&S.a_full[ra.i]), F8W ? rs.ph : ra.ph,
                            abort_flag, p.err, p.wait_ns)))
          break;
        if (!(ok = wait_all(smem_u32(&S.acc_empty[rc.i]), rc.ph ^ 1u, abort_flag, p.err, p.wait_ns))) break;
        tc_fence_after();
        // the descriptor's start-address field counts 16-byte units
        const uint64_t bd = bdesc0 + (uint64_t)(((uint32_t)rs.i * B_STAGE) >> 4);
        const uint32_t d0 = tmem_base + acc0 + (uint32_t)rc.i * SLICE;
        if constexpr (F8W) {
          const uint64_t ad = adesc0 + (uint64_t)(((uint32_t)rs.i * RAW_STAGE) >> 4);
#pragma unroll
          for (int q = 0; q < 4; ++q) {   // K steps of 32 over the hi and lo rows at once
            const uint64_t bq = bd + (uint64_t)((q * 32) >> 4);
            const uint64_t aq = ad + (uint64_t)((q * 32) >> 4);
            if (NMAT == 2)
              mma2_f8_ss_elect(d0, d0 + 2 * GBN, aq, aq + (uint64_t)(F8_CODE_BYTES >> 4), bq, idesc,
                               q > 0 ? 1u : 0u);
            else
              mma_f8_ss_elect(d0, aq, bq, idesc, q > 0 ? 1u : 0u);
          }
        } else {
          const uint32_t a_base = tmem_base + (uint32_t)ra.i * A_COLS;
#pragma unroll
          for (int q = 0; q < 4; ++q) {   // K steps of 32 over the hi and lo rows at once
            const uint64_t bq = bd + (uint64_t)((q * 32) >> 4);
            const uint32_t ak = a_base + (uint32_t)(q * 8);
            if (NMAT == 2)
              mma2_f8_ta_elect(d0, d0 + 2 * GBN, ak, ak + 32, bq, idesc, q > 0 ? 1u : 0u);
            else
              mma_f8_ta_elect(d0, ak, bq, idesc, q > 0 ? 1u : 0u);
          }
          mma_commit_elect(smem_u32(&S.a_empty[ra.i]));
        }
        mma_commit_elect(smem_u32(&S.acc_full[rc.i]));
      }
    }
  } else if (warp < G_FOLD0) {
    // ================================================================ unpack
    // Two teams of four warps (one per TMEM lane quadrant) take alternate
    // groups, so two groups' stores are in flight at once.  Group gc (team
    // gc % 2): wait for its stage and for A slot gc % NA to be free (the MMAs
    // of group gc - NA are done); write all codes of my row (both matrices in
    // the two-matrix modes); release my reads of the stage; hand the slot to
    // the MMA warp once the stores have landed.  Ring positions advance by one
    // per group, owned or not.
    const int team = (warp - G_UP0) >> 2;
    const int quad = warp & 3;               // TMEM lane quadrant of this warp
    const int r = quad * 32 + lane;          // weight row of the tile = TMEM lane
    const uint32_t lane_base = tmem_base + ((uint32_t)(quad * 32) << 16);
    Ring rs{0, 0, n_st}, ra{0, 0, NA > 0 ? NA : 1};
    bool ok = true;
    uint32_t gc = 0;
    for (int ii = 0; ii < (F8W ? 0 : n_mine) && ok; ++ii) {   // fp8: nothing to unpack
      const ItemDesc it = get_item(ii, p, S);
      if (!it.slot) continue;
      const int g0 = it.g0, g1 = it.g1;
      for (int kg = g0; kg < g1 && ok; ++kg, ++gc, rs.next(), ra.next()) {
        if ((int)(gc & 1u) != team) continue;
        if (!(ok = wait_all(smem_u32(&S.full[rs.i]), rs.ph, abort_flag, p.err, p.wait_ns))) break;
        if (!(ok = wait_all(smem_u32(&S.a_empty[ra.i]), ra.ph ^ 1u, abort_flag, p.err, p.wait_ns))) break;
        tc_fence_after();
        const uint8_t* stage = S.raw_ring + (size_t)rs.i * RAW_STAGE;
        const uint32_t ta = lane_base + (uint32_t)ra.i * A_COLS;
#pragma unroll
        for (int m = 0; m < NMAT; ++m) {   // all 128 codes of my row: column h*16 + j*8 + 2w (+1)
          const uint8_t* mat = stage + m * I4_MAT_BYTES;
          uint32_t v[32];
#pragma unroll
          for (int hj = 0; hj < 4; ++hj) {   // quad (h, j) = (hj >> 1, hj & 1)
            const uint4 wq = *reinterpret_cast<const uint4*>(mat + (hj * TILE_M + r) * 16);
            e4m3_codes(wq.x, v[hj * 8 + 0], v[hj * 8 + 1]);
            e4m3_codes(wq.y, v[hj * 8 + 2], v[hj * 8 + 3]);
            e4m3_codes(wq.z, v[hj * 8 + 4], v[hj * 8 + 5]);
            e4m3_codes(wq.w, v[hj * 8 + 6], v[hj * 8 + 7]);
          }
          tmem_st_32(ta + (uint32_t)(m * 32), v);
        }
        mbar_arrive(smem_u32(&S.empty[rs.i]));   // my reads of the stage are done
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(smem_u32(&S.a_full[ra.i]));
      }
    }
  } else {
    // ================================================================ fold + epilogue
    // Two warps per TMEM lane quadrant; each thread owns weight row r of every
    // matrix and half the item's token columns (the SwiGLU epilogue needs gate
    // and up of a token together; for the paired down GEMM a split by output
    // tile measured slower).  Group gc: wait for its accumulator slice, fold
    // it with the group's scale and zero (read from the stage, which this warp
    // releases afterwards) and the token rows' group sums, free the slice.
    constexpr int NM = NMAT;                           // matrices per fold warp
    const int quad = warp & 3;
    const int r = quad * 32 + lane;
    const int m0 = 0;                                  // my first matrix
    const int c0 = ((warp - G_FOLD0) >> 2) * (GBN / 2);   // my token columns [c0, c0 + CW)
    const uint32_t lane_base = tmem_base + ((uint32_t)(quad * 32) << 16);
    constexpr int CW = GBN / 2;                        // token columns per fold thread
    constexpr int CH = 4;                              // columns per tcgen05.ld (and per chunk): an item
                                                       // of n rows folds ceil(n / 4) chunks
    Ring rs{0, 0, n_st}, rc{0, 0, NBUF};
    uint32_t it_count = 0;
    bool ok = true;
    for (int ii = 0; ii < n_mine && ok; ++ii) {
      const ItemDesc it = get_item(ii, p, S);
      if (!it.slot) continue;
      const int g0 = it.g0, g1 = it.g1;
      const int nc = max(0, min(CW, it.n_rows - c0));   // my token columns of this item
      // gate/up: the token rows' unscale factors for the item epilogue, loaded
      // now so that their latency hides behind the item's groups
      float ufac[CW];
#pragma unroll
      for (int i = 0; i < CW; ++i) ufac[i] = (GATEUP && i < nc) ? __ldg(p.b_scale + it.r0 + c0 + i) : 0.f;
      float acc[NM][CW];
#pragma unroll
      for (int m = 0; m < NM; ++m)
#pragma unroll
        for (int i = 0; i < CW; ++i) acc[m][i] = 0.f;
      for (int kg = g0; kg < g1 && ok; ++kg) {
        if (!(ok = wait_all(smem_u32(&S.full[rs.i]), rs.ph, abort_flag, p.err, p.wait_ns))) break;
        const uint8_t* raw = S.raw_ring + (size_t)rs.i * RAW_STAGE;
        // per matrix: int4: 2^9 s (the codes are q 2^-9) and s z; fp8: s and 0
        float s9[NM], sz[NM];
#pragma unroll
        for (int m = 0; m < NM; ++m) {
          if constexpr (F8W) {
            const uint16_t w = *reinterpret_cast<const uint16_t*>(raw + NMAT * F8_CODE_BYTES + (m0 + m) * TILE_M * 2 + r * 2);
            s9[m] = __half2float(__ushort_as_half(w));
            sz[m] = 0.f;
          } else {
            const uint32_t w = *reinterpret_cast<const uint32_t*>(raw + (m0 + m) * I4_MAT_BYTES + I4_PACKED_BYTES + r * 4);
            const float sc = __half2float(__ushort_as_half((unsigned short)(w & 0xFFFFu)));
            s9[m] = 512.f * sc;
            sz[m] = sc * __half2float(__ushort_as_half((unsigned short)(w >> 16)));
          }
        }
        int off;
        sums_src(p.b_sum, ESZ, p.rows_total, kg, it.r0, off);
        // gate/up: sums; down: (sum, unscale) pairs
        const float* bsum = reinterpret_cast<const float*>(raw + SUMS_OFF) + (off + c0) * (ESZ / 4);
        if (!(ok = wait_all(smem_u32(&S.acc_full[rc.i]), rc.ph, abort_flag, p.err, p.wait_ns))) break;
        tc_fence_after();
        const uint32_t ta = lane_base + acc0 + (uint32_t)rc.i * SLICE;
#pragma unroll
        for (int ch = 0; ch < CW / CH; ++ch) {
          if (ch * CH < nc) {
            uint32_t dv[NM][CH], dl[NM][CH];   // hi and lo columns
#pragma unroll
            for (int m = 0; m < NM; ++m) {
              const uint32_t col = ta + (uint32_t)((m0 + m) * 2 * GBN + c0 + ch * CH);
              tmem_ld_4(col, *reinterpret_cast<uint32_t(*)[4]>(dv[m]));
              tmem_ld_4(col + GBN, *reinterpret_cast<uint32_t(*)[4]>(dl[m]));
            }
            // token factors (shared by the matrices) while the loads are in flight
            float bs[CH], bu[CH];
#pragma unroll
            for (int i = 0; i < CH; ++i) {
              const float u = GATEUP ? 1.f : bsum[2 * (ch * CH + i) + 1];
              bu[i] = u;
              bs[i] = F8W ? 0.f : u * bsum[(ch * CH + i) * (ESZ / 4)];
            }
#pragma unroll
            for (int m = 0; m < NM; ++m) {
              tmem_ld_wait_regs(dv[m]);
              tmem_ld_wait_regs(dl[m]);
#pragma unroll
              for (int i = 0; i < CH; ++i) {
                const int n = ch * CH + i;
                const float sd = GATEUP ? s9[m] : s9[m] * bu[i];
                const float dsum = __uint_as_float(dv[m][i]) + __uint_as_float(dl[m][i]);
                acc[m][n] = F8W ? fmaf(sd, dsum, acc[m][n]) : fmaf(sd, dsum, fmaf(-sz[m], bs[i], acc[m][n]));
              }
            }
          }
        }
        tc_fence_before();
        mbar_arrive(smem_u32(&S.acc_empty[rc.i]));
        mbar_arrive(smem_u32(&S.empty[rs.i]));
        rs.next();
        rc.next();
      }
      if (!ok) break;

      if constexpr (GATEUP) {
        if (it.kind == 1) {   // trailing groups: hand the partial sums to the CTA before
          float* part = p.sk_part + (size_t)blockIdx.x * (NMAT * TILE_M * GBN);
#pragma unroll
          for (int m = 0; m < NM; ++m)
#pragma unroll
            for (int i = 0; i < CW; ++i)
              if (i < nc) part[((m0 + m) * TILE_M + r) * GBN + c0 + i] = acc[m][i];
          __threadfence();
          mbar_arrive(smem_u32(S.sk));   // at most one such segment per CTA: phase 0
          if (warp == G_FOLD0 && lane == 0 && mbar_wait(smem_u32(S.sk), 0, abort_flag, p.err, p.wait_ns))
            st_release_gpu(p.sk_flags + blockIdx.x, 1);
          continue;
        }
        if (it.kind == 2) {   // leading groups: add the next CTA's partial sums of the item
          const int* flag = p.sk_flags + blockIdx.x + 1;
          if (ld_acquire_gpu(flag) == 0) {
            const uint64_t t0 = global_timer_ns();
            while (ok && ld_acquire_gpu(flag) == 0) {
              if (*abort_flag) ok = false;
              else if (global_timer_ns() - t0 > p.wait_ns) {
                *abort_flag = 1;
                atomicOr(p.err, MOE_DEVERR_TIMEOUT);
                ok = false;
              }
            }
          }
          if (!__all_sync(0xffffffffu, ok)) {
            ok = false;
            break;
          }
          const float* part = p.sk_part + (size_t)(blockIdx.x + 1) * (NMAT * TILE_M * GBN);
#pragma unroll
          for (int m = 0; m < NM; ++m)
#pragma unroll
            for (int i = 0; i < CW; ++i)
              if (i < nc) acc[m][i] += part[((m0 + m) * TILE_M + r) * GBN + c0 + i];
        }
      }

      // ---- item epilogue from the register accumulators
      if constexpr (GATEUP) {
        // h = silu(gate) * up for my feature row, then its e4m3 hi/lo form for
        // the down GEMM: per token, a power-of-two scale from the largest |h|
        // over the tile's 128 features, the two bytes, and the sum of hi + lo
        // over the 128 features.  The four fold warps combine their partial
        // maxima and sums through shared memory (bounded mbarrier hand-offs).
        const uint32_t par = it_count & 1u;
        float hv[CW];
#pragma unroll
        for (int i = 0; i < CW; ++i) {
          hv[i] = 0.f;
          if (i < nc) {
            const float u = ufac[i];
            hv[i] = silu_f(acc[0][i] * u) * (acc[1][i] * u);
          }
        }
#pragma unroll
        for (int i = 0; i < CW; ++i) {
          float m = fabsf(hv[i]);
#pragma unroll
          for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
          if (lane == i) S.red[quad * 32 + c0 + i] = m;
        }
        mbar_arrive(smem_u32(&S.epi[0]));
        if (!(ok = wait_all(smem_u32(&S.epi[0]), par, abort_flag, p.err, p.wait_ns))) break;
        uint8_t* hq = p.q_out;
        const int f = it.mt * TILE_M + (r & ~7) + k_slot(r & 7);   // stored position of my feature
        float ssum[CW];
#pragma unroll
        for (int i = 0; i < CW; ++i) {
          ssum[i] = 0.f;
          if (i < nc) {
            const int t = c0 + i;   // token column
            const float am = fmaxf(fmaxf(S.red[t], S.red[32 + t]), fmaxf(S.red[64 + t], S.red[96 + t]));
            int ex = 0;
            if (am > 0.f) frexpf(am, &ex);
            const int e = max(-126, min(126, am > 0.f ? 8 - ex : 0));   // 2^e, 2^-e normal
            const float x = hv[i] * __int_as_float((127 + e) << 23);
            const uint16_t hb = f32x2_to_e4m3x2(x, 0.f);
            const float hf = e4m3x2_to_f32x2(hb).x;
            const uint16_t lb = f32x2_to_e4m3x2(x - hf, 0.f);
            ssum[i] = hf + e4m3x2_to_f32x2(lb).x;
            hq[(size_t)(it.r0 + t) * p.out_ld + f] = (uint8_t)(hb & 0xFFu);
            hq[(size_t)(p.rows_total + it.r0 + t) * p.out_ld + f] = (uint8_t)(lb & 0xFFu);
            if (quad == 0 && lane == i)   // h's (sum, unscale) pair: the unscale factor
              p.sum_out[2 * ((size_t)it.mt * p.rows_total + it.r0 + t) + 1] = __int_as_float((127 - e) << 23);
          }
        }
#pragma unroll
        for (int i = 0; i < CW; ++i) {
          float v = ssum[i];
#pragma unroll
          for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
          if (lane == i) S.red[128 + quad * 32 + c0 + i] = v;
        }
        mbar_arrive(smem_u32(&S.epi[1]));
        if (!(ok = wait_all(smem_u32(&S.epi[1]), par, abort_flag, p.err, p.wait_ns))) break;
        if (quad == 0 && lane < nc)   // h's (sum, unscale) pair: the sum
          p.sum_out[2 * ((size_t)it.mt * p.rows_total + it.r0 + c0 + lane)] =
              S.red[128 + c0 + lane] + S.red[160 + c0 + lane] + S.red[192 + c0 + lane] + S.red[224 + c0 + lane];
      } else {
        float* y = reinterpret_cast<float*>(p.out) + (size_t)it.ks * p.out_split_stride;
#pragma unroll
        for (int m = 0; m < NM; ++m) {
          const int f = (MODE == G_DOWN_PAIR ? 2 * it.mt + m0 + m : it.mt) * TILE_M + r;
#pragma unroll
          for (int i = 0; i < CW; ++i)
            if (i < nc) y[(size_t)(it.r0 + c0 + i) * p.out_ld + f] = acc[m][i];
        }
      }
      ++it_count;
    }
  }

  // ------------------------------------------------------------ teardown
  __syncthreads();
  volatile int* no_abort = &S.misc[4];   // stays 0: drain waits are bounded by time only
  if ((warp == 0 || warp == G_PROD1) && lane == 0 && *abort_flag) {
    // for each stage of this producer, wait (bounded) for the last copies issued into it
    const int pid = warp == 0 ? 0 : 1;
    const int iss = S.misc[pid ? 5 : 3];
    for (int sl = pid; sl < n_st && sl < iss; sl += 2) {
      const int q = sl + ((iss - 1 - sl) / n_st) * n_st;
      mbar_wait(smem_u32(&S.full[sl]), (uint32_t)((q / n_st) & 1), no_abort, p.err, p.wait_ns);
    }
  }
  if (warp >= 1 && warp < G_UP0) {   // every MMA this CTA issued has finished
    mma_commit_elect(smem_u32(S.fin));
    mbar_wait(smem_u32(S.fin), 0, no_abort, p.err, p.wait_ns);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, p.tmem_cols);
}

// ------------------------------------------------------------------ host side
GemmPlan plan_gemm_group(int fmt, bool gateup, int bn, int n_groups, int n_mt) {
  GemmPlan pl{};
  pl.group = true;
  pl.pair = !gateup && down_paired(fmt, n_mt);
  const int nmat = (gateup || pl.pair) ? 2 : 1;
  const bool f8w = fmt == MOE_W_FP8_G128;
  pl.ndq = G_NUP + G_NFOLD;
  const size_t budget = 227 * 1024 - 1024;
  int n_st = 3;
  while (n_st < 16 && group_carve_bytes(f8w, nmat, bn, gateup, n_st + 1, n_groups) <= budget) ++n_st;
  n_st &= ~1;   // each stage belongs to one of the two producers
  pl.n_raw = n_st;   // stages (weights + token rows)
  pl.n_b = n_st;
  pl.smem_bytes = group_carve_bytes(f8w, nmat, bn, gateup, n_st, n_groups) + 1024;
  // the kernel derives its A slot and accumulator slice counts from its
  // template arguments so that they fit 512 columns
  pl.n_a = G_MAX_NA;
  pl.tmem_cols = 512;
  return pl;
}

template <int MODE, int GBN, bool F8W>
static cudaError_t launch_group_one(const CUtensorMap& tmap, const GemmArgs& a, const GemmPlan& pl,
                                    int grid, cudaStream_t s, bool pdl) {
  auto kern = grouped_gemm_group_kernel<MODE, GBN, F8W>;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  return launch_kernel(kern, dim3(grid), dim3(G_THREADS), pl.smem_bytes, s, pdl, tmap, a);
}

template <int MODE, bool F8W>
static cudaError_t launch_group_mode(const CUtensorMap& tmap, const GemmArgs& a, const GemmPlan& pl,
                                     int grid, cudaStream_t s, bool pdl) {
  return a.bn == 16 ? launch_group_one<MODE, 16, F8W>(tmap, a, pl, grid, s, pdl)
                    : launch_group_one<MODE, 32, F8W>(tmap, a, pl, grid, s, pdl);
}

template <bool F8W>
static cudaError_t launch_group_fmt(bool gateup, const CUtensorMap& tmap_b, GemmArgs args,
                                    const GemmPlan& plan, int grid, cudaStream_t stream, bool pdl) {
  if (gateup) return launch_group_mode<G_GATEUP, F8W>(tmap_b, args, plan, grid, stream, pdl);
  if (plan.pair) {
    args.n_mt /= 2;   // work items name pairs of output tiles
    return launch_group_mode<G_DOWN_PAIR, F8W>(tmap_b, args, plan, grid, stream, pdl);
  }
  return launch_group_mode<G_DOWN, F8W>(tmap_b, args, plan, grid, stream, pdl);
}

cudaError_t launch_grouped_gemm_group(int fmt, bool gateup, const CUtensorMap& tmap_b, GemmArgs args,
                                      const GemmPlan& plan, int grid, cudaStream_t stream, bool pdl) {
  args.n_a = plan.n_a;
  args.n_b = plan.n_b;
  args.n_raw = plan.n_raw;
  args.tmem_cols = plan.tmem_cols;
  return fmt == MOE_W_FP8_G128 ? launch_group_fmt<true>(gateup, tmap_b, args, plan, grid, stream, pdl)
                               : launch_group_fmt<false>(gateup, tmap_b, args, plan, grid, stream, pdl);
}

}  // namespace moe
