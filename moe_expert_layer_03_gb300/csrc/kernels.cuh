// kernels.cuh -- internal declarations shared by the library's translation units:
// the prepacked slot layout, the grouped-GEMM argument block, launch helpers.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "moe.h"

namespace moe {

// ------------------------------------------------------------------ slot layout
// One expert slot = [gate/up section][down section].
//   bf16: per (128-row tile mt, K step ks of 64) one block of NMAT x 16 KB; each
//         16 KB is the 128 x 64 bf16 tile in the tensor core's 128-byte-swizzled
//         K-major image (16-byte chunk j of row r at chunk j ^ (r % 8)).
//         gate/up blocks hold gate then up for the same rows (NMAT = 2).
//   int4: per (mt, quantisation group g of 128 K) one block of NMAT x 8704 B:
//         8192 B of nibbles then 128 x (fp16 scale | fp16 zero << 16).  The
//         nibbles of row r, half h (K 0-63 / 64-127 of the group), quad j
//         (32 K each) form 16 bytes at ((h*2 + j)*128 + r)*16; each 32-bit word
//         w of a quad covers K elements 8w..8w+7 with element 2i in bits
//         [4i, 4i+4) and element 2i+1 in bits [16+4i, 20+4i).
//         The down section stores output tiles in pairs: per (pair 2p, 2p+1,
//         group g) the two tiles' blocks back to back, so that a GEMM step over
//         both tiles is one contiguous copy; with an odd tile count the last
//         tile follows alone, one block per group (i4_down_block).
//   fp8:  per (mt, g) one block of NMAT x 16640 B: the NMAT code tiles first,
//         each the 128 x 128-byte E4M3 image the tensor core reads (128-byte
//         swizzle: 16-byte chunk j of row r at chunk j ^ (r % 8)), then NMAT x
//         128 fp16 scales.  Within every 8-element K block the codes are stored
//         in the order {0,4,1,5,2,6,3,7} (the K order of the int4 decode path,
//         so both read the same token operand).  The down section pairs output
//         tiles like int4 (fp8_down_block).
constexpr int TILE_M = 128;          // weight rows per MMA tile (the MMA's M)
constexpr int KSTEP = 64;            // K elements per pipeline stage (one 128-byte row)
constexpr int QGROUP = 128;          // int4 quantisation group
constexpr int BF16_TILE_BYTES = TILE_M * KSTEP * 2;          // 16384
constexpr int I4_PACKED_BYTES = TILE_M * QGROUP / 2;         // 8192
constexpr int I4_MAT_BYTES = I4_PACKED_BYTES + TILE_M * 4;   // 8704
constexpr int F8_CODE_BYTES = TILE_M * QGROUP;                // 16384
constexpr int F8_MAT_BYTES = F8_CODE_BYTES + TILE_M * 2;       // 16640
// Readable bytes that must follow a [groups][rows] float array the int4
// decode GEMM reads per stage (group sums, unscale factors): it copies each
// item's row range as a 16-byte-aligned superset (at most 2 (bn + 1) floats past the end).
constexpr int SUMS_PAD_BYTES = 512;

// Bytes of one matrix block (one 128-row tile, one quantisation group) of a
// quantised format.
__host__ __device__ inline int quant_mat_bytes(int fmt) {
  return fmt == MOE_W_FP8_G128 ? F8_MAT_BYTES : I4_MAT_BYTES;
}
__host__ __device__ inline bool fmt_quantised(int fmt) {
  return fmt == MOE_W_INT4_G128 || fmt == MOE_W_FP8_G128;
}
__host__ __device__ inline size_t gateup_section_bytes(int fmt, int d, int F) {
  return fmt_quantised(fmt) ? (size_t)(F / TILE_M) * (d / QGROUP) * (2 * quant_mat_bytes(fmt))
                            : (size_t)(F / TILE_M) * (d / KSTEP) * (2 * BF16_TILE_BYTES);
}
// Byte offset, within the int4 down section, of output tile mt's block for
// quantisation group g (G groups per row, n_mt output tiles).
__host__ __device__ inline size_t i4_down_block(int mt, int g, int G, int n_mt) {
  const int p0 = mt & ~1;
  return p0 + 1 < n_mt ? ((size_t)p0 * G + 2 * g + (mt & 1)) * I4_MAT_BYTES
                       : ((size_t)mt * G + g) * I4_MAT_BYTES;
}
// fp8 down section, output tile mt, group g: where its block (one tile, or
// the pair holding it) starts, and the tile's place in it (0 alone or first,
// 1 second) and the number of tiles in the block.
__host__ __device__ inline size_t fp8_down_block(int mt, int g, int G, int n_mt, int& m, int& nmat) {
  const int p0 = mt & ~1;
  if (p0 + 1 < n_mt) {
    m = mt & 1;
    nmat = 2;
    return ((size_t)p0 * G + 2 * g) * F8_MAT_BYTES;
  }
  m = 0;
  nmat = 1;
  return ((size_t)mt * G + g) * F8_MAT_BYTES;
}
__host__ __device__ inline size_t down_section_bytes(int fmt, int d, int F) {
  return fmt_quantised(fmt) ? (size_t)(d / TILE_M) * (F / QGROUP) * quant_mat_bytes(fmt)
                            : (size_t)(d / TILE_M) * (F / KSTEP) * BF16_TILE_BYTES;
}
// Every slot ends in a 256-byte trailer after its two sections (both sections
// are multiples of 256 bytes, so the trailer keeps the slot 256-byte aligned):
//   float  L[2]   largest row L1 norm of the dequantised gate ([0]) and up ([1])
//                 weights, sum_k |w[n][k]| (accumulated by the prepack)
//   int32  B[2]   ceil(log2(L[m] * (1 + 2^-7))): powers of two that bound every
//                 gate / up output of a token row x by max|x| * 2^B[m]
// The quantised prefill GEMM sizes the fp16 scale of h from B (gemm.cu); the
// bf16 formats leave the trailer zero.
constexpr int SLOT_TRAILER_BYTES = 256;
__host__ __device__ inline size_t slot_payload_bytes(int fmt, int d, int F) {
  return gateup_section_bytes(fmt, d, F) + down_section_bytes(fmt, d, F);
}

// ------------------------------------------------------------------ grouped GEMM
// Row group g (an expert, or the shared expert appended as the last group) owns
// B-operand rows [offsets[g], offsets[g+1]).  Work items are
// (group, 128-row output tile, K split, row chunk of <= bn rows).
struct GemmArgs {
  const int32_t* offsets;               // [n_groups + 1]
  int n_groups;                         // groups (routed experts, + 1 shared)
  int n_routed;                         // groups [0, n_routed) use the routed table
  const uint8_t* pool_r;                // routed pool
  unsigned long long slot_bytes_r;
  const int32_t* e2s_r;                 // routed expert -> slot
  int n_slots_r;
  const uint8_t* pool_s;                // shared-expert pool view (group n_routed)
  unsigned long long slot_bytes_s;
  const int32_t* e2s_s;
  int n_slots_s;
  unsigned long long sec_off;           // byte offset of this GEMM's section in a slot
  int K;                                // reduction length, multiple of 128
  int n_mt;                             // 128-row output tiles
  int ksplit;                           // K splits (whole quantisation groups each)
  int bn;                               // max rows per item = B tile rows (16..256, % 16 == 0)
  int rows_total;                       // rows of the B operand
  void* out;                            // gate/up: bf16 h; down: fp32 partials
  int out_ld;                           // elements per output row
  unsigned long long out_split_stride;  // elements between K-split partial buffers
  int* err;                             // device error word
  // int4 decode GEMM (e4m3 B operand, see gemm_group.cu).  gate/up: per
  // (group, row) sums of the B rows [K/128][rows_total] and the rows' unscale
  // factors [rows_total]; where h goes: bytes [2*rows_total][out_ld] and
  // (sum, unscale factor) pairs [out_ld/128][rows_total][2].  down: b_sum =
  // those pairs of h.
  const float* b_sum;
  const float* b_scale;
  uint8_t* q_out;
  float* sum_out;
  // decode gate/up, stream-K split (gemm_group.cu): per CTA one partial
  // accumulator slot [grid][2][128][bn] and one ready flag [grid] (the flags
  // live in the workspace's error region and are zeroed by the forward's first
  // kernel).  null: every CTA takes whole items.
  float* sk_part;
  int* sk_flags;
  // quantised prefill GEMMs (gemm.cu): the token rows are fp16 copies of x
  // scaled per row by 2^ex (b_scale holds 2^-ex per row), h is fp16 scaled per
  // row by 2^eh, eh from ex and the slot trailer's bounds (at trailer_off)
  unsigned long long trailer_off;
  int n_a, n_b, n_raw;                  // pipeline depths
  uint32_t tmem_cols;                   // TMEM columns (power of two >= 32)
  unsigned long long wait_ns;           // limit of every wait (MOE_WAIT_LIMIT_NS unless a test sets it)
  int stop_stage;                       // test hook: the producer issues no stage at or past this
                                        // index (-1: off), so that a consumer's wait runs out
};

struct GemmPlan {
  bool group;         // int4 group-scaled main loop (row chunks of <= 32)
  bool pair;          // group loop, down GEMM: two 128-row output tiles per stage
  int ndq;            // dequant / epilogue warps
  int n_a, n_b, n_raw;
  size_t smem_bytes;
  uint32_t tmem_cols;
};

// Quantised layers run their prefill-size GEMMs on fp16 operands (x_perm and h
// are fp16, each row scaled by a power of two, see gemm.cu); bf16 layers on
// bf16 operands.
inline bool gemm_uses_fp16(int fmt) { return fmt_quantised(fmt); }

// Uses the group-scaled decode kernel (int4 or fp8, row chunks of <= 32)?
inline bool gemm_is_group(int fmt, int bn) { return fmt_quantised(fmt) && bn <= 32; }
// Work tiles per (group, row chunk, K split) of the down GEMM with n_mt output
// tiles: the quantised kernels pair adjacent tiles when n_mt is even.
inline bool down_paired(int fmt, int n_mt) { return fmt_quantised(fmt) && n_mt % 2 == 0; }
inline int down_work_tiles(int fmt, int n_mt) { return down_paired(fmt, n_mt) ? n_mt / 2 : n_mt; }
// Row-chunk width (the GEMMs' N): a power of two >= twice the mean rows per
// expert, 16..256; quantised layers stop at 192 so that the gate and up
// accumulators (2 x 192 TMEM columns) leave room for the dequantised A tiles.
inline int choose_bn(int A, int E, int fmt) {
  const int mean = (A + E - 1) / E;
  int bn = 16;
  while (bn < 2 * mean && bn < 256) bn <<= 1;
  if (fmt_quantised(fmt) && bn > 128) bn = 192;
  return bn;
}

GemmPlan plan_gemm(int fmt, bool gateup, int bn, int n_groups, int n_mt);
cudaError_t launch_grouped_gemm(int fmt, bool gateup, const CUtensorMap& tmap_b, GemmArgs args,
                                const GemmPlan& plan, int grid, cudaStream_t stream, bool pdl = false);

// One kernel launch; pdl: programmatic stream serialisation (see below).
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                          bool pdl, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

// ------------------------------------------------------------------ other kernels
// logits[t][e] = x[t] . w_router[e] (bf16 inputs, fp32 sums; router.cu).
cudaError_t launch_router_logits(const uint16_t* x, const uint16_t* w_router, int T, int d, int E,
                                 float* logits, int n_sm, cudaStream_t s, bool pdl = false);
// err_clear (nullable): error word zeroed by the first thread (first launch of a forward).
cudaError_t launch_route_topk(const float* logits, int T, int E, int k, int32_t* idx, float* w,
                              int* err_clear, cudaStream_t s, bool pdl = false);
// The launches below take pdl = true when the previous kernel in the stream
// belongs to the same call (programmatic dependent launch: this kernel's
// prologue overlaps that kernel's tail; it reads nothing before
// griddep_wait()).  The first kernel of every entry point launches normally,
// so it never overlaps the caller's earlier work.
cudaError_t launch_permute_index(const int32_t* idx, int T, int k, int E, int t_shared,
                                 int32_t* counts, int32_t* offsets, int32_t* row_of_assign,
                                 int32_t* token_of_row, int* err, cudaStream_t s, bool pdl = false);
// Routing, permutation and row gather in one launch, for batches of up to
// FUSED_ROUTE_MAX_T tokens: the outputs of launch_route_topk,
// launch_permute_index and the row gather (out: GATHER_BF16 into dst.x16
// [rows][d]; GATHER_F16 into dst.x16 and dst.xe, the scaled fp16 rows of
// launch_gather_rows_f16; GATHER_FP8 into dst.xq/xs/xe, the quantised decode
// GEMMs' e4m3 form), rows = T*k (+ t_shared).
constexpr int FUSED_ROUTE_MAX_T = 64;
enum { GATHER_BF16 = 0, GATHER_F16 = 1, GATHER_FP8 = 2 };
struct GatherDst {
  uint16_t* x16;
  uint8_t* xq;
  float *xs, *xe;
};
// router (nullable): compute the logits first, in the same launch, from x and
// the router weight (written to `logits`, then routed; see permute.cu).
struct RouterSrc {
  const uint16_t* w_router;   // bf16 [E][d]
  int tt;                     // token tile of the router GEMM (router_token_tile)
  int* sync;                  // grid-barrier counter, zero at launch
};
cudaError_t launch_route_gather(const float* logits, int T, int k, int E, int t_shared, const uint16_t* x,
                                int d, int32_t* idx, float* w, int32_t* counts, int32_t* offsets,
                                int32_t* row_of_assign, int32_t* token_of_row, int* err, int out,
                                const GatherDst& dst, int n_sm, cudaStream_t s, bool pdl = false,
                                const RouterSrc* router = nullptr);
// x_perm[r] = x[token_of_row[r]] (bf16).  token_of_row == nullptr: x_perm[r] = x[r].
cudaError_t launch_gather_rows(const uint16_t* x, const int32_t* token_of_row, int rows, int T,
                               int d, uint16_t* x_perm, int n_sm, cudaStream_t s, bool pdl = false);
// The quantised prefill GEMMs' fp16 rows: x16[r] = fp16(x[token_of_row[r]] *
// 2^ex_r) with ex_r putting the row's largest magnitude in [2^13, 2^14) (exact
// for bf16 inputs down to 2^-27 of that magnitude), xe[r] = 2^-ex_r.
// token_of_row == nullptr: rows of x in order.
cudaError_t launch_gather_rows_f16(const uint16_t* x, const int32_t* token_of_row, int rows, int T,
                                   int d, uint16_t* x16, float* xe, int n_sm, cudaStream_t s,
                                   bool pdl = false);
// The int4 decode GEMM's e4m3 form of the gathered rows (see permute.cu):
// xq [2*rows][d] bytes (hi rows, then lo rows), xs [d/128][rows], xe [rows].
cudaError_t launch_gather_rows_fp8(const uint16_t* x, const int32_t* token_of_row, int rows, int T,
                                   int d, uint8_t* xq, float* xs, float* xe, int n_sm, cudaStream_t s,
                                   bool pdl = false);
cudaError_t launch_combine_partials(const float* part, int n_split, size_t split_stride,
                                    const int32_t* row_of_assign, const float* topk_w, int T,
                                    int k, int d, int shared_row0, uint16_t* out, cudaStream_t s,
                                    bool pdl = false);
cudaError_t launch_combine_bf16(const uint16_t* y_perm, const int32_t* row_of_assign,
                                const float* topk_w, const uint16_t* shared_y, int T, int k, int d,
                                uint16_t* out, cudaStream_t s);
cudaError_t launch_reduce_splits(const float* part, int n_split, size_t split_stride, int rows,
                                 int d, uint16_t* y, cudaStream_t s, bool pdl = false);
// Zeroes the 256 words of a workspace's error region (error word + GEMM flags).
cudaError_t launch_clear_word(int* p, cudaStream_t s);
cudaError_t launch_prepack(int fmt, int d, int F, const moe_expert_src& src, uint8_t* dst,
                           cudaStream_t s);

}  // namespace moe
