// abi.cu -- the extern "C" entry points declared in include/moe.h: host-side
// argument checks, workspace carve-up, TMA tensor maps and the launch sequence
//   route -> permute -> gather -> gate/up GEMM -> down GEMM -> combine
// (one stream, nothing allocated, nothing synchronised).
#include <cudaTypedefs.h>

#include <mutex>

#include "kernels.cuh"
#include "router_tc.h"
#include "nvtx_range.h"
#include "router_dev.cuh"

using namespace moe;

namespace {

constexpr int MAX_E = 256;
constexpr int MAX_K = 16;
constexpr int MAX_A = 1 << 20;
constexpr int MAX_DIM = 32768;
constexpr int MAX_KSPLIT = 8;
constexpr int SPLIT_GRID = 152;     // persistent CTAs the decode split is balanced for (GB300 SMs)

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

bool have_encoder() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode != nullptr;
}

int sm_count() {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 148;
  if (dev < 64 && cache[dev]) return cache[dev];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
  if (dev < 64) cache[dev] = n;
  return n;
}

inline bool al16(const void* p) { return ((uintptr_t)p & 15u) == 0; }
inline bool al256(const void* p) { return ((uintptr_t)p & 255u) == 0; }
inline size_t up1k(size_t x) { return (x + 1023) & ~(size_t)1023; }

// 16-bit row-major [rows][K] (bf16 or fp16) -> TMA map with a {64 x box_rows}
// box and the 128-byte swizzle.
bool make_row_map(CUtensorMap* m, const void* base, int rows, int K, int box_rows, bool fp16) {
  if (!have_encoder()) return false;
  cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)K * 2};
  cuuint32_t box[2] = {(cuuint32_t)KSTEP, (cuuint32_t)box_rows};
  cuuint32_t es[2] = {1, 1};
  return g_encode(m, fp16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                  const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Byte rows [rows][K] (e4m3) -> TMA map with a {128 x box_rows} box (one
// 128-byte row per token row and quantisation group) and the 128-byte swizzle.
bool make_byte_row_map(CUtensorMap* m, const void* base, int rows, int K, int box_rows) {
  if (!have_encoder()) return false;
  cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)K};
  cuuint32_t box[2] = {(cuuint32_t)QGROUP, (cuuint32_t)box_rows};
  cuuint32_t es[2] = {1, 1};
  return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

moe_status check_pool(const moe_pool* p, bool single) {
  if (!p || !p->pool || !p->expert_to_slot) return MOE_ERR_INVALID_ARG;
  if (p->fmt != MOE_W_BF16 && !fmt_quantised(p->fmt)) return MOE_ERR_INVALID_ARG;
  if (p->n_experts < 1 || p->n_slots < 1) return MOE_ERR_INVALID_ARG;
  if (single && p->n_experts != 1) return MOE_ERR_INVALID_ARG;
  if (p->n_experts > MAX_E) return MOE_ERR_UNSUPPORTED;
  if (p->d_model < 128 || p->d_ff < 128 || p->d_model % 128 || p->d_ff % 128)
    return MOE_ERR_INVALID_ARG;
  if (p->d_model > MAX_DIM || p->d_ff > MAX_DIM) return MOE_ERR_UNSUPPORTED;
  if (!al256(p->pool) || p->slot_bytes % 256 ||
      p->slot_bytes < moe_slot_bytes(p->fmt, p->d_model, p->d_ff))
    return MOE_ERR_INVALID_ARG;
  if (!al16(p->expert_to_slot)) return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

// Largest chunk of one expert's rows that one work item covers (the B tile height).
// K split of the down GEMM.  Decode (group kernel): the split whose items
// spread most evenly over the persistent CTAs (fewest quantisation groups on
// the busiest CTA; its fp32 partials are small).  Otherwise the same count of
// waves times groups per item, each group priced at its MMA time or its weight
// streaming time (whichever is longer, from nominal per-SM rates), plus the
// fp32 partials each split writes and the combine reads back (rows x d x 8
// bytes per split, large for long batches).
int choose_ksplit(int A, int E, bool has_shared, int bn, int fmt, int d, int F, int rows) {
  const int active = (A < E ? A : E) + (has_shared ? 1 : 0);
  const int mean = (A + E - 1) / E;
  const int nch = mean > bn ? (mean + bn - 1) / bn : 1;
  const int G = F / QGROUP;
  const int smax = MAX_KSPLIT < G ? MAX_KSPLIT : G;
  const long items = (long)active * down_work_tiles(fmt, d / TILE_M) * nch;
  if (gemm_is_group(fmt, bn)) {
    int best_s = 1;
    long best = -1;
    for (int s = 1; s <= smax; ++s) {
      const long waves = (items * s + SPLIT_GRID - 1) / SPLIT_GRID;
      const long cost = waves * ((G + s - 1) / s);
      if (best < 0 || cost < best) { best = cost; best_s = s; }
    }
    return best_s;
  }
  const double sm_flops = 1.9e15 / SPLIT_GRID, sm_bytes = 6.8e12 / SPLIT_GRID;   // per SM per s
  const int tiles = down_paired(fmt, d / TILE_M) ? 2 : 1;                        // output tiles per item
  const double wbytes = fmt == MOE_W_BF16 ? 2.0 : (double)quant_mat_bytes(fmt) / (TILE_M * QGROUP);
  const double chunk_rows = mean < bn ? mean : bn;
  const double t_mma = 2.0 * tiles * TILE_M * chunk_rows * QGROUP / sm_flops;
  const double t_stream = tiles * TILE_M * QGROUP * wbytes / sm_bytes;
  const double t_group = t_mma > t_stream ? t_mma : t_stream;
  const double t_split = (double)rows * d * 8.0 / 6.8e12;
  int best_s = 1;
  double best = -1.0;
  for (int s = 1; s <= smax; ++s) {
    const long waves = (items * s + SPLIT_GRID - 1) / SPLIT_GRID;
    const double cost = (double)waves * ((G + s - 1) / s) * t_group + s * t_split;
    if (best < 0 || cost < best) { best = cost; best_s = s; }
  }
  return best_s;
}

// The int4 decode GEMMs' e4m3 operands (see gemm_group.cu): the gathered rows
// and h as hi/lo byte rows [2*rows][K]; for x per (group, row) sums
// [d/128][rows] and per-row unscale factors [rows]; for h per (group, row)
// (sum, unscale factor) pairs [F/128][rows][2].
struct Fp8Rows {
  uint8_t* xq;
  float *xs, *xe;
  uint8_t* hq;
  float* hs;
  float* skp;   // the gate/up GEMM's stream-K partial slots [grid][2][128][bn]
};
struct Fp8Offsets {
  size_t xq, xs, xe, hq, hs, skp;
};
// Appends the e4m3 regions at offset o (1 KB aligned) and returns the new end.
size_t fp8_regions(Fp8Offsets& f, size_t o, int rows, int d, int F, int bn) {
  f.xq = o;  o = up1k(o + 2 * (size_t)rows * d);
  f.xs = o;  o = up1k(o + (size_t)(d / QGROUP) * rows * 4 + SUMS_PAD_BYTES);
  f.xe = o;  o = up1k(o + (size_t)rows * 4);
  f.hq = o;  o = up1k(o + 2 * (size_t)rows * F);
  f.hs = o;  o = up1k(o + (size_t)(F / QGROUP) * rows * 8 + SUMS_PAD_BYTES);
  f.skp = o; o = up1k(o + (size_t)sm_count() * 2 * TILE_M * bn * 4);
  return o;
}
Fp8Rows fp8_rows(uint8_t* W, const Fp8Offsets& f) {
  return Fp8Rows{W + f.xq, (float*)(W + f.xs), (float*)(W + f.xe), W + f.hq, (float*)(W + f.hs),
                 (float*)(W + f.skp)};
}

struct LayerLayout {
  int A, Tsh, rows, E, d, F, bn, ksplit;
  size_t sync;   // the fused router's grid-barrier counter
  bool fp8;   // quantised decode path: e4m3 operands instead of x_perm / h
  bool f16;   // quantised prefill path: fp16 x_perm and h, scaled per row (xe: 2^-ex per row)
  size_t err, idx, w, counts, offsets, roa, tor, xperm, xe, h, part, total;
  Fp8Offsets f8;
};

LayerLayout layer_layout(int T, int k, const moe_pool* routed, const moe_pool* shared) {
  LayerLayout L{};
  L.A = T * k;
  L.Tsh = shared ? T : 0;
  L.rows = L.A + L.Tsh;
  L.E = routed->n_experts;
  L.d = routed->d_model;
  L.F = routed->d_ff;
  L.bn = choose_bn(L.A, L.E, routed->fmt);
  L.ksplit = choose_ksplit(L.A, L.E, shared != nullptr, L.bn, routed->fmt, L.d, L.F, L.rows);
  size_t o = 0;
  L.err = o;      o += 1024;
  L.sync = o;     o += 1024;
  L.idx = o;      o = up1k(o + (size_t)L.A * 4);
  L.w = o;        o = up1k(o + (size_t)L.A * 4);
  L.counts = o;   o = up1k(o + (size_t)(L.E + 1) * 4);
  L.offsets = o;  o = up1k(o + (size_t)(L.E + 2) * 4);
  L.roa = o;      o = up1k(o + (size_t)L.A * 4);
  L.tor = o;      o = up1k(o + (size_t)L.rows * 4);
  L.fp8 = gemm_is_group(routed->fmt, L.bn);
  L.f16 = !L.fp8 && gemm_uses_fp16(routed->fmt);
  L.xperm = o;    o = up1k(o + (L.fp8 ? 0 : (size_t)L.rows * L.d * 2));
  L.xe = o;       o = up1k(o + (L.f16 ? (size_t)L.rows * 4 : 0));
  L.h = o;        o = up1k(o + (L.fp8 ? 0 : (size_t)L.rows * L.F * 2));
  L.part = o;     o = up1k(o + (size_t)L.ksplit * L.rows * L.d * 4);
  if (L.fp8) o = fp8_regions(L.f8, o, L.rows, L.d, L.F, L.bn);
  L.total = o;
  return L;
}

// Failure-path test hook (moe_debug_gemm_fault): the gate/up GEMM's producer
// stops after this many stages (-1: never) and the GEMMs' waits give up after
// this long.  Host globals, read when a forward is enqueued.
int g_fault_stop_stage = -1;
unsigned long long g_fault_wait_ns = MOE_WAIT_LIMIT_NS;

// The router GEMM: tensor cores for long batches of at most 16 experts, else
// the CUDA-core kernel.
// With idx != nullptr the tensor-core kernel also does the top-k gating of its
// rows (*topk_done = true); the CUDA-core kernel leaves it to the routing kernel.
cudaError_t run_router(const uint16_t* x, const uint16_t* w_router, int T, int d, int E, float* logits,
                       int* err, cudaStream_t s, bool pdl, int k = 0, int32_t* idx = nullptr,
                       float* w = nullptr, bool* topk_done = nullptr) {
  if (topk_done) *topk_done = false;
  if (router_uses_tensor_cores(T, d, E)) {
    CUtensorMap tx, tw;
    if (!make_row_map(&tx, x, T, d, 128, false) || !make_row_map(&tw, w_router, E, d, 16, false))
      return cudaErrorInvalidValue;
    if (topk_done) *topk_done = idx != nullptr;
    return launch_router_topk_tc(tx, tw, T, d, E, logits, idx != nullptr ? k : 0, idx, w, err, g_fault_stop_stage,
                                 g_fault_wait_ns, s, pdl);
  }
  return launch_router_logits(x, w_router, T, d, E, logits, sm_count(), s, pdl);
}

GemmArgs base_args(const moe_pool* routed, const moe_pool* shared, int* err) {
  GemmArgs a{};
  a.wait_ns = g_fault_wait_ns;
  a.stop_stage = -1;
  a.n_routed = routed->n_experts;
  a.pool_r = (const uint8_t*)routed->pool;
  a.slot_bytes_r = routed->slot_bytes;
  a.e2s_r = routed->expert_to_slot;
  a.n_slots_r = routed->n_slots;
  if (shared) {
    a.pool_s = (const uint8_t*)shared->pool;
    a.slot_bytes_s = shared->slot_bytes;
    a.e2s_s = shared->expert_to_slot;
    a.n_slots_s = shared->n_slots;
  } else {
    a.pool_s = a.pool_r;
    a.slot_bytes_s = a.slot_bytes_r;
    a.e2s_s = a.e2s_r;
    a.n_slots_s = a.n_slots_r;
  }
  a.err = err;
  return a;
}

// gate/up (SwiGLU) then down over the row groups described by `offsets`.
// x_rows and h are fp16 for quantised pools (x_rows scaled per row, x_unscale =
// 2^-ex per row), bf16 otherwise; with f8 (the quantised decode path) the GEMMs
// read and write the e4m3 forms instead.  pdl: both
// launches follow a kernel of the same call (dependent launch).
moe_status run_ffn(const uint16_t* x_rows, const float* x_unscale, const int32_t* offsets, int n_groups,
                   int rows, const moe_pool* routed, const moe_pool* shared, int bn, int ksplit, uint16_t* h,
                   float* part, const Fp8Rows* f8, int* err, cudaStream_t s, bool pdl,
                   cudaEvent_t ev_mid, cudaEvent_t ev_down) {
  const int d = routed->d_model, F = routed->d_ff, fmt = routed->fmt;
  const bool f16 = gemm_uses_fp16(fmt);
  const int grid = sm_count();
  CUtensorMap mx, mh;
  if (f8) {
    if (!make_byte_row_map(&mx, f8->xq, 2 * rows, d, bn) || !make_byte_row_map(&mh, f8->hq, 2 * rows, F, bn))
      return MOE_ERR_CUDA;
  } else if (!make_row_map(&mx, x_rows, rows, d, bn, f16) || !make_row_map(&mh, h, rows, F, bn, f16)) {
    return MOE_ERR_CUDA;
  }
  GemmArgs a = base_args(routed, shared, err);
  a.offsets = offsets;
  a.n_groups = n_groups;
  a.bn = bn;
  a.rows_total = rows;
  a.trailer_off = slot_payload_bytes(fmt, d, F);
  a.b_scale = x_unscale;   // the prefill GEMMs' per-row x unscale (decode gate/up: set below)

  GemmArgs g = a;   // gate/up + SwiGLU
  g.sec_off = 0;
  g.K = d;
  g.n_mt = F / TILE_M;
  g.ksplit = 1;
  g.out = h;
  g.out_ld = F;
  g.out_split_stride = 0;
  if (f8) {
    g.out = nullptr;
    g.b_sum = f8->xs;
    g.b_scale = f8->xe;
    g.q_out = f8->hq;
    g.sum_out = f8->hs;
    // ready flags err[1 .. grid] after the error word, in the workspace's 1 KB
    // (256-word) error region; a finishing CTA b reads the flag of CTA b + 1
    if (grid + 2 <= 256) {
      g.sk_part = f8->skp;
      g.sk_flags = err + 1;
    }
  }
  g.stop_stage = g_fault_stop_stage;
  if (launch_grouped_gemm(fmt, true, mx, g, plan_gemm(fmt, true, bn, n_groups, F / TILE_M), grid, s,
                          pdl) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (ev_mid && cudaEventRecord(ev_mid, s) != cudaSuccess) return MOE_ERR_CUDA;

  GemmArgs dn = a;   // down, K-split fp32 partial sums
  dn.sec_off = gateup_section_bytes(fmt, d, F);
  dn.K = F;
  dn.n_mt = d / TILE_M;
  dn.ksplit = ksplit;
  dn.out = part;
  dn.out_ld = d;
  dn.out_split_stride = (unsigned long long)rows * d;
  if (f8) {
    dn.b_sum = f8->hs;
  }
  if (launch_grouped_gemm(fmt, false, mh, dn, plan_gemm(fmt, false, bn, n_groups, d / TILE_M), grid, s,
                          pdl && !ev_mid) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (ev_down && cudaEventRecord(ev_down, s) != cudaSuccess) return MOE_ERR_CUDA;
  return MOE_OK;
}

moe_status check_route_args(const float* logits, int T, int E, int k, const void* idx,
                            const void* w) {
  if (!logits || !idx || !w) return MOE_ERR_INVALID_ARG;
  if (T < 1 || E < 1 || k < 1 || k > E) return MOE_ERR_INVALID_ARG;
  if (E > MAX_E || k > MAX_K || (long)T * k > MAX_A) return MOE_ERR_UNSUPPORTED;
  if (!al16(logits) || !al16(idx) || !al16(w)) return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

// w_router (nullable): the router GEMM comes first and writes `logits` (then
// an output of the call): fused into the routing launch for batches of up to
// FUSED_ROUTE_MAX_T tokens, its own launch before the routing kernel (which may
// then start early) otherwise.
moe_status layer_forward_impl(const uint16_t* x, const float* logits, int T, int k,
                              const moe_pool* routed, const moe_pool* shared, uint16_t* out,
                              void* ws, size_t ws_bytes, cudaStream_t s, void* const* ev,
                              const uint16_t* w_router = nullptr) {
  moe_status st = check_pool(routed, false);
  if (st != MOE_OK) return st;
  if (shared) {
    if ((st = check_pool(shared, true)) != MOE_OK) return st;
    if (shared->d_model != routed->d_model || shared->d_ff != routed->d_ff ||
        shared->fmt != routed->fmt)
      return MOE_ERR_UNSUPPORTED;
  }
  if (!x || !logits || !out || !ws) return MOE_ERR_INVALID_ARG;
  const int E = routed->n_experts;
  if (T < 1 || k < 1 || k > E) return MOE_ERR_INVALID_ARG;
  if (k > MAX_K || (long)T * k > MAX_A) return MOE_ERR_UNSUPPORTED;
  if (!al16(x) || !al16(logits) || !al16(out) || !al256(ws)) return MOE_ERR_INVALID_ARG;
  const LayerLayout L = layer_layout(T, k, routed, shared);
  if (ws_bytes < L.total) return MOE_ERR_WORKSPACE;
  uint8_t* W = (uint8_t*)ws;
  int* err = (int*)(W + L.err);
  int32_t* idx = (int32_t*)(W + L.idx);
  float* w = (float*)(W + L.w);
  int32_t* counts = (int32_t*)(W + L.counts);
  int32_t* offsets = (int32_t*)(W + L.offsets);
  int32_t* roa = (int32_t*)(W + L.roa);
  int32_t* tor = (int32_t*)(W + L.tor);
  uint16_t* xperm = (uint16_t*)(W + L.xperm);
  float* xe = L.f16 ? (float*)(W + L.xe) : nullptr;
  uint16_t* h = (uint16_t*)(W + L.h);
  float* part = (float*)(W + L.part);
  const Fp8Rows f8 = L.fp8 ? fp8_rows(W, L.f8) : Fp8Rows{};
  auto rec = [&](int i) -> bool {
    return !ev || !ev[i] || cudaEventRecord((cudaEvent_t)ev[i], s) == cudaSuccess;
  };
  // the kernels after the first start early (dependent launch), except when
  // stage events sit between them
  const bool pdl = ev == nullptr;

  if (!rec(MOE_STAGE_ROUTE)) return MOE_ERR_CUDA;
  if (T <= FUSED_ROUTE_MAX_T) {   // one launch; its time is reported as the routing stage
    const GatherDst dst{xperm, f8.xq, f8.xs, L.fp8 ? f8.xe : xe};
    const int out_kind = L.fp8 ? GATHER_FP8 : L.f16 ? GATHER_F16 : GATHER_BF16;
    const RouterSrc rs{w_router, router_token_tile(T, E, sm_count()), (int*)(W + L.sync)};
    // the router's barrier counter and the error region (which the routing
    // kernel then leaves as it is), zero before the cooperative launch
    if (w_router && cudaMemsetAsync(W + L.err, 0, L.sync + sizeof(int) - L.err, s) != cudaSuccess)
      return MOE_ERR_CUDA;
    if (launch_route_gather(logits, T, k, E, L.Tsh, x, L.d, idx, w, counts, offsets, roa, tor, err,
                            out_kind, dst, sm_count(), s, false, w_router ? &rs : nullptr) != cudaSuccess)
      return MOE_ERR_CUDA;
    if (!rec(MOE_STAGE_PERMUTE) || !rec(MOE_STAGE_GATHER)) return MOE_ERR_CUDA;
  } else {
    // the router (on the tensor cores: with the top-k gating of its rows fused in)
    bool topk_done = false;
    if (w_router && run_router(x, w_router, T, L.d, E, const_cast<float*>(logits), nullptr, s, false, k, idx, w,
                               &topk_done) != cudaSuccess)
      return MOE_ERR_CUDA;
    if (!topk_done && launch_route_topk(logits, T, E, k, idx, w, nullptr, s, w_router != nullptr && pdl) != cudaSuccess)
      return MOE_ERR_CUDA;
    if (!rec(MOE_STAGE_PERMUTE)) return MOE_ERR_CUDA;
    if (launch_permute_index(idx, T, k, E, L.Tsh, counts, offsets, roa, tor, err, s, pdl) != cudaSuccess)
      return MOE_ERR_CUDA;
    if (!rec(MOE_STAGE_GATHER)) return MOE_ERR_CUDA;
    if (L.fp8) {
      if (launch_gather_rows_fp8(x, tor, L.rows, T, L.d, f8.xq, f8.xs, f8.xe, sm_count(), s, pdl) !=
          cudaSuccess)
        return MOE_ERR_CUDA;
    } else if (L.f16) {
      if (launch_gather_rows_f16(x, tor, L.rows, T, L.d, xperm, xe, sm_count(), s, pdl) != cudaSuccess)
        return MOE_ERR_CUDA;
    } else if (launch_gather_rows(x, tor, L.rows, T, L.d, xperm, sm_count(), s, pdl) != cudaSuccess) {
      return MOE_ERR_CUDA;
    }
  }
  if (!rec(MOE_STAGE_GATE_UP)) return MOE_ERR_CUDA;
  st = run_ffn(xperm, xe, offsets, E + (shared ? 1 : 0), L.rows, routed, shared, L.bn, L.ksplit, h, part,
               L.fp8 ? &f8 : nullptr, err, s, pdl, ev ? (cudaEvent_t)ev[MOE_STAGE_DOWN] : nullptr,
               ev ? (cudaEvent_t)ev[MOE_STAGE_COMBINE] : nullptr);
  if (st != MOE_OK) return st;
  if (launch_combine_partials(part, L.ksplit, (size_t)L.rows * L.d, roa, w, T, k, L.d,
                              shared ? L.A : -1, out, s, pdl) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (!rec(MOE_N_STAGES)) return MOE_ERR_CUDA;
  return MOE_OK;
}

}  // namespace

// ===================================================================== C ABI
extern "C" {

const char* moe_status_str(int status) {
  switch (status) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported size or format";
    case MOE_ERR_WORKSPACE: return "workspace too small";
    case MOE_ERR_CUDA: return "CUDA launch failed";
    case MOE_ERR_DEVICE: return "device-side error code set";
    default: return "unknown status";
  }
}

size_t moe_slot_bytes(int fmt, int d_model, int d_ff) {
  if ((fmt != MOE_W_BF16 && !fmt_quantised(fmt)) || d_model < 128 || d_ff < 128 ||
      d_model % 128 || d_ff % 128)
    return 0;
  return slot_payload_bytes(fmt, d_model, d_ff) + SLOT_TRAILER_BYTES;
}

moe_status moe_prepack_expert(int fmt, int d_model, int d_ff, const moe_expert_src* src,
                              void* slot_dst, moe_stream_t stream) {
  const moe::NvtxRange nvtx_range("moe_prepack_expert");
  if (!src || !slot_dst || moe_slot_bytes(fmt, d_model, d_ff) == 0) return MOE_ERR_INVALID_ARG;
  if (d_model > MAX_DIM || d_ff > MAX_DIM) return MOE_ERR_UNSUPPORTED;
  if (!al256(slot_dst)) return MOE_ERR_INVALID_ARG;
  for (int m = 0; m < 3; ++m) {
    if (!src->w[m] || !al16(src->w[m])) return MOE_ERR_INVALID_ARG;
    if (fmt == MOE_W_INT4_G128 && (!src->scale[m] || !src->zero[m])) return MOE_ERR_INVALID_ARG;
    if (fmt == MOE_W_FP8_G128 && !src->scale[m]) return MOE_ERR_INVALID_ARG;
  }
  return launch_prepack(fmt, d_model, d_ff, *src, (uint8_t*)slot_dst, (cudaStream_t)stream) ==
                 cudaSuccess
             ? MOE_OK
             : MOE_ERR_CUDA;
}

moe_status check_router_args(const uint16_t* x, const uint16_t* w_router, int T, int d, int E,
                             const float* logits) {
  if (!x || !w_router || !logits) return MOE_ERR_INVALID_ARG;
  if (T < 1 || d < 8 || d % 8 || E < 1) return MOE_ERR_INVALID_ARG;
  if (E > MAX_E || d > MAX_DIM) return MOE_ERR_UNSUPPORTED;
  if (!al16(x) || !al16(w_router) || !al16(logits)) return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

moe_status moe_router_logits(const uint16_t* x, const uint16_t* w_router, int T, int d, int E,
                             float* logits, moe_stream_t stream) {
  const moe::NvtxRange nvtx_range("moe_router_logits");
  const moe_status st = check_router_args(x, w_router, T, d, E, logits);
  if (st != MOE_OK) return st;
  return run_router(x, w_router, T, d, E, logits, nullptr, (cudaStream_t)stream, false) == cudaSuccess
             ? MOE_OK
             : MOE_ERR_CUDA;
}

moe_status moe_route_topk(const float* logits, int T, int E, int k, int32_t* topk_idx,
                          float* topk_w, moe_stream_t stream) {
  const moe::NvtxRange nvtx_range("moe_route_topk");
  const moe_status st = check_route_args(logits, T, E, k, topk_idx, topk_w);
  if (st != MOE_OK) return st;
  return launch_route_topk(logits, T, E, k, topk_idx, topk_w, nullptr, (cudaStream_t)stream) ==
                 cudaSuccess
             ? MOE_OK
             : MOE_ERR_CUDA;
}

size_t moe_permute_workspace_bytes(void) { return 1024; }

moe_status moe_permute(const int32_t* topk_idx, const uint16_t* x, int T, int k, int E, int d,
                       int32_t* counts, int32_t* offsets, int32_t* row_of_assign,
                       int32_t* token_of_row, uint16_t* x_perm, void* ws, size_t ws_bytes,
                       moe_stream_t stream) {
  const moe::NvtxRange nvtx_range("moe_permute");
  if (!topk_idx || !x || !counts || !offsets || !row_of_assign || !token_of_row || !x_perm || !ws)
    return MOE_ERR_INVALID_ARG;
  if (T < 1 || E < 1 || k < 1 || k > E || d < 128 || d % 128) return MOE_ERR_INVALID_ARG;
  if (E > MAX_E || k > MAX_K || (long)T * k > MAX_A || d > MAX_DIM) return MOE_ERR_UNSUPPORTED;
  if (!al16(topk_idx) || !al16(x) || !al16(x_perm) || !al256(ws)) return MOE_ERR_INVALID_ARG;
  if (ws_bytes < moe_permute_workspace_bytes()) return MOE_ERR_WORKSPACE;
  cudaStream_t s = (cudaStream_t)stream;
  int* err = (int*)ws;
  if (launch_permute_index(topk_idx, T, k, E, 0, counts, offsets, row_of_assign, token_of_row, err,
                           s) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (launch_gather_rows(x, token_of_row, T * k, T, d, x_perm, sm_count(), s, true) !=
      cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}

// Workspace of the standalone grouped FFN: error word, h, down partials and,
// for quantised pools, the scaled fp16 copy of x_perm with its per-row unscale
// factors (prefill path) or the e4m3 operands (decode path).
struct FfnLayout {
  int bn, ksplit;
  bool fp8;
  size_t h, part, x16, xe, total;
  Fp8Offsets f8;
};

FfnLayout ffn_layout(int A, const moe_pool* pool) {
  FfnLayout L{};
  const int d = pool->d_model, F = pool->d_ff;
  L.bn = choose_bn(A, pool->n_experts, pool->fmt);
  L.ksplit = choose_ksplit(A, pool->n_experts, false, L.bn, pool->fmt, d, F, A);
  const bool f16 = gemm_uses_fp16(pool->fmt);
  L.fp8 = gemm_is_group(pool->fmt, L.bn);
  size_t o = 1024;
  L.h = o;     o = up1k(o + (L.fp8 ? 0 : (size_t)A * F * 2));
  L.part = o;  o = up1k(o + (size_t)L.ksplit * A * d * 4);
  L.x16 = o;   o = up1k(o + (f16 && !L.fp8 ? (size_t)A * d * 2 : 0));
  L.xe = o;    o = up1k(o + (f16 && !L.fp8 ? (size_t)A * 4 : 0));
  if (L.fp8) o = fp8_regions(L.f8, o, A, d, F, L.bn);
  L.total = o;
  return L;
}

size_t moe_grouped_ffn_workspace_bytes(int A, const moe_pool* pool) {
  if (A < 1 || check_pool(pool, false) != MOE_OK) return 0;
  return ffn_layout(A, pool).total;
}

moe_status moe_grouped_ffn(const uint16_t* x_perm, const int32_t* offsets, int A,
                           const moe_pool* pool, uint16_t* y_perm, void* ws, size_t ws_bytes,
                           moe_stream_t stream) {
  const moe::NvtxRange nvtx_range("moe_grouped_ffn");
  moe_status st = check_pool(pool, false);
  if (st != MOE_OK) return st;
  if (!x_perm || !offsets || !y_perm || !ws || A < 1) return MOE_ERR_INVALID_ARG;
  if (A > MAX_A) return MOE_ERR_UNSUPPORTED;
  if (!al16(x_perm) || !al16(offsets) || !al16(y_perm) || !al256(ws)) return MOE_ERR_INVALID_ARG;
  const FfnLayout L = ffn_layout(A, pool);
  if (ws_bytes < L.total) return MOE_ERR_WORKSPACE;
  uint8_t* W = (uint8_t*)ws;
  int* err = (int*)W;
  uint16_t* h = (uint16_t*)(W + L.h);
  float* part = (float*)(W + L.part);
  cudaStream_t s = (cudaStream_t)stream;
  const bool f16 = gemm_uses_fp16(pool->fmt);
  const uint16_t* rows_in = x_perm;
  float* xe = nullptr;
  const Fp8Rows f8 = L.fp8 ? fp8_rows(W, L.f8) : Fp8Rows{};
  if (launch_clear_word(err, s) != cudaSuccess) return MOE_ERR_CUDA;
  if (L.fp8) {   // the quantised decode GEMMs read e4m3 rows
    if (launch_gather_rows_fp8(x_perm, nullptr, A, A, pool->d_model, f8.xq, f8.xs, f8.xe, sm_count(), s,
                               true) != cudaSuccess)
      return MOE_ERR_CUDA;
  } else if (f16) {   // the quantised prefill GEMMs read scaled fp16 rows
    uint16_t* x16 = (uint16_t*)(W + L.x16);
    xe = (float*)(W + L.xe);
    if (launch_gather_rows_f16(x_perm, nullptr, A, A, pool->d_model, x16, xe, sm_count(), s, true) !=
        cudaSuccess)
      return MOE_ERR_CUDA;
    rows_in = x16;
  }
  st = run_ffn(rows_in, xe, offsets, pool->n_experts, A, pool, nullptr, L.bn, L.ksplit, h, part,
               L.fp8 ? &f8 : nullptr, err, s, true, nullptr, nullptr);
  if (st != MOE_OK) return st;
  return launch_reduce_splits(part, L.ksplit, (size_t)A * pool->d_model, A, pool->d_model, y_perm,
                              s, true) == cudaSuccess
             ? MOE_OK
             : MOE_ERR_CUDA;
}

moe_status moe_combine(const uint16_t* y_perm, const int32_t* row_of_assign, const float* topk_w,
                       const uint16_t* shared_y, int T, int k, int d, uint16_t* out,
                       moe_stream_t stream) {
  const moe::NvtxRange nvtx_range("moe_combine");
  if (!y_perm || !row_of_assign || !topk_w || !out) return MOE_ERR_INVALID_ARG;
  if (T < 1 || k < 1 || d < 128 || d % 128) return MOE_ERR_INVALID_ARG;
  if (k > MAX_K || (long)T * k > MAX_A || d > MAX_DIM) return MOE_ERR_UNSUPPORTED;
  if (!al16(y_perm) || !al16(out) || (shared_y && !al16(shared_y))) return MOE_ERR_INVALID_ARG;
  return launch_combine_bf16(y_perm, row_of_assign, topk_w, shared_y, T, k, d, out,
                             (cudaStream_t)stream) == cudaSuccess
             ? MOE_OK
             : MOE_ERR_CUDA;
}

size_t moe_layer_workspace_bytes(int T, int k, const moe_pool* routed, const moe_pool* shared) {
  if (T < 1 || k < 1 || check_pool(routed, false) != MOE_OK) return 0;
  if (shared && check_pool(shared, true) != MOE_OK) return 0;
  return layer_layout(T, k, routed, shared).total;
}

moe_status moe_layer_forward(const uint16_t* x, const float* logits, int T, int k,
                             const moe_pool* routed, const moe_pool* shared, uint16_t* out,
                             void* ws, size_t ws_bytes, moe_stream_t stream) {
  const moe::NvtxRange nvtx_range("moe_layer_forward");
  return layer_forward_impl(x, logits, T, k, routed, shared, out, ws, ws_bytes,
                            (cudaStream_t)stream, nullptr);
}

moe_status moe_layer_forward_router(const uint16_t* x, const uint16_t* w_router, int T, int k,
                                    const moe_pool* routed, const moe_pool* shared,
                                    float* logits, uint16_t* out, void* ws, size_t ws_bytes,
                                    moe_stream_t stream) {
  const moe::NvtxRange nvtx_range("moe_layer_forward_router");
  moe_status st = check_pool(routed, false);
  if (st != MOE_OK) return st;
  if ((st = check_router_args(x, w_router, T, routed->d_model, routed->n_experts, logits)) != MOE_OK)
    return st;
  // every check of the layer runs before the first launch
  if (!out || !ws || k < 1 || k > routed->n_experts) return MOE_ERR_INVALID_ARG;
  if (ws_bytes < moe_layer_workspace_bytes(T, k, routed, shared)) return MOE_ERR_WORKSPACE;
  if (moe_layer_workspace_bytes(T, k, routed, shared) == 0) return MOE_ERR_INVALID_ARG;
  return layer_forward_impl(x, logits, T, k, routed, shared, out, ws, ws_bytes, (cudaStream_t)stream, nullptr,
                            w_router);
}

moe_status moe_layer_forward_timed(const uint16_t* x, const float* logits, int T, int k,
                                   const moe_pool* routed, const moe_pool* shared, uint16_t* out,
                                   void* ws, size_t ws_bytes, moe_stream_t stream,
                                   void* const* stage_events) {
  const moe::NvtxRange nvtx_range("moe_layer_forward_timed");
  return layer_forward_impl(x, logits, T, k, routed, shared, out, ws, ws_bytes,
                            (cudaStream_t)stream, stage_events);
}

int moe_layer_launch_count(int T, int k, const moe_pool* routed, const moe_pool* shared) {
  if (moe_layer_workspace_bytes(T, k, routed, shared) == 0) return 0;
  // route + permute + gather in one launch for small batches; gate/up, down, combine
  return T <= FUSED_ROUTE_MAX_T ? 4 : 6;
}

int moe_layer_router_launch_count(int T, int k, const moe_pool* routed, const moe_pool* shared) {
  const int n = moe_layer_launch_count(T, k, routed, shared);
  if (n == 0 || T <= FUSED_ROUTE_MAX_T) return n;   // the router runs inside the routing launch
  // its own launch; on the tensor cores it also does the top-k (one launch fewer)
  return router_uses_tensor_cores(T, routed->d_model, routed->n_experts) ? n : n + 1;
}

moe_status moe_debug_gemm_fault(int stop_stage, unsigned long long wait_ns) {
  if (stop_stage < -1) return MOE_ERR_INVALID_ARG;
  g_fault_stop_stage = stop_stage;
  g_fault_wait_ns = wait_ns > 0 ? wait_ns : MOE_WAIT_LIMIT_NS;
  return MOE_OK;
}

moe_status moe_last_device_error(const void* ws, int* code, moe_stream_t stream) {
  if (!ws || !code) return MOE_ERR_INVALID_ARG;
  if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return MOE_ERR_CUDA;
  int v = 0;
  if (cudaMemcpy(&v, ws, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
  *code = v;
  return v ? MOE_ERR_DEVICE : MOE_OK;
}

}  // extern "C"

// ===================================================================== allocation-free variant
// Scratch for moe_layer_forward_noalloc: one file-scope device array per GPU
// that loads the library.  In host code `g_noalloc_scratch` names a host-side
// stand-in, never a device address: the device address is looked up with
// cudaGetSymbolAddress, with the device current, at the first call in each
// CUDA context and passed to the kernels as their workspace.  The cache is
// keyed by the context's unique id (cuCtxGetId, never reused within a process),
// so a context created anew -- after cudaDeviceReset, or another context made
// current -- gets its own lookup instead of a stale address.
namespace {
__device__ __align__(256) uint8_t g_noalloc_scratch[MOE_NOALLOC_SCRATCH_BYTES];

constexpr int NOALLOC_CACHE = 64;
std::mutex g_noalloc_mu;
struct NoallocEntry {
  unsigned long long ctx_id;
  void* ptr;
};
NoallocEntry g_noalloc_cache[NOALLOC_CACHE] = {};
int g_noalloc_next = 0;

PFN_cuCtxGetCurrent_v4000 g_ctx_current = nullptr;
PFN_cuCtxGetId_v12000 g_ctx_id = nullptr;
std::once_flag g_ctx_once;

// Unique id of the calling thread's current CUDA context (the runtime's
// primary context once the runtime is initialised on the current device).
bool current_context_id(unsigned long long* id) {
  std::call_once(g_ctx_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_ctx_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(fn);
    fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_ctx_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(fn);
  });
  if (!g_ctx_current || !g_ctx_id) return false;
  CUcontext ctx = nullptr;
  if (g_ctx_current(&ctx) != CUDA_SUCCESS) return false;
  if (ctx == nullptr) {   // no context bound to this thread yet: the runtime's primary one
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaSetDevice(dev) != cudaSuccess) return false;
    if (g_ctx_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return false;
  }
  return g_ctx_id(ctx, id) == CUDA_SUCCESS;
}

moe_status noalloc_scratch_for_current_context(void** ptr) {
  unsigned long long id = 0;
  if (!current_context_id(&id)) return MOE_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  for (int i = 0; i < NOALLOC_CACHE; ++i)
    if (g_noalloc_cache[i].ptr != nullptr && g_noalloc_cache[i].ctx_id == id) {
      *ptr = g_noalloc_cache[i].ptr;
      return MOE_OK;
    }
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return MOE_ERR_CUDA;
  g_noalloc_cache[g_noalloc_next] = NoallocEntry{id, p};
  g_noalloc_next = (g_noalloc_next + 1) % NOALLOC_CACHE;
  *ptr = p;
  return MOE_OK;
}
}  // namespace

extern "C" moe_status moe_layer_forward_noalloc(const uint16_t* x, const float* logits, int T,
                                                int k, const moe_pool* routed,
                                                const moe_pool* shared, uint16_t* out,
                                                moe_stream_t stream) {
  const moe::NvtxRange nvtx_range("moe_layer_forward_noalloc");
  const size_t need = moe_layer_workspace_bytes(T, k, routed, shared);
  if (need == 0) return MOE_ERR_INVALID_ARG;
  if (need > MOE_NOALLOC_SCRATCH_BYTES) return MOE_ERR_WORKSPACE;
  void* ws = nullptr;
  const moe_status st = noalloc_scratch_for_current_context(&ws);
  if (st != MOE_OK) return st;
  return layer_forward_impl(x, logits, T, k, routed, shared, out, ws, MOE_NOALLOC_SCRATCH_BYTES,
                            (cudaStream_t)stream, nullptr);
}

extern "C" moe_status moe_noalloc_last_device_error(int* code, moe_stream_t stream) {
  if (!code) return MOE_ERR_INVALID_ARG;
  void* ws = nullptr;
  const moe_status st = noalloc_scratch_for_current_context(&ws);
  if (st != MOE_OK) return st;
  return moe_last_device_error(ws, code, stream);
}
