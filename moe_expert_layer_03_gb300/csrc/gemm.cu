// gemm.cu -- grouped expert GEMM on the 5th-generation tensor cores (tcgen05),
// A operand in shared memory: bf16 experts, and int4 experts with row chunks of
// more than 32 rows (prefill).  Decode-sized int4 chunks use gemm_group.cu.
//
// "125B MoE on an RTX 3090 at 100+ tok/s": sec. 3.2 -- each expert FFN is a
// two-layer MLP; the tokens of each expert form one contiguous batch and the
// active experts run as one grouped GEMM instead of many small ones; sec. 3.1 --
// per-expert int4 weights with their own scale and zero-point, dequantised to
// fp16 for the tensor cores on the way in rather than in a separate pass.
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
//   warp 1      TMEM owner and MMA issuer: tcgen05.mma kind::f16 with fp32
//               accumulators in TMEM (gate at column 0, up at column bn); bf16
//               operands for bf16 weights, fp16 for int4 weights
//   warps 2..   int4: write fp16((q - z) * s) ((q - z) exact, one rounding of the
//               product) into the swizzled A tile; then, per item, the
//               epilogue: tcgen05.ld, SwiGLU -> h, or fp32 K-split partials.
//
// Every wait is bounded (ptx.cuh); on a timeout the CTA drains its in-flight
// copies and MMAs, frees TMEM and returns with MOE_DEVERR_TIMEOUT set.
#include "gemm_common.cuh"

namespace moe {

using namespace gemm;

namespace {

constexpr int MISC_INTS = 10;   // [0] tmem [1] abort [2] items; consumed raw/a/b [3..5];
                                // issued raw/a/b [6..8]; [9] stays 0

struct Shared {   // views into the dynamic shared-memory carve-out
  uint8_t* a_ring;
  uint8_t* b_ring;
  uint8_t* raw_ring;
  uint64_t *a_full, *a_empty, *b_full, *b_empty, *raw_full, *raw_empty;
  uint64_t *tmem_full, *tmem_empty, *fin;
  int* misc;
  WorkList W;
};

size_t carve_bytes(int nmat, bool int4, int bn, int n_a, int n_b, int n_raw, int n_groups) {
  size_t s = (size_t)n_a * nmat * BF16_TILE_BYTES + (size_t)n_b * bn * 128;
  if (int4) s += (size_t)n_raw * nmat * I4_MAT_BYTES;
  s = align_up(s, 16);
  s += 8 * (size_t)(2 * (n_a + n_b + (int4 ? n_raw : 0)) + 3);
  s += 4 * (MISC_INTS + worklist_ints(n_groups));
  return s;
}

// One 16-byte quad (32 K elements of one weight row) -> 4 chunks of the swizzled
// A row: fp16((q - z) * s).
__device__ __forceinline__ void dequant_quad(uint4 wq, __half2 c2, __half2 s2, uint8_t* arow, int j,
                                             int r) {
  const uint32_t words[4] = {wq.x, wq.y, wq.z, wq.w};
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    uint32_t o[4];
    codes_of_word(words[w], o);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      __half2 b = *reinterpret_cast<const __half2*>(&o[i]);
      b = __hmul2(__hsub2(b, c2), s2);   // (q - z) exact, then one rounding of * s
      o[i] = *reinterpret_cast<uint32_t*>(&b);
    }
    const int chunk = (j * 4 + w) ^ (r & 7);
    *reinterpret_cast<uint4*>(arow + chunk * 16) = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

}  // namespace

template <int FMT, bool GATEUP, int NDQ>
__global__ void __launch_bounds__((2 + NDQ) * 32, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmap_b, const GemmArgs p) {
  constexpr int NMAT = GATEUP ? 2 : 1;
  constexpr bool INT4 = (FMT == MOE_W_INT4_G128);
  static_assert(!INT4 || NDQ == 8, "int4 dequantisation assumes 8 warps (2 per TMEM quadrant)");
  constexpr uint32_t AB_BF16 = INT4 ? 0u : 1u;   // operand type of the MMA
  constexpr uint32_t A_STAGE = NMAT * BF16_TILE_BYTES;
  constexpr uint32_t RAW_STAGE = NMAT * I4_MAT_BYTES;
  constexpr int NDQ_THREADS = NDQ * 32;
  const uint32_t B_STAGE = (uint32_t)p.bn * 128u;

  extern __shared__ uint8_t smem_dyn[];
  const uint32_t pad = (1024u - (smem_u32(smem_dyn) & 1023u)) & 1023u;
  uint8_t* base = smem_dyn + pad;

  Shared S;
  S.a_ring = base;
  S.b_ring = S.a_ring + (size_t)p.n_a * A_STAGE;
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
          if (INT4) {
            if (!(ok = mbar_wait(smem_u32(&S.raw_empty[rr.i]), rr.ph ^ 1u, abort_flag, p.err))) break;
            const uint32_t bar = smem_u32(&S.raw_full[rr.i]);
            mbar_arrive_expect_tx(bar, RAW_STAGE);
            bulk_g2s_hint(smem_u32(S.raw_ring + (size_t)rr.i * RAW_STAGE),
                          sec + ((size_t)it.mt * (p.K / QGROUP) + kg) * RAW_STAGE, RAW_STAGE, bar, pol);
            rr.next();
            ++issued_raw;
          }
          for (int h = 0; h < 2 && ok; ++h) {
            const int kstep = 2 * kg + h;
            if (!INT4) {
              if (!(ok = mbar_wait(smem_u32(&S.a_empty[ra.i]), ra.ph ^ 1u, abort_flag, p.err))) break;
              const uint32_t bar = smem_u32(&S.a_full[ra.i]);
              mbar_arrive_expect_tx(bar, A_STAGE);
              bulk_g2s_hint(smem_u32(S.a_ring + (size_t)ra.i * A_STAGE),
                            sec + ((size_t)it.mt * (p.K / KSTEP) + kstep) * A_STAGE, A_STAGE, bar, pol);
              ra.next();
              ++issued_a;
            }
            if (!(ok = mbar_wait(smem_u32(&S.b_empty[rb.i]), rb.ph ^ 1u, abort_flag, p.err))) break;
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
    // ---------------- MMA issuer.  The whole warp runs the loop and lane 0
    // issues; the next K step's operands are prepared while this step's MMAs
    // issue (they depend only on ring positions).
    Ring ra{0, 0, p.n_a}, rb{0, 0, p.n_b};
    int consumed_a = 0, consumed_b = 0;
    uint32_t it_count = 0;
    bool ok = true;
    struct Ops {
      uint64_t a[NMAT][4];
      uint64_t b[4];
    };
    const uint32_t a_ring0 = smem_u32(S.a_ring), b_ring0 = smem_u32(S.b_ring);
    auto prep = [&](int ai, int bi) -> Ops {
      Ops o;
#pragma unroll
      for (int kk = 0; kk < KSTEP / 16; ++kk) {
        o.b[kk] = sdesc_kmajor_sw128(b_ring0 + (uint32_t)bi * B_STAGE + kk * 32);
#pragma unroll
        for (int m = 0; m < NMAT; ++m)
          o.a[m][kk] = sdesc_kmajor_sw128(a_ring0 + (uint32_t)ai * A_STAGE + m * BF16_TILE_BYTES + kk * 32);
      }
      return o;
    };
    Ops curo = prep(ra.i, rb.i);
    for (int item = blockIdx.x; item < total && ok; item += gridDim.x) {
      Item it;
      if (!decode_item(item, p, S.W, it)) continue;
      int g0, g1;
      kgroups(p, it.ks, g0, g1);
      if (!(ok = mbar_wait(smem_u32(S.tmem_empty), (it_count & 1u) ^ 1u, abort_flag, p.err))) break;
      tc_fence_after();
      const uint32_t idesc = idesc_f16kind_f32(TILE_M, (uint32_t)((it.n_rows + 15) & ~15), AB_BF16);
      for (int kg = g0; kg < g1 && ok; ++kg) {
        for (int h = 0; h < 2; ++h) {
          if (!(ok = mbar_wait(smem_u32(&S.a_full[ra.i]), ra.ph, abort_flag, p.err))) break;
          if (!(ok = mbar_wait(smem_u32(&S.b_full[rb.i]), rb.ph, abort_flag, p.err))) break;
          tc_fence_after();
          const Ops nxt = prep(ra.i + 1 == p.n_a ? 0 : ra.i + 1, rb.i + 1 == p.n_b ? 0 : rb.i + 1);
          const bool fresh = (kg == g0 && h == 0);
          if (lane == 0) {
#pragma unroll
            for (int kk = 0; kk < KSTEP / 16; ++kk)
#pragma unroll
              for (int m = 0; m < NMAT; ++m)
                mma_f16kind(tmem_base + (uint32_t)(m * p.bn), curo.a[m][kk], curo.b[kk], idesc,
                            (fresh && kk == 0) ? 0u : 1u);
            mma_commit(smem_u32(&S.a_empty[ra.i]));
            mma_commit(smem_u32(&S.b_empty[rb.i]));
          }
          __syncwarp();
          curo = nxt;
          ra.next();
          rb.next();
          ++consumed_a;
          ++consumed_b;
        }
      }
      if (!ok) break;
      if (lane == 0) mma_commit(smem_u32(S.tmem_full));
      __syncwarp();
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
    // int4 ownership: gate/up -> matrix m_own of row r (both quads); down -> quad j_own of row r
    const int m_own = GATEUP ? (wr >> 2) : 0;
    const int j_own = GATEUP ? 0 : (wr >> 2);
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
          ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&S.raw_full[rr.i]), rr.ph, abort_flag, p.err));
          if (!ok) break;
          const uint8_t* mat = S.raw_ring + (size_t)rr.i * RAW_STAGE + m_own * I4_MAT_BYTES;
          const uint32_t sz = *reinterpret_cast<const uint32_t*>(mat + I4_PACKED_BYTES + r * 4);
          const __half sh = __ushort_as_half((unsigned short)(sz & 0xFFFFu));
          const __half zh = __ushort_as_half((unsigned short)(sz >> 16));
          const __half2 s2 = __halves2half2(sh, sh);
          const __half2 c2 = __hadd2(__halves2half2(zh, zh), __float2half2_rn(1024.f));
          for (int h = 0; h < 2; ++h) {
            ok = __all_sync(0xffffffffu,
                            mbar_wait(smem_u32(&S.a_empty[ra.i]), ra.ph ^ 1u, abort_flag, p.err));
            if (!ok) break;
            uint8_t* arow = S.a_ring + (size_t)ra.i * A_STAGE + m_own * BF16_TILE_BYTES + r * 128;
#pragma unroll
            for (int jj = 0; jj < (GATEUP ? 2 : 1); ++jj) {
              const int j = GATEUP ? jj : j_own;
              const uint4 wq = *reinterpret_cast<const uint4*>(mat + ((h * 2 + j) * TILE_M + r) * 16);
              dequant_quad(wq, c2, s2, arow, j, r);
            }
            fence_proxy_async_smem();
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
      const uint32_t tl = tmem_base + ((uint32_t)(quad * 32) << 16);
      ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(S.tmem_full), it_count & 1u, abort_flag, p.err));
      if (!ok) break;
      tc_fence_after();
      const int half = wr >> 2;
      const int f = it.mt * TILE_M + r;   // output feature of this thread
      const int n_chunks = (it.n_rows + 15) >> 4;
      for (int c = half; c < n_chunks; c += NHALF) {
        uint32_t acc0[16];
        tmem_ld_16(tl + (uint32_t)(c * 16), acc0);
        if (GATEUP) {
          uint32_t acc1[16];
          tmem_ld_16(tl + (uint32_t)(p.bn + c * 16), acc1);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int n = c * 16 + i;
            if (n < it.n_rows) {
              const float hv = silu_f(__uint_as_float(acc0[i])) * __uint_as_float(acc1[i]);
              const size_t o = (size_t)(it.r0 + n) * p.out_ld + f;
              if (INT4)
                reinterpret_cast<__half*>(p.out)[o] = to_half_sat(hv);
              else
                reinterpret_cast<__nv_bfloat16*>(p.out)[o] = __float2bfloat16_rn(hv);
            }
          }
        } else {
          tmem_ld_wait();
          float* y = reinterpret_cast<float*>(p.out) + (size_t)it.ks * p.out_split_stride;
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int n = c * 16 + i;
            if (n < it.n_rows) y[(size_t)(it.r0 + n) * p.out_ld + f] = __uint_as_float(acc0[i]);
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
        mbar_wait(smem_u32(&fulls[rg][q % ns[rg]]), (uint32_t)((q / ns[rg]) & 1), no_abort, p.err);
    }
  }
  if (warp == 1 && lane == 0) {   // every MMA this CTA issued has finished
    mma_commit(smem_u32(S.fin));
    mbar_wait(smem_u32(S.fin), 0, no_abort, p.err);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, p.tmem_cols);
}

// ------------------------------------------------------------------ host side
GemmPlan plan_gemm_group(bool gateup, int bn, int n_groups, int n_mt);
cudaError_t launch_grouped_gemm_group(bool gateup, const CUtensorMap& tmap_b, GemmArgs args,
                                      const GemmPlan& plan, int grid, cudaStream_t stream, bool pdl);

GemmPlan plan_gemm(int fmt, bool gateup, int bn, int n_groups, int n_mt) {
  const bool int4 = fmt == MOE_W_INT4_G128;
  if (gemm_is_group(fmt, bn)) return plan_gemm_group(gateup, bn, n_groups, n_mt);
  GemmPlan pl{};
  const int nmat = gateup ? 2 : 1;
  pl.group = false;
  pl.pair = false;
  pl.ndq = int4 ? 8 : 4;
  const size_t budget = 227 * 1024 - 1024;   // opt-in maximum minus the alignment pad
  pl.n_b = bn >= 128 ? 3 : (bn >= 64 ? 4 : 8);
  if (int4) {
    pl.n_a = gateup ? (bn >= 128 ? 2 : 3) : (bn >= 128 ? 3 : 4);
    pl.n_raw = 2;
    while (pl.n_raw < 12 &&
           carve_bytes(nmat, true, bn, pl.n_a, pl.n_b, pl.n_raw + 1, n_groups) <= budget)
      ++pl.n_raw;
  } else {
    pl.n_raw = 0;
    pl.n_a = 2;
    while (pl.n_a < 8 && carve_bytes(nmat, false, bn, pl.n_a + 1, pl.n_b, 0, n_groups) <= budget)
      ++pl.n_a;
  }
  pl.smem_bytes = carve_bytes(nmat, int4, bn, pl.n_a, pl.n_b, pl.n_raw, n_groups) + 1024;
  uint32_t cols = 32;
  while (cols < (uint32_t)(nmat * bn)) cols <<= 1;
  pl.tmem_cols = cols;
  return pl;
}

template <int FMT, bool GATEUP, int NDQ>
static cudaError_t launch_one(const CUtensorMap& tmap, const GemmArgs& a, const GemmPlan& pl,
                              int grid, cudaStream_t s, bool pdl) {
  auto kern = grouped_gemm_kernel<FMT, GATEUP, NDQ>;
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
  if (plan.group) return launch_grouped_gemm_group(gateup, tmap_b, args, plan, grid, stream, pdl);
  args.n_a = plan.n_a;
  args.n_b = plan.n_b;
  args.n_raw = plan.n_raw;
  args.tmem_cols = plan.tmem_cols;
  constexpr int I4 = MOE_W_INT4_G128, B16 = MOE_W_BF16;
  if (fmt == I4)
    return gateup ? launch_one<I4, true, 8>(tmap_b, args, plan, grid, stream, pdl)
                  : launch_one<I4, false, 8>(tmap_b, args, plan, grid, stream, pdl);
  return gateup ? launch_one<B16, true, 4>(tmap_b, args, plan, grid, stream, pdl)
                : launch_one<B16, false, 4>(tmap_b, args, plan, grid, stream, pdl);
}

}  // namespace moe
