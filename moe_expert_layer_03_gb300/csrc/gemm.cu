// gemm.cu -- grouped expert GEMM on the 5th-generation tensor cores (tcgen05).
//
// "125B MoE on an RTX 3090 at 100+ tok/s": sec. 3.2 -- each expert FFN is a
// two-layer MLP; the tokens of each expert form one contiguous batch and the
// active experts run as one grouped GEMM instead of many small ones; sec. 3.1 --
// per-expert int4 weights with their own scale and zero-point, dequantised on
// the way in rather than in a separate pass over memory.
//
// One persistent CTA per SM walks a list of work items
//   (expert group g, 128-row weight tile mt, K split ks, row chunk nc)
// built on the device from the group offsets, so experts without rows cost
// nothing.  The MMA is "swap-AB": weight rows are the M = 128 side and the
// expert's token rows the N side (16..256, a multiple of 16 set per item), so a
// decode batch of a few tokens per expert still fills the tensor core's M.
//
//   warp 0      producer: 1-D bulk copies of the prepacked weight blocks
//               (int4 nibbles + scales, or pre-swizzled bf16 tiles) and 2-D TMA
//               loads of the 64-wide K slices of the token rows (128-byte swizzle)
//   warp 1      TMEM owner and MMA issuer: tcgen05.mma kind::f16, bf16 x bf16 ->
//               fp32 accumulators in TMEM (gate at column 0, up at column bn)
//   warps 2..   int4: unpack nibbles to bf16 (magic-exponent trick), apply
//               (q - z) * s, write the swizzled A tile; then, for every item,
//               the epilogue: tcgen05.ld of the accumulators, SwiGLU
//               (gate/up) or fp32 partial sums (down), global stores.
//
// Every wait is bounded (ptx.cuh); on a timeout the CTA drains its in-flight
// copies and MMAs, frees TMEM and returns with MOE_DEVERR_TIMEOUT set.
#include "kernels.cuh"
#include "ptx.cuh"

namespace moe {

namespace {

struct Item {
  int g, mt, ks, r0, n_rows;
  const uint8_t* slot;
};

struct Shared {   // views into the dynamic shared-memory carve-out
  uint8_t* a_ring;
  uint8_t* b_ring;
  uint8_t* raw_ring;
  uint64_t* a_full;
  uint64_t* a_empty;
  uint64_t* b_full;
  uint64_t* b_empty;
  uint64_t* raw_full;
  uint64_t* raw_empty;
  uint64_t* tmem_full;
  uint64_t* tmem_empty;
  uint64_t* fin;
  int* misc;     // [0] tmem base [1] abort [2] items; consumed raw/a/b [3..5]; issued raw/a/b [6..8]
  int* prefix;   // [n_groups + 1] first item of each group
  int* nch;      // [n_groups] row chunks per group
  int* goff;     // [n_groups + 1] group row offsets
};

constexpr int MISC_INTS = 10;

__host__ __device__ inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

__host__ __device__ inline size_t carve_bytes(int nmat, bool int4, int bn, int n_a, int n_b,
                                              int n_raw, int n_groups) {
  size_t s = (size_t)n_a * nmat * BF16_TILE_BYTES + (size_t)n_b * bn * 128;
  if (int4) s += (size_t)n_raw * nmat * I4_MAT_BYTES;
  s = align_up(s, 16);
  s += 8 * (size_t)(2 * (n_a + n_b + (int4 ? n_raw : 0)) + 3);
  s += 4 * (size_t)(MISC_INTS + 3 * (n_groups + 1));
  return s;
}

__device__ __forceinline__ bool decode_item(int item, const GemmArgs& p, const Shared& S, Item& it) {
  int lo = 0, hi = p.n_groups - 1;
  while (lo < hi) {   // last group whose first item is <= item (empty groups are skipped)
    const int mid = (lo + hi + 1) >> 1;
    if (S.prefix[mid] <= item) lo = mid; else hi = mid - 1;
  }
  const int g = lo;
  const int local = item - S.prefix[g];
  const int nch = S.nch[g];
  const int nc = local % nch;
  const int t2 = local / nch;
  it.g = g;
  it.ks = t2 % p.ksplit;
  it.mt = t2 / p.ksplit;
  const int cnt = S.goff[g + 1] - S.goff[g];
  const int rpc = (((cnt + nch - 1) / nch) + 15) & ~15;   // rows per chunk, multiple of 16
  it.r0 = S.goff[g] + nc * rpc;
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

// int4 -> bf16 for one 16-byte quad (32 K elements of one row): 4 words, each
// 8 nibbles -> 4 bf16x2 = one 16-byte chunk of the swizzled A row.
__device__ __forceinline__ void dequant_quad(uint4 wq, __nv_bfloat162 c2, __nv_bfloat162 s2,
                                             uint8_t* arow, int j, int r) {
  const uint32_t words[4] = {wq.x, wq.y, wq.z, wq.w};
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t v = lop3_and_or(words[w] >> (4 * i), 0x000F000Fu, 0x43004300u);   // 128 + q
      __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&v);
      b = __hmul2(__hsub2(b, c2), s2);   // (q - z) exact, then one rounding of * s
      o[i] = *reinterpret_cast<uint32_t*>(&b);
    }
    const int chunk = (j * 4 + w) ^ (r & 7);
    *reinterpret_cast<uint4*>(arow + chunk * 16) = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

__device__ __forceinline__ float silu_f(float g) { return g / (1.0f + __expf(-g)); }

}  // namespace

template <int FMT, bool GATEUP, int NDQ>
__global__ void __launch_bounds__((2 + NDQ) * 32, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmap_b, const GemmArgs p) {
  constexpr int NMAT = GATEUP ? 2 : 1;
  constexpr bool INT4 = (FMT == MOE_W_INT4_G128);
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
  uint8_t* after_rings = S.raw_ring + (INT4 ? (size_t)p.n_raw * RAW_STAGE : 0);
  uint64_t* bars = reinterpret_cast<uint64_t*>(
      base + align_up((size_t)(after_rings - base), 16));
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
  S.prefix = S.misc + MISC_INTS;
  S.nch = S.prefix + (p.n_groups + 1);
  S.goff = S.nch + (p.n_groups + 1);

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
    // misc[0] is written by tcgen05.alloc and misc[2] by warp 2, both before the barrier
    for (int i = 1; i < MISC_INTS; ++i)
      if (i != 2) S.misc[i] = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) prefetch_tensormap(&tmap_b);
  if (warp == 1) {
    tmem_alloc(smem_u32(&S.misc[0]), p.tmem_cols);
    tmem_relinquish();
  }
  if (warp == 2) {   // work list: items per group = chunks * tiles * splits, exclusive prefix
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
        S.goff[g] = lo;
        if (g == p.n_groups - 1) S.goff[g + 1] = hi;
      }
      int incl = items;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += o;
      }
      if (g < p.n_groups) {
        S.prefix[g] = running + incl - items;
        S.nch[g] = nch;
      }
      running += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (bad) atomicOr(p.err, MOE_DEVERR_OFFSETS);
    if (lane == 0) {
      S.prefix[p.n_groups] = running;
      S.misc[2] = running;
    }
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
        if (!decode_item(item, p, S, it)) continue;
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
      // publish issue counts for the drain after the role loops
      S.misc[6] = issued_raw;
      S.misc[7] = issued_a;
      S.misc[8] = issued_b;
    }
  } else if (warp == 1) {
    if (lane == 0) {   // ---------------- MMA issuer
      Ring ra{0, 0, p.n_a}, rb{0, 0, p.n_b};
      int consumed_a = 0, consumed_b = 0;
      uint32_t it_count = 0;
      bool ok = true;
      for (int item = blockIdx.x; item < total && ok; item += gridDim.x) {
        Item it;
        if (!decode_item(item, p, S, it)) continue;
        int g0, g1;
        kgroups(p, it.ks, g0, g1);
        if (!(ok = mbar_wait(smem_u32(S.tmem_empty), (it_count & 1u) ^ 1u, abort_flag, p.err))) break;
        tc_fence_after();
        const uint32_t n_mma = (uint32_t)((it.n_rows + 15) & ~15);
        const uint32_t idesc = idesc_bf16_f32(TILE_M, n_mma);
        const int nk = 2 * (g1 - g0);
        for (int s = 0; s < nk; ++s) {
          if (!(ok = mbar_wait(smem_u32(&S.a_full[ra.i]), ra.ph, abort_flag, p.err))) break;
          if (!(ok = mbar_wait(smem_u32(&S.b_full[rb.i]), rb.ph, abort_flag, p.err))) break;
          tc_fence_after();
          const uint32_t a0 = smem_u32(S.a_ring + (size_t)ra.i * A_STAGE);
          const uint32_t b0 = smem_u32(S.b_ring + (size_t)rb.i * B_STAGE);
#pragma unroll
          for (int kk = 0; kk < KSTEP / 16; ++kk) {
            const uint64_t bdesc = sdesc_kmajor_sw128(b0 + kk * 32);
#pragma unroll
            for (int m = 0; m < NMAT; ++m)
              mma_bf16(tmem_base + (uint32_t)(m * p.bn),
                       sdesc_kmajor_sw128(a0 + m * BF16_TILE_BYTES + kk * 32), bdesc, idesc,
                       (s | kk) != 0 ? 1u : 0u);
          }
          mma_commit(smem_u32(&S.a_empty[ra.i]));
          mma_commit(smem_u32(&S.b_empty[rb.i]));
          ra.next();
          rb.next();
          ++consumed_a;
          ++consumed_b;
        }
        if (!ok) break;
        mma_commit(smem_u32(S.tmem_full));
        ++it_count;
      }
      S.misc[4] = consumed_a;
      S.misc[5] = consumed_b;
    }
  } else {   // ---------------- dequant + epilogue warps
    const int dq = threadIdx.x - 64;                 // 0 .. NDQ*32-1
    const int quad = warp & 3;                       // TMEM lane quadrant this warp may access
    const int half = (warp - 2) >> 2;                // column interleave among warps of one quadrant
    constexpr int NHALF = NDQ / 4;
    Ring ra{0, 0, p.n_a}, rr{0, 0, p.n_raw};
    int consumed_raw = 0;
    uint32_t it_count = 0;
    bool ok = true;
    for (int item = blockIdx.x; item < total && ok; item += gridDim.x) {
      Item it;
      if (!decode_item(item, p, S, it)) continue;
      int g0, g1;
      kgroups(p, it.ks, g0, g1);
      if (INT4) {
        for (int kg = g0; kg < g1 && ok; ++kg) {
          ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&S.raw_full[rr.i]), rr.ph, abort_flag, p.err));
          if (!ok) break;
          const uint8_t* raw = S.raw_ring + (size_t)rr.i * RAW_STAGE;
          for (int h = 0; h < 2; ++h) {
            ok = __all_sync(0xffffffffu,
                            mbar_wait(smem_u32(&S.a_empty[ra.i]), ra.ph ^ 1u, abort_flag, p.err));
            if (!ok) break;
            uint8_t* a = S.a_ring + (size_t)ra.i * A_STAGE;
            for (int u = dq; u < NMAT * 2 * TILE_M; u += NDQ_THREADS) {
              const int m = u / (2 * TILE_M), j = (u / TILE_M) & 1, r = u & (TILE_M - 1);
              const uint8_t* mat = raw + m * I4_MAT_BYTES;
              const uint4 wq = *reinterpret_cast<const uint4*>(mat + ((h * 2 + j) * TILE_M + r) * 16);
              const uint32_t sz = *reinterpret_cast<const uint32_t*>(mat + I4_PACKED_BYTES + r * 4);
              const float s = __half2float(__ushort_as_half((unsigned short)(sz & 0xFFFFu)));
              const float z = __half2float(__ushort_as_half((unsigned short)(sz >> 16)));
              const __nv_bfloat162 s2 = __float2bfloat162_rn(s);
              const __nv_bfloat162 c2 = __float2bfloat162_rn(128.0f + z);
              dequant_quad(wq, c2, s2, a + m * BF16_TILE_BYTES + r * 128, j, r);
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
      // ---- epilogue
      ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(S.tmem_full), it_count & 1u, abort_flag, p.err));
      if (!ok) break;
      tc_fence_after();
      const uint32_t tl = tmem_base + ((uint32_t)(quad * 32) << 16);
      const int f = it.mt * TILE_M + quad * 32 + lane;   // output feature of this thread
      const int n_chunks = (it.n_rows + 15) >> 4;
      for (int c = half; c < n_chunks; c += NHALF) {
        uint32_t acc0[16];
        tmem_ld_16(tl + (uint32_t)(c * 16), acc0);
        if (GATEUP) {
          uint32_t acc1[16];
          tmem_ld_16(tl + (uint32_t)(p.bn + c * 16), acc1);
          tmem_ld_wait();
          __nv_bfloat16* h = reinterpret_cast<__nv_bfloat16*>(p.out);
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int n = c * 16 + i;
            if (n < it.n_rows) {
              const float gv = __uint_as_float(acc0[i]), uv = __uint_as_float(acc1[i]);
              h[(size_t)(it.r0 + n) * p.out_ld + f] = __float2bfloat16_rn(silu_f(gv) * uv);
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
    if (dq == 0) S.misc[3] = consumed_raw;
  }

  // ------------------------------------------------------------ teardown
  __syncthreads();
  // misc[9] stays 0: the drain waits are bounded by time only, never cut short
  volatile int* no_abort = &S.misc[9];
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
GemmPlan plan_gemm(int fmt, bool gateup, int bn, int n_groups) {
  GemmPlan pl{};
  const bool int4 = fmt == MOE_W_INT4_G128;
  const int nmat = gateup ? 2 : 1;
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
                              int grid, cudaStream_t s) {
  auto kern = grouped_gemm_kernel<FMT, GATEUP, NDQ>;
  static bool attr_set = false;   // per instantiation; the maximum is requested once
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  kern<<<grid, (2 + NDQ) * 32, pl.smem_bytes, s>>>(tmap, a);
  return cudaGetLastError();
}

cudaError_t launch_grouped_gemm(int fmt, bool gateup, const CUtensorMap& tmap_b, GemmArgs args,
                                const GemmPlan& plan, int grid, cudaStream_t stream) {
  args.n_a = plan.n_a;
  args.n_b = plan.n_b;
  args.n_raw = plan.n_raw;
  args.tmem_cols = plan.tmem_cols;
  if (fmt == MOE_W_INT4_G128) {
    return gateup ? launch_one<MOE_W_INT4_G128, true, 8>(tmap_b, args, plan, grid, stream)
                  : launch_one<MOE_W_INT4_G128, false, 8>(tmap_b, args, plan, grid, stream);
  }
  return gateup ? launch_one<MOE_W_BF16, true, 4>(tmap_b, args, plan, grid, stream)
                : launch_one<MOE_W_BF16, false, 4>(tmap_b, args, plan, grid, stream);
}

}  // namespace moe
