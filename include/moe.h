/*
 * moe.h -- C ABI of the GB300 (sm_103a) MoE FFN layer forward.
 *
 * The layer is the inference forward of one Mixture-of-Experts FFN layer:
 *
 *   router logits -> top-k gating -> regroup tokens by expert -> grouped SwiGLU
 *   expert FFN over the active experts -> weighted combine back to token order
 *
 * Sources (page title, section):
 *   [Mira]   "Mira: adaptive caching and predictive expert staging for MoE
 *            inference" (gsyq.cn/news/338825): sec. 4.2 (Top-K gating).
 *   [CoInf]  "CPU-GPU co-inference for MoE models" (maplevalley.com.cn/news/2111104):
 *            sec. 2.1 (router and expert cache on the GPU), sec. 2.2 (expert
 *            slots, S = floor(memory / expert size)), sec. 5.1 (group quantisation).
 *   [Strata] "125B MoE on an RTX 3090 at 100+ tok/s: a full-stack inference
 *            optimisation log" (bjdmk.com.cn/news/6009460): sec. 1.1 (top-2 /
 *            top-1 routing), sec. 2.1 (shared expert always resident; hot-expert
 *            pool), sec. 3.1 (per-expert int4 scale and zero-point, dequantise
 *            without a separate pass), sec. 3.2 (expert FFN is a two-layer MLP;
 *            one grouped GEMM over the active experts), sec. 4.2 (tokens
 *            regrouped by expert id, contiguous per expert).
 *
 * Conventions for every entry point
 *   - Pointers are DEVICE pointers owned by the caller unless stated otherwise.
 *     The library never allocates, frees or synchronises (except
 *     moe_last_device_error, which reads one word back synchronously).
 *   - bf16 and fp16 tensors are passed as their 16-bit patterns (uint16_t).
 *     Matrices are row-major; "[rows][cols]" lists the slow index first.
 *   - All work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *     stream) in call order.  Nothing is launched when a host-side check fails.
 *   - Every pointer must be 16-byte aligned; workspaces and pools 256-byte aligned.
 *   - Host-side argument errors return MOE_ERR_INVALID_ARG / MOE_ERR_UNSUPPORTED /
 *     MOE_ERR_WORKSPACE; a failed launch returns MOE_ERR_CUDA.  Device-side
 *     checks (an expert index outside [0,E), a slot outside [0,n_slots), a
 *     pipeline wait that exceeds its time limit) never trap: they OR a code into
 *     the workspace error word, skip the affected work and return; read it with
 *     moe_last_device_error().  No C++ exception crosses this ABI.
 *   - Logits must be finite.
 *
 * Limits: 1 <= E <= 256, 1 <= k <= min(E, 16), T*k <= 1<<20, d_model and d_ff
 * multiples of 128 and <= 32768.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* moe_stream_t;   /* identical to cudaStream_t */

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,   /* null pointer, bad size, misaligned pointer, k outside 1..E */
  MOE_ERR_UNSUPPORTED = 2,   /* outside the documented limits */
  MOE_ERR_WORKSPACE = 3,     /* workspace smaller than the *_workspace_bytes() answer */
  MOE_ERR_CUDA = 4,          /* a CUDA launch or attribute call failed */
  MOE_ERR_DEVICE = 5         /* moe_last_device_error found a device-side error code */
} moe_status;

/* Device-side error codes ORed into the workspace error word. */
enum {
  MOE_DEVERR_TIMEOUT = 1,       /* a pipeline wait ran past its limit (~2 s) */
  MOE_DEVERR_EXPERT_RANGE = 2,  /* topk_idx outside [0, E) */
  MOE_DEVERR_SLOT_RANGE = 4,    /* expert_to_slot[e] outside [0, n_slots) */
  MOE_DEVERR_OFFSETS = 8        /* offsets not non-decreasing or beyond the row count */
};

/* Expert weight formats. */
typedef enum {
  MOE_W_BF16 = 0,       /* bf16 weights */
  MOE_W_INT4_G128 = 1,  /* int4, asymmetric, one fp16 scale + one fp16 zero (integer 0..15)
                           per row and group of 128 input elements: w = (q - z) * s
                           ([Strata] sec. 3.1; [CoInf] sec. 5.1) */
  MOE_W_FP8_G128 = 2    /* 8 bits: OCP fp8 E4M3 codes, one fp16 scale per row and group of
                           128 input elements: w = e4m3(q) * s ([CoInf] sec. 5.1: 8-bit
                           group quantisation of the expert layers only) */
} moe_wfmt;

/* The expert pool: n_slots equally sized slots in one device allocation, and
 * the table that maps an expert id to its slot ([CoInf] sec. 2.2 slots;
 * [Strata] sec. 2.1 resident expert pool).  Described by, not owned by, the
 * library.  Slot s starts at pool + s * slot_bytes and holds one expert in the
 * library's prepacked layout (see moe_prepack_expert). */
typedef struct {
  int n_experts;                  /* E: entries of expert_to_slot */
  int n_slots;                    /* slots in the pool */
  int d_model, d_ff;              /* d and F of every expert in this pool */
  int fmt;                        /* moe_wfmt */
  const void* pool;               /* device, 256-byte aligned */
  size_t slot_bytes;              /* >= moe_slot_bytes(fmt, d_model, d_ff), multiple of 256 */
  const int32_t* expert_to_slot;  /* device int32 [n_experts], values in [0, n_slots) */
} moe_pool;

/* Canonical (interchange) weights of one expert, device pointers.
 * bf16:  w[0] = W_gate [F][d], w[1] = W_up [F][d], w[2] = W_down [d][F]  (bf16)
 * int4:  w[m] = packed bytes [rows][K/2]: byte j holds element 2j in its low
 *        nibble and 2j+1 in its high nibble; scale[m], zero[m] = fp16
 *        [rows][K/128]; (rows, K) = (F, d) for gate/up and (d, F) for down.
 * fp8:   w[m] = E4M3 code bytes [rows][K]; scale[m] = fp16 [rows][K/128];
 *        zero[m] unused. */
typedef struct {
  const void* w[3];
  const uint16_t* scale[3];   /* int4 and fp8 */
  const uint16_t* zero[3];    /* int4 only */
} moe_expert_src;

/* ---------------------------------------------------------------- information */

const char* moe_status_str(int status);

/* Bytes one expert occupies in the prepacked slot layout (no padding):
 * bf16: 6*d*F;  int4: 1.5*d*F + 3*F*(d/128)*4;  fp8: 3*d*F + 3*F*(d/128)*2.
 * 0 for unsupported shapes. */
size_t moe_slot_bytes(int fmt, int d_model, int d_ff);

/* ---------------------------------------------------------------- weight preparation
 * Not on the hot path.  Rewrites one expert from the canonical layout into the
 * slot layout the grouped GEMM streams: per (matrix, 128-row tile, K step) one
 * contiguous block, bf16 tiles pre-swizzled for the tensor core, int4 nibbles
 * reordered for in-register unpacking with the group's scale and zero beside
 * them.  slot_dst must hold moe_slot_bytes() bytes. */
moe_status moe_prepack_expert(int fmt, int d_model, int d_ff, const moe_expert_src* src,
                              void* slot_dst, moe_stream_t stream);

/* ---------------------------------------------------------------- hot path */

/* Router logits ([CoInf] sec. 2.1: the router runs on the GPU; sec. 5.1: the
 * router network keeps full precision):
 *   logits[t][e] = sum_i x[t][i] * w_router[e][i]
 * x bf16 [T][d] and w_router bf16 [E][d], both row-major with the input dim
 * contiguous; logits fp32 [T][E].  Products and sums in fp32 (the order is
 * fixed, so results are reproducible run to run).  Long batches
 * (T * max(E, 8) >= 8192) with E <= 16 and d % 64 == 0 run on the tensor cores
 * (one cluster of 8 K-slice CTAs per 128 tokens, the slices' fp32 partial sums
 * added in a fixed order); the rest on CUDA cores.  Requires d % 8 == 0, 1 <= E <= 256, 16-byte
 * aligned pointers; otherwise MOE_ERR_INVALID_ARG / MOE_ERR_UNSUPPORTED and
 * nothing is launched.  One kernel launch.  Every wait of the tensor-core
 * kernel is bounded: if one runs out, that tile's logits are NaN. */
moe_status moe_router_logits(const uint16_t* x, const uint16_t* w_router, int T, int d, int E,
                             float* logits, moe_stream_t stream);

/* Top-k gating ([Mira] sec. 4.2; [Strata] sec. 1.1).
 * logits: fp32 [T][E].  For each token the k largest logits (the lower expert
 * index first among equal logits), in descending order -> topk_idx int32 [T][k];
 * topk_w fp32 [T][k] = softmax over the k selected logits (same as softmax over
 * all E renormalised over the k). */
moe_status moe_route_topk(const float* logits, int T, int E, int k, int32_t* topk_idx,
                          float* topk_w, moe_stream_t stream);

/* Regroup tokens by expert ([Strata] sec. 4.2): histogram, exclusive scan and a
 * stable scatter of the A = T*k assignments a = t*k + j.
 *   counts int32 [E]: assignments per expert;  offsets int32 [E+1], offsets[E] = A;
 *   row_of_assign int32 [A]: row of assignment a = offsets[e] + number of earlier
 *     assignments with the same expert e = topk_idx[a];
 *   token_of_row int32 [A]: token of each row (ascending within an expert);
 *   x_perm bf16 [A][d]: x_perm[row_of_assign[a]] = x[a / k]  (x is bf16 [T][d]).
 * ws: moe_permute_workspace_bytes() bytes (holds the error word). */
size_t moe_permute_workspace_bytes(void);
moe_status moe_permute(const int32_t* topk_idx, const uint16_t* x, int T, int k, int E, int d,
                       int32_t* counts, int32_t* offsets, int32_t* row_of_assign,
                       int32_t* token_of_row, uint16_t* x_perm, void* ws, size_t ws_bytes,
                       moe_stream_t stream);

/* Grouped SwiGLU expert FFN over the active experts ([Strata] sec. 3.2, 3.1).
 * Rows [offsets[e], offsets[e+1]) of x_perm (bf16 [A][d]) belong to expert e and
 * use the weights in slot expert_to_slot[e] of `pool`:
 *   h = bf16(silu(x W_gate^T) * (x W_up^T))  [rows][F]     (fp32 accumulation)
 *   y_perm = bf16(h W_down^T)                 bf16 [A][d]
 * int4 weights are dequantised inside the GEMM main loop; experts with no rows
 * are never read.  ws: moe_grouped_ffn_workspace_bytes(A, pool) bytes. */
size_t moe_grouped_ffn_workspace_bytes(int A, const moe_pool* pool);
moe_status moe_grouped_ffn(const uint16_t* x_perm, const int32_t* offsets, int A,
                           const moe_pool* pool, uint16_t* y_perm, void* ws, size_t ws_bytes,
                           moe_stream_t stream);

/* Weighted combine back to token order:
 *   out[t] = bf16( sum_{j<k} topk_w[t][j] * y_perm[row_of_assign[t*k+j]]  + shared_y[t] )
 * summed in fp32 in the order j = 0..k-1, shared_y (bf16 [T][d]) last; shared_y
 * may be NULL.  out bf16 [T][d]. */
moe_status moe_combine(const uint16_t* y_perm, const int32_t* row_of_assign, const float* topk_w,
                       const uint16_t* shared_y, int T, int k, int d, uint16_t* out,
                       moe_stream_t stream);

/* The whole layer: route -> permute -> grouped FFN -> combine, with an optional
 * always-on shared expert ([Strata] sec. 2.1) of weight 1.0 added to every token.
 * x bf16 [T][d]; logits fp32 [T][E] (E = routed->n_experts); out bf16 [T][d].
 * shared: NULL, or a pool view with n_experts == 1 and the same d_model, d_ff and
 * fmt as `routed` (it may point into the same allocation).
 * ws: moe_layer_workspace_bytes(T, k, routed, shared) bytes; its first word is
 * the device error word, cleared at the start of every call. */
size_t moe_layer_workspace_bytes(int T, int k, const moe_pool* routed, const moe_pool* shared);
moe_status moe_layer_forward(const uint16_t* x, const float* logits, int T, int k,
                             const moe_pool* routed, const moe_pool* shared, uint16_t* out,
                             void* ws, size_t ws_bytes, moe_stream_t stream);

/* The whole layer from the token rows and the router weight: the logits of
 * moe_router_logits (the same bits) into `logits` (caller-owned fp32 [T][E],
 * written; E = routed->n_experts), then moe_layer_forward on those logits.
 * w_router bf16 [E][d_model].  Same workspace, checks and results as
 * moe_layer_forward.  For T <= 64 the router GEMM runs inside the routing
 * launch ("CPU-GPU co-inference for MoE models", sec. 2.1: the router in front
 * of the gating on the GPU): a cooperative launch of at most one CTA per SM,
 * so the call launches as many kernels as moe_layer_forward; it fails with
 * MOE_ERR_CUDA where a cooperative launch is refused (fewer resident CTAs than
 * its grid).  Larger batches run the router GEMM as its own launch first; on
 * the tensor cores (T * max(E, 8) >= 8192, E <= 16, d_model % 64 == 0) that
 * launch also does the top-k gating of its rows, with the routing kernel's
 * selection and arithmetic (the same indices and weights), in place of the
 * routing launch. */
moe_status moe_layer_forward_router(const uint16_t* x, const uint16_t* w_router, int T, int k,
                                    const moe_pool* routed, const moe_pool* shared,
                                    float* logits, uint16_t* out, void* ws, size_t ws_bytes,
                                    moe_stream_t stream);

/* Stage boundaries of moe_layer_forward, for timing with CUDA events. */
enum {
  MOE_STAGE_ROUTE = 0,    /* top-k gating */
  MOE_STAGE_PERMUTE = 1,  /* histogram, scan, stable scatter of the indices */
  MOE_STAGE_GATHER = 2,   /* x rows copied into expert order */
  MOE_STAGE_GATE_UP = 3,  /* grouped gate/up GEMM + SwiGLU */
  MOE_STAGE_DOWN = 4,     /* grouped down GEMM (K-split partial sums) */
  MOE_STAGE_COMBINE = 5,  /* weighted combine (+ shared expert) */
  MOE_N_STAGES = 6
};

/* Same as moe_layer_forward; if stage_events is non-NULL it must point to
 * MOE_N_STAGES + 1 cudaEvent_t handles, recorded on `stream` before each stage
 * and after the last one. */
moe_status moe_layer_forward_timed(const uint16_t* x, const float* logits, int T, int k,
                                   const moe_pool* routed, const moe_pool* shared, uint16_t* out,
                                   void* ws, size_t ws_bytes, moe_stream_t stream,
                                   void* const* stage_events);

/* Allocation-free variant of moe_layer_forward, for callers that cannot
 * allocate device memory at call time and cannot hand the library a
 * workspace: code running inside stream capture (an allocation there is not
 * part of the graph and may synchronise), hosts that own every device
 * allocation through their own pool and forbid libraries from calling
 * cudaMalloc, and real-time loops where an allocation's latency is not
 * allowed.  The pages have no counterpart to this entry point.
 *
 * Same arguments and results as moe_layer_forward, without ws / ws_bytes: the
 * scratch is a file-scope device array of MOE_NOALLOC_SCRATCH_BYTES that every
 * GPU loading the library holds until the process exits.  A call whose
 * moe_layer_workspace_bytes(T, k, routed, shared) exceeds that size returns
 * MOE_ERR_WORKSPACE and launches nothing (decode-sized batches fit; large
 * prefill chunks do not).  No cudaMalloc, cudaFree or allocating library call
 * is made.  The first call in a CUDA context (normally: on a device) looks up
 * that device's address of the array (cudaGetSymbolAddress, with the device
 * current); make that first call before any stream capture.  A new context
 * (after cudaDeviceReset, or another context made current) is detected by its
 * unique id and gets a fresh lookup on its first call.  Device-side errors of
 * these calls are read with moe_noalloc_last_device_error.  All calls share the one array and it keeps the
 * last call's contents (its error word is cleared at the start of each call):
 * calls that overlap on the GPU -- on different streams, or from different
 * host threads -- race on it and must be serialised by the caller. */
#define MOE_NOALLOC_SCRATCH_BYTES ((size_t)16 << 20)
moe_status moe_layer_forward_noalloc(const uint16_t* x, const float* logits, int T, int k,
                                     const moe_pool* routed, const moe_pool* shared,
                                     uint16_t* out, moe_stream_t stream);

/* Device-side error word of the allocation-free scratch on the current device
 * (the caller of moe_layer_forward_noalloc has no workspace pointer to pass to
 * moe_last_device_error).  Synchronises `stream`, then copies the word: *code
 * = the OR of the MOE_DEVERR_* bits raised by the most recent
 * moe_layer_forward_noalloc call on this device (each call clears it first);
 * returns MOE_OK if it is 0, MOE_ERR_DEVICE otherwise, MOE_ERR_CUDA on a
 * failed synchronisation or copy.  The pages have no counterpart to this entry
 * point.  Allocates nothing. */
moe_status moe_noalloc_last_device_error(int* code, moe_stream_t stream);

/* ---------------------------------------------------------------- expert streaming
 * Pools larger than HBM ([Strata] sec. 2.1: a resident hot-expert pool, cold
 * experts in system memory loaded on demand; [CoInf] sec. 2.2: an expert cache
 * with LRU replacement).  On a Grace-Blackwell node the cold tier is pinned host
 * memory reached over NVLink-C2C; the hot tier is the HBM pool of a moe_pool.
 *
 * moe_cache_create: `routed` describes the hot tier (n_experts = E experts,
 * n_slots slots of slot_bytes; its expert_to_slot table is rewritten by the
 * cache); host_images = pinned host memory holding all E experts' prepacked
 * slot images (expert e at host_images + e * slot_bytes, as moe_prepack_expert
 * writes them).  Both are owned by the caller and must outlive the cache.  The
 * cache starts empty; it allocates only its host-side bookkeeping.  copy_mode:
 * MOE_CACHE_COPY_ENGINE copies each image with cudaMemcpyAsync (the DMA
 * engines); MOE_CACHE_COPY_SM with a kernel whose threads read the host images
 * over the C2C link and write the slot (needs host_images to be mapped into the
 * device address space, checked with cudaHostGetDevicePointer; otherwise
 * MOE_ERR_UNSUPPORTED); MOE_CACHE_COPY_AUTO picks the kernel when the images
 * are mapped, else the DMA engines.
 *
 * moe_cache_ensure: makes the n listed experts (host int32, distinct, in
 * [0, E), n <= n_slots) resident before the work that follows on `stream`.
 * A listed expert already in a slot is a hit; each other one takes an empty
 * slot, else the least recently used slot holding no listed expert (LRU), and
 * its image is copied host -> device on `stream`.  Then the device
 * expert_to_slot table is rewritten on `stream`: resident experts map to their
 * slot, all others to -1, so routing a token to an expert that was not made
 * resident flags MOE_DEVERR_SLOT_RANGE instead of reading another expert's
 * weights.  Every copy is ordered on `stream` after the work already queued
 * there, so a slot is never overwritten while an earlier forward on the same
 * stream reads it.
 *
 * moe_cache_plan: the same decisions and bookkeeping as moe_cache_ensure
 * without any CUDA call; writes the experts to load and their slots
 * (load_expert / load_slot, n_slots entries each) and *n_loads.
 *
 * Overlapped streaming ([Strata] sec. 2.2: the next layer's experts are
 * prefetched into a double buffer while the current one computes; [CoInf]
 * sec. 3.1: transfers on their own stream, overlapped with compute):
 * moe_cache_prefetch makes the n listed experts resident on `copy_stream`
 * without touching the table: each missing one takes an empty slot, else the
 * least recently used slot that holds neither a listed expert nor one of the
 * committed set; before overwriting a slot the copy stream waits for that
 * slot's release event (below).  MOE_ERR_UNSUPPORTED if listed + committed
 * experts exceed the slots.  moe_cache_commit makes the n listed experts (all
 * resident, e.g. prefetched) the committed set on `compute_stream`: the stream
 * waits for their copies, each slot whose expert leaves the committed set gets
 * a release event recorded on `compute_stream` (complete once the work queued
 * there before the commit -- the forwards that may read it -- has finished),
 * and the table is rewritten on `compute_stream`: committed experts -> their
 * slot, all others -> -1.  Forwards queued after the commit read the new set.
 * A decode loop per step i: prefetch(A[i+1], copy); forward(i); commit(A[i+1],
 * compute).  No host synchronisation; use either ensure or prefetch/commit
 * with one cache.  The events are created by the cache on first use and
 * destroyed with it.
 *
 * moe_cache_stats: hits, misses (= expert images copied), bytes copied. */
typedef struct moe_expert_cache moe_expert_cache;
enum { MOE_CACHE_COPY_AUTO = 0, MOE_CACHE_COPY_ENGINE = 1, MOE_CACHE_COPY_SM = 2 };
typedef struct {
  long long hits, misses, bytes_copied;
} moe_cache_counters;
moe_status moe_cache_create(const moe_pool* routed, const void* host_images, int copy_mode,
                            moe_expert_cache** out);
moe_status moe_cache_ensure(moe_expert_cache* cache, const int32_t* experts, int n, moe_stream_t stream);
moe_status moe_cache_plan(moe_expert_cache* cache, const int32_t* experts, int n, int32_t* load_expert,
                          int32_t* load_slot, int* n_loads);
moe_status moe_cache_prefetch(moe_expert_cache* cache, const int32_t* experts, int n, moe_stream_t copy_stream);
moe_status moe_cache_commit(moe_expert_cache* cache, const int32_t* experts, int n, moe_stream_t compute_stream);
moe_status moe_cache_stats(const moe_expert_cache* cache, moe_cache_counters* out);
void moe_cache_destroy(moe_expert_cache* cache);

/* Kernel launches one moe_layer_forward enqueues for these arguments (0 on error). */
int moe_layer_launch_count(int T, int k, const moe_pool* routed, const moe_pool* shared);
/* The same for moe_layer_forward_router: T <= 64, as moe_layer_forward (the
 * router runs inside the routing launch); longer batches one more (the router
 * launch), except on the tensor-core router, whose launch also does the top-k
 * gating (T * max(E, 8) >= 8192, E <= 16). */
int moe_layer_router_launch_count(int T, int k, const moe_pool* routed, const moe_pool* shared);

/* Test hook for the failure paths (not for production use; the pages have no
 * counterpart).  Every wait in the grouped-GEMM kernels is bounded: past its
 * limit the CTA sets MOE_DEVERR_TIMEOUT in the error word, drains the copies
 * it issued, waits for its MMAs, frees its tensor memory and returns, so the
 * context stays usable.  This call makes that path run on purpose: forwards
 * enqueued afterwards leave the gate/up GEMM's pipeline stage number
 * stop_stage of each CTA (counting from 0; -1: none) unissued, so the
 * consumers' waits for it run out, and every GEMM wait give up after wait_ns
 * (0: the default, 2 s).  The tensor-core router kernel (moe_router_logits on
 * long batches) takes the same setting.  Host-side setting, read when a
 * forward is enqueued; not thread-safe.  moe_debug_gemm_fault(-1, 0) restores
 * the defaults.  MOE_ERR_INVALID_ARG for stop_stage < -1. */
moe_status moe_debug_gemm_fault(int stop_stage, unsigned long long wait_ns);

/* Synchronously reads the device error word of a workspace written by
 * moe_permute, moe_grouped_ffn or moe_layer_forward (waits for `stream`).
 * *code = the ORed MOE_DEVERR_* bits; returns MOE_ERR_DEVICE if any bit is set. */
moe_status moe_last_device_error(const void* ws, int* code, moe_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif
