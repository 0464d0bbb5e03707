// cache.cu -- expert streaming for pools larger than HBM ("125B MoE on an RTX
// 3090 at 100+ tok/s", sec. 2.1: a hot-expert pool in GPU memory, cold experts
// in system memory brought in on demand; "CPU-GPU co-inference for MoE models",
// sec. 2.2: an expert cache with LRU replacement).
//
// Host-side bookkeeping (which expert sits in which HBM slot, when each was last
// listed) and, per ensure(), one host -> device copy per missing expert image
// followed by one tiny kernel that rewrites the device expert -> slot table
// (the whole table travels as a kernel argument, so nothing host-side has to
// outlive the call).  All on the caller's stream, in order.  A copy is either
// cudaMemcpyAsync (DMA engines) or a kernel whose threads stream the image
// across the C2C link with 16-byte loads and write it to HBM (all SMs pull at
// once; the images must be mapped into the device address space).
//
// Overlapped streaming ("125B MoE on an RTX 3090", sec. 2.2: the next experts
// are prefetched into a double buffer while the current layer computes;
// "CPU-GPU co-inference", sec. 3.1: transfers on their own stream, overlapped
// with compute): prefetch() copies on a copy stream into slots that hold
// neither a listed expert nor one of the committed set (the experts the
// forwards already queued may read); each overwrite first waits on the slot's
// release event.  commit() makes the listed experts the committed set on the
// compute stream: the stream waits for their copies, the slots that leave the
// set get a release event recorded there (complete once every forward queued
// before the commit has finished), and the table is rewritten on the compute
// stream (committed experts -> their slot, all others -> -1).  No host
// synchronisation anywhere.
#include <algorithm>
#include <new>
#include <vector>

#include "kernels.cuh"
#include "nvtx_range.h"

struct moe_expert_cache {
  int n_experts = 0, n_slots = 0;
  size_t slot_bytes = 0;
  const uint8_t* host = nullptr;   // cold tier: pinned host images [E][slot_bytes]
  const uint8_t* host_dev = nullptr;   // the same images' device-side address (SM copies), or null
  uint8_t* dev = nullptr;          // hot tier: HBM slots [n_slots][slot_bytes]
  int32_t* dev_table = nullptr;    // device expert -> slot table [E]
  std::vector<int> slot_expert;    // expert in each slot, -1 = empty
  std::vector<int> expert_slot;    // slot of each expert, -1 = not resident
  std::vector<unsigned long long> last_use;   // per slot: tick of the last ensure listing it
  unsigned long long tick = 0;
  moe_cache_counters counters{};
  // overlapped streaming (prefetch / commit)
  std::vector<char> committed;        // per expert: in the committed set
  std::vector<cudaEvent_t> copied;    // per slot: its last prefetch copy has landed
  std::vector<cudaEvent_t> released;  // per slot: the forwards that may read its previous expert are done
  std::vector<char> has_copied, has_released;
  ~moe_expert_cache() {
    for (cudaEvent_t e : copied)
      if (e) cudaEventDestroy(e);
    for (cudaEvent_t e : released)
      if (e) cudaEventDestroy(e);
  }
};

namespace moe {
namespace {

constexpr int TABLE_MAX = 256;   // = the layer's limit on E
struct Table {
  int32_t v[TABLE_MAX];
};

__global__ void set_table_kernel(Table t, int n, int32_t* __restrict__ dst) {
  for (int i = threadIdx.x; i < n; i += blockDim.x) dst[i] = t.v[i];
}

// dst[0, n16) = src[0, n16) in 16-byte units, 4 loads in flight per thread.
constexpr int CP_THREADS = 256;
__global__ void __launch_bounds__(CP_THREADS)
    image_copy_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst, size_t n16) {
  const size_t stride = (size_t)gridDim.x * CP_THREADS;
  size_t i = (size_t)blockIdx.x * CP_THREADS + threadIdx.x;
  for (; i + 3 * stride < n16; i += 4 * stride) {
    const uint4 a = src[i], b = src[i + stride], c = src[i + 2 * stride], d = src[i + 3 * stride];
    dst[i] = a;
    dst[i + stride] = b;
    dst[i + 2 * stride] = c;
    dst[i + 3 * stride] = d;
  }
  for (; i < n16; i += stride) dst[i] = src[i];
}

// The decisions of one ensure() (or, with keep_committed, one prefetch(),
// which never evicts a committed expert): updates the bookkeeping and lists the
// loads.
moe_status plan_loads(moe_expert_cache* c, const int32_t* experts, int n, int32_t* load_expert,
                      int32_t* load_slot, int* n_loads, bool keep_committed = false) {
  if (!c || (!experts && n > 0) || n < 0) return MOE_ERR_INVALID_ARG;
  if (n > c->n_slots) return MOE_ERR_UNSUPPORTED;
  std::vector<char> listed(c->n_experts, 0);
  for (int i = 0; i < n; ++i) {
    const int e = experts[i];
    if (e < 0 || e >= c->n_experts || listed[e]) return MOE_ERR_INVALID_ARG;
    listed[e] = 1;
  }
  {   // enough slots to take every missing listed expert? (checked before any change)
    int missing = 0, free_slots = 0;
    for (int i = 0; i < n; ++i) missing += c->expert_slot[experts[i]] < 0;
    for (int s = 0; s < c->n_slots; ++s) {
      const int e = c->slot_expert[s];
      free_slots += e < 0 || (!listed[e] && !(keep_committed && c->committed[e]));
    }
    if (missing > free_slots) return MOE_ERR_UNSUPPORTED;
  }
  ++c->tick;
  int nl = 0;
  for (int i = 0; i < n; ++i) {   // hits first, so that no listed expert is evicted below
    const int s = c->expert_slot[experts[i]];
    if (s >= 0) {
      c->last_use[s] = c->tick;
      ++c->counters.hits;
    }
  }
  for (int i = 0; i < n; ++i) {
    const int e = experts[i];
    if (c->expert_slot[e] >= 0) continue;
    int victim = -1;
    for (int s = 0; s < c->n_slots && victim < 0; ++s)
      if (c->slot_expert[s] < 0) victim = s;   // an empty slot
    if (victim < 0)
      for (int s = 0; s < c->n_slots; ++s) {   // least recently used, not listed now
        if (listed[c->slot_expert[s]]) continue;
        if (keep_committed && c->committed[c->slot_expert[s]]) continue;
        if (victim < 0 || c->last_use[s] < c->last_use[victim]) victim = s;
      }
    if (victim < 0) return MOE_ERR_UNSUPPORTED;   // unreachable: checked above
    if (c->slot_expert[victim] >= 0) c->expert_slot[c->slot_expert[victim]] = -1;
    c->slot_expert[victim] = e;
    c->expert_slot[e] = victim;
    c->last_use[victim] = c->tick;
    ++c->counters.misses;
    c->counters.bytes_copied += (long long)c->slot_bytes;
    load_expert[nl] = e;
    load_slot[nl] = victim;
    ++nl;
  }
  *n_loads = nl;
  return MOE_OK;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" {

moe_status moe_cache_create(const moe_pool* routed, const void* host_images, int copy_mode,
                            moe_expert_cache** out) {
  if (!routed || !host_images || !out) return MOE_ERR_INVALID_ARG;
  if (copy_mode < MOE_CACHE_COPY_AUTO || copy_mode > MOE_CACHE_COPY_SM) return MOE_ERR_INVALID_ARG;
  if (routed->slot_bytes % 16) return MOE_ERR_INVALID_ARG;
  if (!routed->pool || !routed->expert_to_slot || routed->n_experts < 1 || routed->n_slots < 1 ||
      routed->slot_bytes == 0)
    return MOE_ERR_INVALID_ARG;
  if (routed->n_experts > TABLE_MAX) return MOE_ERR_UNSUPPORTED;
  moe_expert_cache* c = new (std::nothrow) moe_expert_cache;
  if (!c) return MOE_ERR_UNSUPPORTED;
  c->n_experts = routed->n_experts;
  c->n_slots = routed->n_slots;
  c->slot_bytes = routed->slot_bytes;
  c->host = static_cast<const uint8_t*>(host_images);
  if (copy_mode != MOE_CACHE_COPY_ENGINE) {   // the images' address as the device sees it, if mapped
    void* d = nullptr;
    if (cudaHostGetDevicePointer(&d, const_cast<void*>(host_images), 0) == cudaSuccess && d &&
        reinterpret_cast<uintptr_t>(d) % 16 == 0)
      c->host_dev = static_cast<const uint8_t*>(d);
    else
      (void)cudaGetLastError();   // not mapped: clear the sticky-free error and use the DMA engines
    if (copy_mode == MOE_CACHE_COPY_SM && !c->host_dev) {
      delete c;
      return MOE_ERR_UNSUPPORTED;
    }
  }
  c->dev = static_cast<uint8_t*>(const_cast<void*>(routed->pool));
  c->dev_table = const_cast<int32_t*>(routed->expert_to_slot);
  c->slot_expert.assign(c->n_slots, -1);
  c->expert_slot.assign(c->n_experts, -1);
  c->last_use.assign(c->n_slots, 0);
  c->committed.assign(c->n_experts, 0);
  c->copied.assign(c->n_slots, nullptr);
  c->released.assign(c->n_slots, nullptr);
  c->has_copied.assign(c->n_slots, 0);
  c->has_released.assign(c->n_slots, 0);
  *out = c;
  return MOE_OK;
}

moe_status moe_cache_plan(moe_expert_cache* c, const int32_t* experts, int n, int32_t* load_expert,
                          int32_t* load_slot, int* n_loads) {
  if (!load_expert || !load_slot || !n_loads) return MOE_ERR_INVALID_ARG;
  return plan_loads(c, experts, n, load_expert, load_slot, n_loads);
}

// One expert image host -> slot on stream s (DMA engines, or the SM copy kernel).
static moe_status copy_image(moe_expert_cache* c, int e, int slot, cudaStream_t s) {
  uint8_t* dst = c->dev + (size_t)slot * c->slot_bytes;
  if (c->host_dev) {
    int n_sm = 0, dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return MOE_ERR_CUDA;
    image_copy_kernel<<<4 * n_sm, CP_THREADS, 0, s>>>(
        reinterpret_cast<const uint4*>(c->host_dev + (size_t)e * c->slot_bytes), reinterpret_cast<uint4*>(dst),
        c->slot_bytes / 16);
    return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
  }
  return cudaMemcpyAsync(dst, c->host + (size_t)e * c->slot_bytes, c->slot_bytes, cudaMemcpyHostToDevice, s) ==
                 cudaSuccess
             ? MOE_OK
             : MOE_ERR_CUDA;
}

moe_status moe_cache_ensure(moe_expert_cache* c, const int32_t* experts, int n, moe_stream_t stream) {
  const moe::NvtxRange nvtx_range("moe_cache_ensure");
  if (!c) return MOE_ERR_INVALID_ARG;
  std::vector<int32_t> le(c->n_slots), ls(c->n_slots);
  int nl = 0;
  const moe_status st = plan_loads(c, experts, n, le.data(), ls.data(), &nl);
  if (st != MOE_OK) return st;
  cudaStream_t s = (cudaStream_t)stream;
  for (int i = 0; i < nl; ++i) {   // one copy per expert image, in stream order
    const moe_status cs = copy_image(c, le[i], ls[i], s);
    if (cs != MOE_OK) return cs;
  }
  Table t;
  for (int e = 0; e < c->n_experts; ++e) t.v[e] = c->expert_slot[e];
  set_table_kernel<<<1, 256, 0, s>>>(t, c->n_experts, c->dev_table);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

static bool make_event(cudaEvent_t* e) {
  return *e != nullptr || cudaEventCreateWithFlags(e, cudaEventDisableTiming) == cudaSuccess;
}

moe_status moe_cache_prefetch(moe_expert_cache* c, const int32_t* experts, int n, moe_stream_t copy_stream) {
  const moe::NvtxRange nvtx_range("moe_cache_prefetch");
  if (!c) return MOE_ERR_INVALID_ARG;
  std::vector<int32_t> le(c->n_slots), ls(c->n_slots);
  int nl = 0;
  const moe_status st = plan_loads(c, experts, n, le.data(), ls.data(), &nl, true);
  if (st != MOE_OK) return st;
  cudaStream_t s = (cudaStream_t)copy_stream;
  for (int i = 0; i < nl; ++i) {
    const int slot = ls[i];
    // the forwards that may still read the slot's previous expert come first
    if (c->has_released[slot] && cudaStreamWaitEvent(s, c->released[slot], 0) != cudaSuccess) return MOE_ERR_CUDA;
    const moe_status cs = copy_image(c, le[i], slot, s);
    if (cs != MOE_OK) return cs;
    if (!make_event(&c->copied[slot]) || cudaEventRecord(c->copied[slot], s) != cudaSuccess) return MOE_ERR_CUDA;
    c->has_copied[slot] = 1;
  }
  return MOE_OK;
}

moe_status moe_cache_commit(moe_expert_cache* c, const int32_t* experts, int n, moe_stream_t compute_stream) {
  const moe::NvtxRange nvtx_range("moe_cache_commit");
  if (!c || (!experts && n > 0) || n < 0 || n > c->n_slots) return MOE_ERR_INVALID_ARG;
  std::vector<char> listed(c->n_experts, 0);
  for (int i = 0; i < n; ++i) {
    const int e = experts[i];
    if (e < 0 || e >= c->n_experts || listed[e] || c->expert_slot[e] < 0) return MOE_ERR_INVALID_ARG;
    listed[e] = 1;
  }
  cudaStream_t s = (cudaStream_t)compute_stream;
  ++c->tick;
  for (int i = 0; i < n; ++i) {   // the listed experts' copies land before what follows
    const int slot = c->expert_slot[experts[i]];
    c->last_use[slot] = c->tick;
    if (c->has_copied[slot] && cudaStreamWaitEvent(s, c->copied[slot], 0) != cudaSuccess) return MOE_ERR_CUDA;
  }
  for (int e = 0; e < c->n_experts; ++e) {   // slots leaving the committed set
    if (!c->committed[e] || listed[e]) continue;
    const int slot = c->expert_slot[e];
    if (slot < 0) continue;
    if (!make_event(&c->released[slot]) || cudaEventRecord(c->released[slot], s) != cudaSuccess)
      return MOE_ERR_CUDA;
    c->has_released[slot] = 1;
  }
  Table t;
  for (int e = 0; e < c->n_experts; ++e) {
    c->committed[e] = listed[e];
    t.v[e] = listed[e] ? c->expert_slot[e] : -1;
  }
  set_table_kernel<<<1, 256, 0, s>>>(t, c->n_experts, c->dev_table);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

moe_status moe_cache_stats(const moe_expert_cache* c, moe_cache_counters* out) {
  if (!c || !out) return MOE_ERR_INVALID_ARG;
  *out = c->counters;
  return MOE_OK;
}

void moe_cache_destroy(moe_expert_cache* c) { delete c; }

}  // extern "C"
