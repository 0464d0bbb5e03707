// nvtx_range.h -- an NVTX range around one C-ABI call (the call's name on a
// profiler's timeline; the NVTX v3 header-only API, a no-op unless a tool is
// attached).
#pragma once
#include <nvtx3/nvToolsExt.h>

namespace moe {

struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

}  // namespace moe
