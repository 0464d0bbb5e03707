// router_tc.h -- the tensor-core router GEMM with the top-k gating of its rows
// fused in (router.cu).  logits[t][e] = x[t] . w_router[e] as
// launch_router_logits_tc; with idx != nullptr it also writes, per token, the
// k largest logits' expert indices in descending order (ties: the lower
// index; NaN below every number) to idx [T][k] and their softmax weights
// (max-subtracted, summed in selection order) to w [T][k] -- the selection
// and arithmetic of the routing kernels, so the same bits.  1 <= k <= E <= 16.
#pragma once
#include "kernels.cuh"

namespace moe {

cudaError_t launch_router_topk_tc(const CUtensorMap& tx, const CUtensorMap& tw, int T, int d, int E, float* logits,
                                  int k, int32_t* idx, float* w, int* err, int stop_stage, uint64_t wait_ns,
                                  cudaStream_t s, bool pdl = false);

}  // namespace moe
