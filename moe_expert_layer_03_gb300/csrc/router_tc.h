// router_tc.h -- the tensor-core router GEMM for long batches of few experts,
// with the top-k gating of its rows fused in (router.cu).
//   logits[t][e] = x[t] . w_router[e]
// tx = x [T][d] and tw = w_router [E][d] as bf16 row maps with {64 x 128} and
// {64 x 16} boxes and the 128-byte swizzle.  err (nullable) gets
// MOE_DEVERR_TIMEOUT if a pipeline wait ran past wait_ns (the tile's logits are
// then NaN); stop_stage >= 0 is the fault-injection hook (-1 off).  With
// idx != nullptr the launch also writes, per token, the k largest logits'
// expert indices in descending order (ties: the lower index; NaN below every
// number) to idx [T][k] and their softmax weights (max-subtracted, summed in
// selection order) to w [T][k] -- the selection and arithmetic of the routing
// kernels, so the same bits; 1 <= k <= E <= 16 (k is ignored without idx).
#pragma once
#include "kernels.cuh"

namespace moe {

// The tensor-core kernel's domain: T * max(E, 8) >= 8192, E <= 16, d % 64 == 0.
bool router_uses_tensor_cores(int T, int d, int E);
cudaError_t launch_router_topk_tc(const CUtensorMap& tx, const CUtensorMap& tw, int T, int d, int E, float* logits,
                                  int k, int32_t* idx, float* w, int* err, int stop_stage, uint64_t wait_ns,
                                  cudaStream_t s, bool pdl = false);

}  // namespace moe
