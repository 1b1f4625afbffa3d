// Router, second half: per-token top-k with renormalised gates.
//
// A lightweight gating network scores every expert for each token and sends
// the token to its top-K experts ('PagedAttention, speculative decoding, MoE
// and Blackwell', section 2; 'Chapter 9. Distributed inference', section
// 9.3.4: the router picks eight experts per token).  The logits come from the
// tensor-core kernel as fp32 partial sums over 512-wide K ranges (for large
// batches already added, in the same order, by that kernel: one range); here
// one warp per token adds the ranges in range order (deterministic), adds the
// router bias, selects the k largest logits (an equal logit loses to a lower
// expert index) by k rounds of a warp-wide arg-max, and computes the gates
// as the softmax of the chosen logits, which equals the full softmax
// renormalised over the chosen k.  Slots are written in ascending expert id.

#include <climits>

#include "moe_internal.h"
#include "moe_router.cuh"

namespace moe {
namespace {

constexpr int kTokensPerCta = 8;  // one warp each

// Five CTAs per SM (at most 51 registers a thread): a 6000-token batch is
// one wave of warps.
__global__ void __launch_bounds__(kTokensPerCta * 32, 5)
    moe_router_topk_kernel(const float* __restrict__ partial, int splits, int T, int npad, int E,
                           int k, const float* __restrict__ bias, int sel_only,
                           int32_t* __restrict__ ids, float* __restrict__ gates) {
  pdl_wait_and_release();
  const int t = blockIdx.x * kTokensPerCta + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (t >= T) return;  // whole warps only
  if (E <= 64) topk_warp<2>(partial, splits, T, npad, E, k, bias, sel_only, t, lane, ids, gates);
  else if (E <= 128) topk_warp<4>(partial, splits, T, npad, E, k, bias, sel_only, t, lane, ids, gates);
  else topk_warp<8>(partial, splits, T, npad, E, k, bias, sel_only, t, lane, ids, gates);
}

}  // namespace

cudaError_t launch_router(cudaStream_t s, const void* x, const void* w_router, const float* bias,
                          int bias_selection_only, int T, int d, int E, int top_k, int32_t* ids,
                          float* gates, float* partial, unsigned* status,
                          unsigned long long timeout_ns) {
  cudaError_t e = launch_router_logits(s, x, w_router, T, d, E, partial, status, timeout_ns);
  if (e != cudaSuccess) return e;
  KernelScope scope(s, "moe_router_topk");
  return launch_kernel(moe_router_topk_kernel, dim3((T + kTokensPerCta - 1) / kTokensPerCta),
                       dim3(kTokensPerCta * 32), 0, s, partial, router_ranges_written(T, d, E), T,
                       router_npad(E), E, top_k, bias, bias_selection_only ? 1 : 0, ids, gates);
}

}  // namespace moe
