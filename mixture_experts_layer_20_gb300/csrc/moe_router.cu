// Router, second half: per-token top-k with renormalised gates.
//
// A lightweight gating network scores every expert for each token and sends
// the token to its top-K experts ('PagedAttention, speculative decoding, MoE
// and Blackwell', section 2; 'Chapter 9. Distributed inference', section
// 9.3.4: the router picks eight experts per token).  The logits come from the
// tensor-core kernel as fp32 partial sums over 512-wide K ranges; here one
// warp per token adds the ranges in range order (deterministic), adds the
// router bias, selects the k largest logits (an equal logit loses to a lower
// expert index) by k rounds of a warp-wide arg-max, and computes the gates
// as the softmax of the chosen logits, which equals the full softmax
// renormalised over the chosen k.  Slots are written in ascending expert id.

#include <climits>

#include "moe_internal.h"

namespace moe {
namespace {

constexpr int kTokensPerCta = 8;  // one warp each

__global__ void __launch_bounds__(kTokensPerCta * 32)
    moe_router_topk_kernel(const float* __restrict__ partial, int splits, int T, int npad, int E,
                           int k, const float* __restrict__ bias, int32_t* __restrict__ ids,
                           float* __restrict__ gates) {
  pdl_wait_and_release();
  const int t = blockIdx.x * kTokensPerCta + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (t >= T) return;  // whole warps only

  // lane owns experts lane, lane+32, ... (at most 8 of them)
  float L[kMaxExperts / 32];
#pragma unroll
  for (int i = 0; i < kMaxExperts / 32; ++i) L[i] = 0.0f;
  // K ranges in order; the loads of one range are independent of each other
#pragma unroll 2
  for (int sp = 0; sp < splits; ++sp) {
    const float* row = partial + ((size_t)sp * T + t) * npad;
#pragma unroll
    for (int i = 0; i < kMaxExperts / 32; ++i)
      if (lane + 32 * i < E) L[i] += __ldg(row + lane + 32 * i);
  }
#pragma unroll
  for (int i = 0; i < kMaxExperts / 32; ++i) {
    const int e = lane + 32 * i;
    L[i] = e < E ? L[i] + (bias ? __ldg(bias + e) : 0.0f) : -INFINITY;
  }

  float sel_v[kMaxTopK];
  int sel_e[kMaxTopK];
  unsigned taken = 0;
#pragma unroll
  for (int j = 0; j < kMaxTopK; ++j) {
    sel_v[j] = -INFINITY;
    sel_e[j] = INT_MAX;
    if (j < k) {
      float bv = -INFINITY;
      int be = INT_MAX;
#pragma unroll
      for (int i = 0; i < kMaxExperts / 32; ++i) {
        const int e = lane + 32 * i;
        const bool free = e < E && !((taken >> i) & 1u);
        if (free && (L[i] > bv || (L[i] == bv && e < be))) { bv = L[i]; be = e; }
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
        const int oe = __shfl_xor_sync(0xffffffffu, be, off);
        if (ov > bv || (ov == bv && oe < be)) { bv = ov; be = oe; }
      }
      sel_v[j] = bv;
      sel_e[j] = be;
#pragma unroll
      for (int i = 0; i < kMaxExperts / 32; ++i)
        if (lane + 32 * i == be) taken |= 1u << i;
    }
  }

  if (lane == 0) {
    float w[kMaxTopK];
    float sum = 0.0f;
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j) {
      w[j] = (j < k) ? expf(sel_v[j] - sel_v[0]) : 0.0f;
      sum += w[j];
    }
    // ascending expert id (unused slots hold INT_MAX and sort last)
#pragma unroll
    for (int a = 0; a < kMaxTopK - 1; ++a) {
#pragma unroll
      for (int b = 0; b < kMaxTopK - 1 - a; ++b) {
        if (sel_e[b] > sel_e[b + 1]) {
          const int te = sel_e[b]; sel_e[b] = sel_e[b + 1]; sel_e[b + 1] = te;
          const float tw = w[b]; w[b] = w[b + 1]; w[b + 1] = tw;
        }
      }
    }
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j) {
      if (j < k) {
        ids[(size_t)t * k + j] = sel_e[j];
        gates[(size_t)t * k + j] = w[j] / sum;
      }
    }
  }
}

}  // namespace

cudaError_t launch_router(cudaStream_t s, const void* x, const void* w_router, const float* bias,
                          int T, int d, int E, int top_k, int32_t* ids, float* gates,
                          float* partial, unsigned* status, unsigned long long timeout_ns) {
  cudaError_t e = launch_router_logits(s, x, w_router, T, d, E, partial, status, timeout_ns);
  if (e != cudaSuccess) return e;
  KernelScope scope(s, "moe_router_topk");
  return launch_kernel(moe_router_topk_kernel, dim3((T + kTokensPerCta - 1) / kTokensPerCta),
                       dim3(kTokensPerCta * 32), 0, s, partial, router_splits(d), T,
                       router_npad(E), E, top_k, bias, ids, gates);
}

}  // namespace moe
