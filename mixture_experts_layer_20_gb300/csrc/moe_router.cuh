// Per-token top-k with renormalised gates: one warp per token (moe_router.cu
// and the single-launch decode kernel).
//
// The logits arrive as fp32 partial sums over ranges of d, laid out
// [range][T][npad]; the warp adds the ranges in range order (deterministic,
// independent of the other tokens of the batch), adds the router bias,
// selects the k largest logits (an equal logit loses to a lower expert
// index) by k rounds of a warp-wide arg-max, and computes the gates as the
// softmax of the chosen logits, which equals the full softmax renormalised
// over the chosen k ('PagedAttention, speculative decoding, MoE and
// Blackwell', section 2; 'Chapter 9. Distributed inference', section 9.3.4).
// Slots are written in ascending expert id.
#pragma once

#include <climits>
#include <cstdint>

#include "moe_internal.h"

namespace moe {

// A float's bits mapped to an unsigned key with the same order.
__device__ __forceinline__ uint32_t order_key(float v) {
  const uint32_t u = __float_as_uint(v);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// SLOTS: experts per lane (lane, lane + 32, ...; SLOTS * 32 >= E).  COHERENT:
// the partial sums were written by this kernel (see ld_in).
template <int SLOTS, bool COHERENT = false>
__device__ __forceinline__ void topk_warp(const float* partial, int splits, int T,
                                          int npad, int E, int k, const float* __restrict__ bias,
                                          int sel_only, int t, int lane,
                                          int32_t* __restrict__ ids, float* __restrict__ gates) {
  // K ranges summed in range order (a token's logits do not depend on the
  // batch); all loads of a range are issued before its adds
  float L[SLOTS];
#pragma unroll
  for (int i = 0; i < SLOTS; ++i) L[i] = 0.0f;
#pragma unroll 4
  for (int sp = 0; sp < splits; ++sp) {
    const float* row = partial + ((size_t)sp * T + t) * npad;
    float v[SLOTS];
#pragma unroll
    for (int i = 0; i < SLOTS; ++i) v[i] = lane + 32 * i < E ? ld_in<COHERENT>(row + lane + 32 * i) : 0.0f;
#pragma unroll
    for (int i = 0; i < SLOTS; ++i) L[i] += v[i];
  }
  // 64-bit keys: selection-logit order in the high word, lower expert index
  // wins ties.  Each key carries the logit its gate is computed from: the
  // same biased logit, or the unbiased one when the bias only selects.
  unsigned long long key[SLOTS];
  float gl[SLOTS];
#pragma unroll
  for (int i = 0; i < SLOTS; ++i) {
    const int e = lane + 32 * i;
    float l = e < E ? L[i] + (bias ? __ldg(bias + e) : 0.0f) : -INFINITY;
    gl[i] = sel_only ? L[i] : l;
    if (l == 0.0f) l = 0.0f;  // -0 and +0 compare equal: one key for both
    key[i] = e < E ? (static_cast<unsigned long long>(order_key(l)) << 32) |
                         static_cast<uint32_t>(kMaxExperts - 1 - e)
                   : 0ull;
  }
  // each lane sorts its own keys, descending
#pragma unroll
  for (int a = 0; a < SLOTS - 1; ++a)
#pragma unroll
    for (int b = 0; b < SLOTS - 1 - a; ++b)
      if (key[b] < key[b + 1]) {
        const unsigned long long x = key[b]; key[b] = key[b + 1]; key[b + 1] = x;
        const float y = gl[b]; gl[b] = gl[b + 1]; gl[b + 1] = y;
      }

  // k rounds: the warp's largest head wins; its lane pops it.  The 64-bit
  // maximum is taken as two 32-bit warp reductions: the largest high word
  // (the logit's order), then the largest low word among the lanes holding
  // it (the lowest expert index).
  unsigned long long sel[kMaxTopK];
  float sel_g[kMaxTopK];
#pragma unroll
  for (int j = 0; j < kMaxTopK; ++j) {
    sel[j] = 0ull;
    sel_g[j] = 0.0f;
    if (j < k) {
      const uint32_t hi = static_cast<uint32_t>(key[0] >> 32);
      const uint32_t m_hi = __reduce_max_sync(0xffffffffu, hi);
      const uint32_t m_lo =
          __reduce_max_sync(0xffffffffu, hi == m_hi ? static_cast<uint32_t>(key[0]) : 0u);
      const unsigned long long best = (static_cast<unsigned long long>(m_hi) << 32) | m_lo;
      const unsigned owner = __ballot_sync(0xffffffffu, key[0] == best);
      sel[j] = best;
      sel_g[j] = __shfl_sync(0xffffffffu, gl[0], __ffs(owner) - 1);
      if (key[0] == best) {
#pragma unroll
        for (int i = 0; i < SLOTS - 1; ++i) { key[i] = key[i + 1]; gl[i] = gl[i + 1]; }
        key[SLOTS - 1] = 0ull;
      }
    }
  }

  // The selections are the same in every lane.  Gates: softmax of the chosen
  // logits (max subtracted, sum in selection order); lane j < k writes the
  // selection whose expert id is the j-th smallest, so a token's slots hold
  // ascending expert ids.
  float top = sel_g[0];
#pragma unroll
  for (int j = 1; j < kMaxTopK; ++j)
    if (j < k) top = fmaxf(top, sel_g[j]);
  int e_of[kMaxTopK];
  float w[kMaxTopK];
  float sum = 0.0f;
#pragma unroll
  for (int j = 0; j < kMaxTopK; ++j) {
    e_of[j] = j < k ? kMaxExperts - 1 - static_cast<int>(sel[j] & 0xffffffffu) : INT_MAX;
    w[j] = j < k ? expf(sel_g[j] - top) : 0.0f;
    sum += w[j];
  }
  int my_e = INT_MAX;
  float my_w = 0.0f;
#pragma unroll
  for (int j = 0; j < kMaxTopK; ++j)
    if (j == lane) { my_e = e_of[j]; my_w = w[j]; }
  int rank = 0;
#pragma unroll
  for (int j = 0; j < kMaxTopK; ++j) rank += e_of[j] < my_e ? 1 : 0;
  if (lane < k) {
    ids[(size_t)t * k + rank] = my_e;
    gates[(size_t)t * k + rank] = my_w / sum;
  }
}

}  // namespace moe
