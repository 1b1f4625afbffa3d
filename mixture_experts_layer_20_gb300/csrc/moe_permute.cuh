// Device functions shared by the grouping / combine kernels (moe_permute.cu)
// and the single-launch decode kernel: the one-CTA grouping of up to a few
// thousand assignments and the per-thread combine.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "moe_device.cuh"
#include "moe_internal.h"

namespace moe {

// All of count, scan and scatter in one CTA when the T*k assignments fit one
// chunk (decode batches): the same stable positions as the multi-CTA path, two
// launches fewer.  Each warp owns a contiguous range of flat indices and walks
// it 32 at a time in index order (loads issued kPrefetch groups ahead); a
// per-warp, per-expert count then a scan over warps and experts give every
// warp its start position per expert.  (One CTA for much larger batches is
// slower than the three-kernel path: a single SM issues all the scattered
// position stores.)
constexpr int kPrefetch = 8;

// WARPS: the block's warps (blockDim.x = 32 * WARPS).  COHERENT: the ids were
// written by this kernel (see ld_in).  Ends with a block-wide barrier.
template <int WARPS, bool COHERENT = false>
__device__ __forceinline__ void permute_small_block(const int32_t* ids, int n, int E,
                                                    int32_t* __restrict__ counts,
                                                    int32_t* __restrict__ offsets,
                                                    int32_t* __restrict__ perm,
                                                    int32_t* __restrict__ slot_pos,
                                                    unsigned* status) {
  __shared__ int wbase[WARPS][kMaxExperts];
  __shared__ int s_scan[kMaxExperts];
  const int w = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  for (int i = threadIdx.x; i < WARPS * kMaxExperts; i += blockDim.x) (&wbase[0][0])[i] = 0;
  __syncthreads();
  pdl_wait_and_release();
  const int per_warp = ((n + WARPS * 32 - 1) / (WARPS * 32)) * 32;
  const int wbeg = w * per_warp;
  const int wend = min(n, wbeg + per_warp);
  const unsigned lt_mask = (1u << lane) - 1u;
  bool bad = false;
  for (int g0 = wbeg; g0 < wend; g0 += 32 * kPrefetch) {
    int ev[kPrefetch];
#pragma unroll
    for (int b = 0; b < kPrefetch; ++b) {
      const int f = g0 + 32 * b + lane;
      ev[b] = f < wend ? ld_in<COHERENT>(ids + f) : -1;
    }
#pragma unroll
    for (int b = 0; b < kPrefetch; ++b) {
      const int f = g0 + 32 * b + lane;
      const int e = ev[b];
      const bool valid = static_cast<unsigned>(e) < static_cast<unsigned>(E);
      bad |= f < wend && !valid;
      const unsigned peers = __match_any_sync(0xffffffffu, e);
      if (valid && lane == __ffs(peers) - 1) wbase[w][e] += __popc(peers);
      __syncwarp();
    }
  }
  if (bad) atomicOr(status, kStatusDeviceCheck);
  __syncthreads();
  // per-expert totals and the exclusive scan over experts
  for (int e = threadIdx.x; e < kMaxExperts; e += blockDim.x) {
    int total = 0;
    if (e < E)
      for (int ww = 0; ww < WARPS; ++ww) total += wbase[ww][e];
    s_scan[e] = total;
  }
  __syncthreads();
  // inclusive scan over the 256 entries by warp 0 (any block size): lane l
  // takes entries 8 l .. 8 l + 7, then a warp scan of the lanes' sums
  if (w == 0) {
    constexpr int kPer = kMaxExperts / 32;
    int v[kPer];
    int sum = 0;
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      sum += s_scan[lane * kPer + i];
      v[i] = sum;
    }
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += t;
    }
    const int before = incl - sum;
#pragma unroll
    for (int i = 0; i < kPer; ++i) s_scan[lane * kPer + i] = before + v[i];
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int run = e > 0 ? s_scan[e - 1] : 0;
    offsets[e] = run;
    counts[e] = s_scan[e] - run;
    for (int ww = 0; ww < WARPS; ++ww) {
      const int v = wbase[ww][e];
      wbase[ww][e] = run;
      run += v;
    }
  }
  if (threadIdx.x == 0) offsets[E] = s_scan[E - 1];
  __syncthreads();
  for (int g0 = wbeg; g0 < wend; g0 += 32 * kPrefetch) {
    int ev[kPrefetch];
#pragma unroll
    for (int b = 0; b < kPrefetch; ++b) {
      const int f = g0 + 32 * b + lane;
      ev[b] = f < wend ? ld_in<COHERENT>(ids + f) : -1;
    }
#pragma unroll
    for (int b = 0; b < kPrefetch; ++b) {
      const int f = g0 + 32 * b + lane;
      const int e = ev[b];
      const bool valid = static_cast<unsigned>(e) < static_cast<unsigned>(E);
      const unsigned peers = __match_any_sync(0xffffffffu, e);
      if (valid) {
        const int pos = wbase[w][e] + __popc(peers & lt_mask);
        perm[pos] = f;
        slot_pos[f] = pos;
      }
      __syncwarp();
      if (valid && lane == __ffs(peers) - 1) wbase[w][e] += __popc(peers);
      __syncwarp();
    }
  }
  __syncthreads();
}

// One thread: 8 columns of one token, all k slot rows of fp16 y loaded before
// the sum (k independent 16-byte loads in flight per thread), then the fp32
// sum in slot order and one bf16 rounding.
constexpr int kCombineThreads = 256;

// Columns c .. c + 7 of token t (c a multiple of 8, c < d).
template <bool COHERENT = false>
__device__ __forceinline__ void combine_cols(const __half* y, const int32_t* slot_pos,
                                             const float* gates, const __half* y_shared, int d,
                                             int k, int rows, int t, int c,
                                             __nv_bfloat16* __restrict__ out, unsigned* status) {
  int pos[kMaxTopK];
  float g[kMaxTopK];
  bool bad = false;
#pragma unroll
  for (int j = 0; j < kMaxTopK; ++j) {
    pos[j] = 0;
    g[j] = 0.0f;
    if (j < k) {
      const int p = ld_in<COHERENT>(slot_pos + (size_t)t * k + j);
      if (static_cast<unsigned>(p) < static_cast<unsigned>(rows)) {
        pos[j] = p;
        g[j] = ld_in<COHERENT>(gates + (size_t)t * k + j);
      } else {
        bad = true;
      }
    }
  }
  if (bad && c == 0) atomicOr(status, kStatusDeviceCheck);
  // eight fp16 columns per thread: one 16-byte load per expert row
  uint4 v[kMaxTopK];
#pragma unroll
  for (int j = 0; j < kMaxTopK; ++j)
    if (j < k) v[j] = ld_in<COHERENT>(reinterpret_cast<const uint4*>(y + (size_t)pos[j] * d + c));
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int j = 0; j < kMaxTopK; ++j) {
    if (j < k) {
      const uint32_t w[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
        acc[2 * i] = fmaf(g[j], f.x, acc[2 * i]);
        acc[2 * i + 1] = fmaf(g[j], f.y, acc[2 * i + 1]);
      }
    }
  }
  if (y_shared) {
    const uint4 a = ld_in<COHERENT>(reinterpret_cast<const uint4*>(y_shared + (size_t)t * d + c));
    const uint32_t w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
      acc[2 * i] += f.x;
      acc[2 * i + 1] += f.y;
    }
  }
  uint4 o;
  o.x = pack_bf16x2(acc[0], acc[1]);
  o.y = pack_bf16x2(acc[2], acc[3]);
  o.z = pack_bf16x2(acc[4], acc[5]);
  o.w = pack_bf16x2(acc[6], acc[7]);
  *reinterpret_cast<uint4*>(out + (size_t)t * d + c) = o;
}

}  // namespace moe
