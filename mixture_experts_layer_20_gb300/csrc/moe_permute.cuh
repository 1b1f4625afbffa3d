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

// One thread: 8 columns of one token, all k slot rows of y loaded before the
// sum (k independent 16-byte loads in flight per thread, two each for fp32
// y), then the fp32 sum in slot order and one bf16 rounding.
constexpr int kCombineThreads = 256;

// 8 columns of y (fp16 or fp32) as floats, from the 16-byte pieces raw[].
template <typename YT>
__device__ __forceinline__ void y8_to_float(const uint4* raw, float (&f)[8]) {
  if constexpr (sizeof(YT) == 4) {
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      f[4 * u + 0] = __uint_as_float(raw[u].x);
      f[4 * u + 1] = __uint_as_float(raw[u].y);
      f[4 * u + 2] = __uint_as_float(raw[u].z);
      f[4 * u + 3] = __uint_as_float(raw[u].w);
    }
  } else {
    const uint32_t w[4] = {raw[0].x, raw[0].y, raw[0].z, raw[0].w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 p = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
      f[2 * i] = p.x;
      f[2 * i + 1] = p.y;
    }
  }
}

// Columns c .. c + 7 of token t (c a multiple of 8, c < d).  YT: the type
// of y and y_shared, __half or float.
template <bool COHERENT = false, typename YT = __half>
__device__ __forceinline__ void combine_cols(const YT* y, const int32_t* slot_pos,
                                             const float* gates, const YT* y_shared, int d,
                                             int k, int rows, int t, int c,
                                             __nv_bfloat16* __restrict__ out, unsigned* status) {
  constexpr int kPieces = sizeof(YT) == 4 ? 2 : 1;  // 16-byte loads per row
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
  // all k rows' loads first
  uint4 v[kMaxTopK][kPieces];
#pragma unroll
  for (int j = 0; j < kMaxTopK; ++j)
    if (j < k)
#pragma unroll
      for (int u = 0; u < kPieces; ++u)
        v[j][u] = ld_in<COHERENT>(reinterpret_cast<const uint4*>(y + (size_t)pos[j] * d + c) + u);
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int j = 0; j < kMaxTopK; ++j) {
    if (j < k) {
      float f[8];
      y8_to_float<YT>(v[j], f);
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] = fmaf(g[j], f[i], acc[i]);
    }
  }
  if (y_shared) {
    uint4 a[kPieces];
#pragma unroll
    for (int u = 0; u < kPieces; ++u)
      a[u] = ld_in<COHERENT>(reinterpret_cast<const uint4*>(y_shared + (size_t)t * d + c) + u);
    float f[8];
    y8_to_float<YT>(a, f);
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] += f[i];
  }
  uint4 o;
  o.x = pack_bf16x2(acc[0], acc[1]);
  o.y = pack_bf16x2(acc[2], acc[3]);
  o.z = pack_bf16x2(acc[4], acc[5]);
  o.w = pack_bf16x2(acc[6], acc[7]);
  *reinterpret_cast<uint4*>(out + (size_t)t * d + c) = o;
}

}  // namespace moe
