// Grouping of the T*k token-expert assignments by expert, and the combine.
//
// Grouping ('Chapter 9. Distributed inference', section 9.3.4: permute the
// input rows by expert; section 9.4.1: the per-expert row counts m_j sum to
// n k).  The flat assignment index f = t*k + j is cut into chunks of 1024:
//   count   : one CTA per chunk, shared-memory histogram -> chunk_table[c][e]
//   scatter : one CTA per chunk.  Each CTA scans the chunk table itself:
//             expert totals (counts[e]), their exclusive scan (offsets[e]),
//             and its chunk's base per expert = offsets[e] + rows of expert e
//             in earlier chunks.  Each warp owns 256 consecutive assignments;
//             warp histograms (match.any) -> per-warp bases -> each lane's
//             rank among earlier equal ids in its warp.  Small chunks give
//             the grouping of a prefill batch (48k assignments) ~50 CTAs.  Positions are thus
//             offsets[e] + (number of earlier f with the same e): a stable
//             counting sort, deterministic with no global atomics.
//   gather  : x_perm[slot_pos[t k + j]] = x[t], one warp per token: its row
//             read once, written to its k slots, 16-byte copies.
// Up to 4096 assignments, one CTA does count, scan and scatter.
//
// Combine ('Chapter 9. Distributed inference', section 9.3.4, step four;
// 'Hosting Qwen on Blackwell', "MoE Dispatch - Combine": weighted
// accumulation): each thread sums 8 columns of one token's k weighted rows
// (fp16 expert outputs) in fp32 in slot order, then rounds once to bf16.

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "moe_device.cuh"
#include "moe_internal.h"
#include "moe_permute.cuh"

namespace moe {
namespace {

constexpr int kScatterWarps = 16;
constexpr int kPerWarp = kPermuteChunk / kScatterWarps;  // 64

__global__ void __launch_bounds__(512) moe_permute_count_kernel(const int32_t* __restrict__ ids, int n,
                                                            int E, int32_t* __restrict__ table,
                                                            unsigned* status) {
  __shared__ int hist[kMaxExperts];
  pdl_wait_and_release();
  for (int i = threadIdx.x; i < E; i += blockDim.x) hist[i] = 0;
  __syncthreads();
  const int beg = blockIdx.x * kPermuteChunk;
  const int end = min(n, beg + kPermuteChunk);
  bool bad = false;
  for (int f = beg + threadIdx.x; f < end; f += blockDim.x) {
    const int e = __ldg(ids + f);
    if (static_cast<unsigned>(e) < static_cast<unsigned>(E)) atomicAdd(&hist[e], 1);
    else bad = true;
  }
  if (bad) atomicOr(status, kStatusDeviceCheck);
  __syncthreads();
  for (int i = threadIdx.x; i < E; i += blockDim.x) table[(size_t)blockIdx.x * E + i] = hist[i];
}

__global__ void __launch_bounds__(kScatterWarps * 32)
    moe_permute_scatter_kernel(const int32_t* __restrict__ ids, int n, int E, int nchunks,
                           const int32_t* __restrict__ table, int32_t* __restrict__ counts,
                           int32_t* __restrict__ offsets, int32_t* __restrict__ perm,
                           int32_t* __restrict__ slot_pos) {
  __shared__ int wbase[kScatterWarps][kMaxExperts];
  __shared__ int s_scan[kMaxExperts];
  __shared__ int s_before[kMaxExperts];
  pdl_wait_and_release();
  const int w = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  for (int i = threadIdx.x; i < kScatterWarps * kMaxExperts; i += blockDim.x)
    (&wbase[0][0])[i] = 0;
  __syncthreads();
  const int wbeg = blockIdx.x * kPermuteChunk + w * kPerWarp;
  const unsigned lt_mask = (1u << lane) - 1u;

  // per-warp histogram
  for (int r = 0; r < kPerWarp / 32; ++r) {
    const int f = wbeg + r * 32 + lane;
    const int e = f < n ? __ldg(ids + f) : -1;
    const bool valid = static_cast<unsigned>(e) < static_cast<unsigned>(E);
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    if (valid && lane == __ffs(peers) - 1) wbase[w][e] += __popc(peers);
    __syncwarp();
  }
  // Every CTA scans the per-chunk counts itself: expert totals, the exclusive
  // scan over experts (the offsets; CTA 0 stores them and the counts) and this
  // chunk's base = offset + the expert's rows in earlier chunks.
  for (int e = threadIdx.x; e < kMaxExperts; e += blockDim.x) {
    int total = 0, before = 0;
    if (e < E)
      for (int c = 0; c < nchunks; ++c) {
        const int v = __ldg(table + (size_t)c * E + e);
        if (c < static_cast<int>(blockIdx.x)) before += v;
        total += v;
      }
    s_scan[e] = total;
    s_before[e] = before;
  }
  __syncthreads();
  for (int o = 1; o < kMaxExperts; o <<= 1) {
    int v = 0;
    if (threadIdx.x < kMaxExperts && threadIdx.x >= o) v = s_scan[threadIdx.x - o];
    __syncthreads();
    if (threadIdx.x < kMaxExperts) s_scan[threadIdx.x] += v;
    __syncthreads();
  }
  if (blockIdx.x == 0) {
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
      const int excl = e > 0 ? s_scan[e - 1] : 0;
      offsets[e] = excl;
      counts[e] = s_scan[e] - excl;
    }
    if (threadIdx.x == 0) offsets[E] = s_scan[E - 1];
  }
  // per-expert exclusive scan across the warps, on top of the chunk's base
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int run = (e > 0 ? s_scan[e - 1] : 0) + s_before[e];
    for (int ww = 0; ww < kScatterWarps; ++ww) {
      const int v = wbase[ww][e];
      wbase[ww][e] = run;
      run += v;
    }
  }
  __syncthreads();
  // positions
  for (int r = 0; r < kPerWarp / 32; ++r) {
    const int f = wbeg + r * 32 + lane;
    const int e = f < n ? __ldg(ids + f) : -1;
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

template <int WARPS>
__global__ void __launch_bounds__(WARPS * 32)
    moe_permute_small_kernel(const int32_t* __restrict__ ids, int n, int E,
                             int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
                             int32_t* __restrict__ perm, int32_t* __restrict__ slot_pos,
                             unsigned* status) {
  permute_small_block<WARPS>(ids, n, E, counts, offsets, perm, slot_pos, status);
}

// One warp per token: its row of x is loaded once (each lane issues all of its
// 16-byte loads of the row, up to kGatherVec, before any store) and stored to
// each of its k slots x_perm[slot_pos[t k + j]].  Reading x once in token order,
// instead of once per slot in slot order, keeps the reads sequential and
// independent of L2 holding x (the DeepSeek-like layer's x is about L2-sized).
// The stores are streaming (evict first): x_perm exceeds L2, and measured on
// the prefill layer the layer was faster although gate_up, which reads x_perm
// next, finds less of it in L2.
constexpr int kGatherVec = 16;  // uint4 per lane and pass: 32 * 16 * 8 = 4096 bf16

__global__ void __launch_bounds__(256) moe_permute_gather_kernel(
    const int32_t* __restrict__ slot_pos, const uint4* __restrict__ x, int T, int k, int n,
    int vec_per_row, uint4* __restrict__ x_perm, unsigned* status) {
  pdl_wait_and_release();
  const int lane = threadIdx.x & 31;
  const int warps = (gridDim.x * blockDim.x) >> 5;
  for (int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; t < T; t += warps) {
    int pos[kMaxTopK];
    bool bad = false;
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j) {
      pos[j] = j < k ? __ldg(slot_pos + (size_t)t * k + j) : -1;
      if (j < k && static_cast<unsigned>(pos[j]) >= static_cast<unsigned>(n)) {
        bad = true;
        pos[j] = -1;  // a bad slot position: that copy is skipped
      }
    }
    if (bad && lane == 0) atomicOr(status, kStatusDeviceCheck);
    const uint4* src = x + (size_t)t * vec_per_row;
    for (int v0 = 0; v0 < vec_per_row; v0 += 32 * kGatherVec) {
      uint4 r[kGatherVec];
#pragma unroll
      for (int i = 0; i < kGatherVec; ++i) {
        const int v = v0 + lane + 32 * i;
        if (v < vec_per_row) r[i] = __ldg(src + v);
      }
#pragma unroll
      for (int j = 0; j < kMaxTopK; ++j) {
        if (pos[j] < 0) continue;
        uint4* dst = x_perm + (size_t)pos[j] * vec_per_row;
#pragma unroll
        for (int i = 0; i < kGatherVec; ++i) {
          const int v = v0 + lane + 32 * i;
          if (v < vec_per_row) __stcs(dst + v, r[i]);
        }
      }
    }
  }
}

// One thread per (token, 8-column group), numbered token-major, so a warp's
// threads take consecutive column groups and every thread has work whatever d.
// YT: the type of y, __half or float.
template <typename YT>
__global__ void __launch_bounds__(kCombineThreads) moe_combine_kernel(
    const YT* __restrict__ y, const int32_t* __restrict__ slot_pos,
    const float* __restrict__ gates, const YT* __restrict__ y_shared, int d, int k, int rows,
    long long groups, __nv_bfloat16* __restrict__ out, unsigned* status) {
  pdl_wait_and_release();
  const long long i = static_cast<long long>(blockIdx.x) * kCombineThreads + threadIdx.x;
  if (i >= groups) return;
  const int cpr = d / 8;  // column groups per token
  const int t = static_cast<int>(i / cpr);
  const int c = static_cast<int>(i - static_cast<long long>(t) * cpr) * 8;
  combine_cols<false, YT>(y, slot_pos, gates, y_shared, d, k, rows, t, c, out, status);
}

}  // namespace

cudaError_t launch_permute(cudaStream_t s, const int32_t* ids, const void* x, int T, int d, int E,
                           int top_k, int32_t* counts, int32_t* offsets, int32_t* perm,
                           int32_t* slot_pos, void* x_perm, int32_t* chunk_table,
                           unsigned* status) {
  const int n = T * top_k;
  const int nchunks = (n + kPermuteChunk - 1) / kPermuteChunk;
  cudaError_t e = cudaSuccess;
  if (n <= kPermuteSmallMax) {
    KernelScope scope(s, "moe_permute_small");
    e = launch_kernel(moe_permute_small_kernel<kScatterWarps>, dim3(1), dim3(kScatterWarps * 32),
                      0, s, ids, n, E, counts, offsets, perm, slot_pos, status);
  } else {
    {
      KernelScope scope(s, "moe_permute_count");
      e = launch_kernel(moe_permute_count_kernel, dim3(nchunks), dim3(512), 0, s, ids, n, E,
                        chunk_table, status);
    }
    if (e == cudaSuccess) {
      KernelScope scope(s, "moe_permute_scatter");
      e = launch_kernel(moe_permute_scatter_kernel, dim3(nchunks), dim3(kScatterWarps * 32), 0, s,
                        ids, n, E, nchunks, chunk_table, counts, offsets, perm, slot_pos);
    }
  }
  if (e != cudaSuccess || x == nullptr) return e;
  const int warps_per_cta = 8;
  const int grid = std::min((T + warps_per_cta - 1) / warps_per_cta, device_sm_count() * 8);
  KernelScope scope(s, "moe_permute_gather");
  return launch_kernel(moe_permute_gather_kernel, dim3(grid), dim3(warps_per_cta * 32), 0, s,
                       slot_pos, static_cast<const uint4*>(x), T, top_k, n, d / 8,
                       static_cast<uint4*>(x_perm), status);
}

cudaError_t launch_combine(cudaStream_t s, const void* y, const int32_t* slot_pos,
                           const float* gates, const void* y_shared, int T, int d, int top_k,
                           void* out, unsigned* status, bool y_fp32) {
  const long long groups = static_cast<long long>(T) * (d / 8);
  const long long grid = (groups + kCombineThreads - 1) / kCombineThreads;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidValue;
  KernelScope scope(s, "moe_combine");
  if (y_fp32)
    return launch_kernel(moe_combine_kernel<float>, dim3(static_cast<unsigned>(grid)),
                         dim3(kCombineThreads), 0, s, static_cast<const float*>(y), slot_pos,
                         gates, static_cast<const float*>(y_shared), d, top_k, T * top_k,
                         groups, static_cast<__nv_bfloat16*>(out), status);
  return launch_kernel(moe_combine_kernel<__half>, dim3(static_cast<unsigned>(grid)),
                       dim3(kCombineThreads), 0, s, static_cast<const __half*>(y), slot_pos,
                       gates, static_cast<const __half*>(y_shared), d, top_k, T * top_k, groups,
                       static_cast<__nv_bfloat16*>(out), status);
}

}  // namespace moe
