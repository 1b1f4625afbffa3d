// The whole MoE layer in one kernel launch, for decode-sized batches.
//
// 'Hosting Qwen on Blackwell', "Expert parallelism": for decode the dispatch,
// the expert GEMMs and the combine run as one kernel, while prefill splits
// them.  Here one persistent cooperative launch of CTA pairs (2-CTA clusters,
// every CTA resident at once, one per SM) runs the layer's steps as phases
// separated by grid-wide barriers:
//
//   1. router logits: fp32 partial sums of x W_r^T over 128-wide ranges of d,
//      warp-level tensor-core MMAs (16 experts x 8 tokens per MMA tile);
//   2. top-k and gates: one warp per token adds the ranges in range order
//      (the same warp code as the standalone router);
//   3. grouping: counts, offsets and the stable permutation, by one CTA;
//   4. gate_up with the SwiGLU epilogue and 5. down: the bf16 expert GEMM body
//      of the grouped kernels (2-SM tcgen05 MMAs, weights on M, TMA rings,
//      accumulators in tensor memory), gate_up gathering its token rows from
//      x through the permutation;
//   6. combine: fp32 sum of each token's k rows in slot order, one bf16
//      rounding.
//
// The pair's 512 tensor-memory columns are allocated once for both GEMM
// phases.  A grid-wide barrier is an arrival counter and a generation word in
// the workspace's status region; thread 0 of each CTA arrives and waits for
// the generation to move, bounded by %globaltimer.  A wait that runs out
// records MOE_ERR_TIMEOUT and the CTA carries on (the results are then not to
// be used): every CTA runs every phase, so the cluster barriers inside the
// GEMM phases always meet their peer, and since every wait is bounded the
// kernel always ends.  The last CTA to leave resets the arrival counter for
// the next launch.  Data one phase writes and a later phase reads with
// ordinary loads goes through L2 (ld_in with COHERENT = true); h, which the
// down phase's TMA reads, is ordered by proxy fences on both sides.

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>
#include <mutex>

#include "moe_device.cuh"
#include "moe_expert_gemm.cuh"
#include "moe_internal.h"
#include "moe_permute.cuh"
#include "moe_router.cuh"
#include "moe_smallm.cuh"  // mma_16816, word_of

namespace moe {
namespace {

constexpr int kRouterRange = 128;         // the router's partial sums: 128-wide ranges of d
constexpr int kFuWarps = kThreads / 32;   // warps per CTA (the GEMM body's six roles)

struct FusedParams {
  CUtensorMap mw_gu;              // W_gate_up, interleaved 5-D map
  CUtensorMap mw_dn;              // W_down as [E d, I]
  TokenMapSet tx_gu;              // gate_up token rows: one-row boxes over x (gathered)
  TokenMapSet tx_dn;              // down token rows: boxes over h
  Params gu, dn;                  // the two GEMM phases
  const __nv_bfloat16* x;         // [T, d]
  const __nv_bfloat16* w_router;  // [E, d]
  const float* bias;              // [E] or null
  int sel_only;
  int T, d, E, k;
  float* partial;                 // [d / 128][T][npad]
  int npad;
  int32_t *ids, *counts, *offsets, *perm, *slot_pos;
  float* gates;
  const __half* y;                // [T k, d]
  __nv_bfloat16* out;             // [T, d]
  unsigned* status;
  unsigned* bar_count;            // arrivals at the current barrier
  unsigned* bar_gen;              // barriers completed (only grows)
  unsigned* exit_count;           // CTAs that have left the kernel
  unsigned long long timeout_ns;
};

__device__ __forceinline__ unsigned ld_acquire_gpu(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Grid-wide barrier (every thread of every CTA).  A wait that runs out sets
// MOE_ERR_TIMEOUT; the CTA then goes on (see the file comment).
__device__ __forceinline__ void grid_sync(const FusedParams& p) {
  __syncthreads();
  if (threadIdx.x == 0) {
    const unsigned gen = ld_acquire_gpu(p.bar_gen);
    __threadfence();  // this CTA's writes before its arrival
    if (atomicAdd(p.bar_count, 1u) == gridDim.x - 1) {
      atomicExch(p.bar_count, 0u);
      __threadfence();
      atomicAdd(p.bar_gen, 1u);
    } else {
      const unsigned long long t0 = globaltimer_ns();
      while (ld_acquire_gpu(p.bar_gen) == gen) {
        if (globaltimer_ns() - t0 > p.timeout_ns) {
          atomicOr(p.status, kStatusTimeout);
          break;
        }
      }
    }
    __threadfence();
  }
  __syncthreads();
}

// Phase 1: partial[r][t][e] = sum over the 128 values of range r of
// x[t] . W_r[e].  Warp task = (16 experts, one range, 16 tokens); lane (g, t)
// holds experts e0 + g and e0 + g + 8 and the reduction permutation of the
// small-M GEMMs (16-byte units of 8 values at 8 (4 i + t)).
__device__ __forceinline__ void router_partials(const FusedParams& p) {
  const int lane = threadIdx.x & 31;
  const int g = lane >> 2, tig = lane & 3;
  const int groups = (p.E + 15) / 16;
  const int ranges = p.d / kRouterRange;
  const int passes = (p.T + 15) / 16;
  const int total = groups * ranges * passes;
  const int W = gridDim.x * kFuWarps;
  for (int tau = blockIdx.x * kFuWarps + (threadIdx.x >> 5); tau < total; tau += W) {
    const int rg = tau % groups;
    const int rest = tau / groups;
    const int r = rest % ranges;
    const int pass = rest / ranges;
    const int k0 = r * kRouterRange;
    uint4 a[2][4], b[2][4];
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
      const int e = rg * 16 + g + 8 * rr;
#pragma unroll
      for (int i = 0; i < 4; ++i)
        a[rr][i] = e < p.E ? __ldg(reinterpret_cast<const uint4*>(
                                 p.w_router + static_cast<size_t>(e) * p.d + k0 + 8 * (4 * i + tig)))
                           : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      const int t = pass * 16 + nt * 8 + g;
#pragma unroll
      for (int i = 0; i < 4; ++i)
        b[nt][i] = t < p.T ? __ldg(reinterpret_cast<const uint4*>(
                                 p.x + static_cast<size_t>(t) * p.d + k0 + 8 * (4 * i + tig)))
                           : make_uint4(0u, 0u, 0u, 0u);
    }
    float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 2; ++j)
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
          mma_16816(acc[nt], word_of(a[0][i], 2 * j), word_of(a[1][i], 2 * j),
                    word_of(a[0][i], 2 * j + 1), word_of(a[1][i], 2 * j + 1),
                    word_of(b[nt][i], 2 * j), word_of(b[nt][i], 2 * j + 1));
    // acc[nt] = {(e0 + g, token 2 tig), (e0 + g, 2 tig + 1), (e0 + g + 8, 2 tig), (.., 2 tig + 1)}
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int t = pass * 16 + nt * 8 + 2 * tig + (q & 1);
        const int e = rg * 16 + g + 8 * (q >> 1);
        if (t < p.T && e < p.E)
          p.partial[(static_cast<size_t>(r) * p.T + t) * p.npad + e] = acc[nt][q];
      }
  }
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    moe_decode_fused_kernel(const __grid_constant__ FusedParams p) {
  __shared__ uint32_t s_tmem;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // the pair's tensor memory, for both GEMM phases
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(&s_tmem), kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = s_tmem;

  router_partials(p);
  grid_sync(p);

  const int splits = p.d / kRouterRange;
  for (int t = blockIdx.x * kFuWarps + warp; t < p.T; t += gridDim.x * kFuWarps) {
    if (p.E <= 64)
      topk_warp<2, true>(p.partial, splits, p.T, p.npad, p.E, p.k, p.bias, p.sel_only, t, lane,
                         p.ids, p.gates);
    else if (p.E <= 128)
      topk_warp<4, true>(p.partial, splits, p.T, p.npad, p.E, p.k, p.bias, p.sel_only, t, lane,
                         p.ids, p.gates);
    else
      topk_warp<8, true>(p.partial, splits, p.T, p.npad, p.E, p.k, p.bias, p.sel_only, t, lane,
                         p.ids, p.gates);
  }
  grid_sync(p);

  if (blockIdx.x == 0)
    permute_small_block<kFuWarps, true>(p.ids, p.T * p.k, p.E, p.counts, p.offsets, p.perm,
                                        p.slot_pos, p.status);
  grid_sync(p);

  expert_gemm_body<kGateUp, true>(p.mw_gu, p.tx_gu, p.gu, tmem);
  grid_sync(p);
  expert_gemm_body<kDown, true>(p.mw_dn, p.tx_dn, p.dn, tmem);
  grid_sync(p);

  const int cpr = p.d / 8;  // 8-column groups per token
  const int n = p.T * cpr;
  for (int i = blockIdx.x * kThreads + threadIdx.x; i < n; i += gridDim.x * kThreads) {
    const int t = i / cpr;
    combine_cols<true, __half>(p.y, p.slot_pos, p.gates, nullptr, p.d, p.k, p.T * p.k, t,
                       (i - t * cpr) * 8, p.out, p.status);
  }

  tc_fence_before_sync();
  __syncthreads();
  cluster_sync();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after_sync();
    tmem_dealloc_pair(tmem, kTmemCols);
  }
  // The last CTA to leave resets the arrival counter (after a timeout it may
  // hold stale arrivals) for the next launch.
  if (threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(p.exit_count, 1u) == gridDim.x - 1) {
      atomicExch(p.bar_count, 0u);
      atomicExch(p.exit_count, 0u);
      __threadfence();
    }
  }
}

// Dynamic shared memory (all a block may use beside the kernel's static
// shared memory) and the number of co-resident CTA pairs; 0 on error.
struct FusedLaunchShape {
  int smem, pairs;
};

FusedLaunchShape fused_launch_shape() {
  static std::once_flag once[64];
  static FusedLaunchShape shape[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return {0, 0};
  std::call_once(once[dev], [&] {
    int optin = 0;
    cudaFuncAttributes fa{};
    if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
            cudaSuccess ||
        cudaFuncGetAttributes(&fa, moe_decode_fused_kernel) != cudaSuccess) {
      cudaGetLastError();
      return;
    }
    const int smem = optin - static_cast<int>(fa.sharedSizeBytes);
    if (cudaFuncSetAttribute(moe_decode_fused_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             smem) != cudaSuccess) {
      cudaGetLastError();
      return;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * (device_sm_count() / 2));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, moe_decode_fused_kernel, &cfg) != cudaSuccess ||
        n <= 0) {
      cudaGetLastError();
      return;
    }
    shape[dev] = {smem, std::min(n, device_sm_count() / 2)};
  });
  return shape[dev];
}

}  // namespace

size_t fused_partial_bytes(int T, int d, int E) {
  return static_cast<size_t>(d / kRouterRange) * T * router_npad(E) * sizeof(float);
}

cudaError_t launch_decode_fused(cudaStream_t s, const FusedLayer& L) {
  if (L.d % kRouterRange || L.I % kRouterRange || L.E > kMaxExperts || L.k > kMaxTopK ||
      L.T * L.k > kPermuteSmallMax)
    return cudaErrorInvalidValue;
  const FusedLaunchShape shape = fused_launch_shape();
  if (shape.pairs <= 0) return cudaErrorInvalidConfiguration;
  const int rows = L.T * L.k;
  FusedParams p{};
  // gate_up: interleaved weight map, token rows gathered from x through perm
  cudaError_t e = make_gate_up_weight_map(&p.mw_gu, L.w_gate_up, L.d, L.I, L.E);
  const TokenGather gather{L.x, L.perm, L.k, L.T};
  if (e == cudaSuccess) e = make_gate_up_token_maps(p.tx_gu, p.gu, L.x, rows, L.d, &gather);
  // down: W_down as [E d, I] in 128-row boxes, token rows = h
  if (e == cudaSuccess)
    e = make_bf16_map(&p.mw_dn, L.w_down, static_cast<uint64_t>(L.E) * L.d, L.I, 128);
  if (e == cudaSuccess) e = make_token_maps(p.tx_dn, L.h, rows, L.I);
  if (e != cudaSuccess) return e;
  Params& gu = p.gu;
  gu.K = L.d;
  gu.n_out = L.I;
  gu.slabs = (L.I + 127) / 128;
  gu.groups = L.E;
  gu.offsets = L.offsets;
  gu.total_rows = rows;
  gu.w_rows_per_group = 2 * L.I;
  gu.up_offset = L.I;
  gu.out = L.h;
  gu.ld_out = L.I;
  gu.smem_bytes = shape.smem;
  gu.status = L.status;
  gu.timeout_ns = L.timeout_ns;
  Params& dn = p.dn;
  dn.K = L.I;
  dn.n_out = L.d;
  dn.slabs = (L.d + 255) / 256;
  dn.groups = L.E;
  dn.offsets = L.offsets;
  dn.total_rows = rows;
  dn.w_rows_per_group = L.d;
  dn.up_offset = 0;
  dn.out = L.y;
  dn.ld_out = L.d;
  dn.smem_bytes = shape.smem;
  dn.status = L.status;
  dn.timeout_ns = L.timeout_ns;
  p.x = static_cast<const __nv_bfloat16*>(L.x);
  p.w_router = static_cast<const __nv_bfloat16*>(L.w_router);
  p.bias = L.bias;
  p.sel_only = L.bias_selection_only ? 1 : 0;
  p.T = L.T;
  p.d = L.d;
  p.E = L.E;
  p.k = L.k;
  p.partial = L.partial;
  p.npad = router_npad(L.E);
  p.ids = L.ids;
  p.gates = L.gates;
  p.counts = L.counts;
  p.offsets = L.offsets;
  p.perm = L.perm;
  p.slot_pos = L.slot_pos;
  p.y = static_cast<const __half*>(L.y);
  p.out = static_cast<__nv_bfloat16*>(L.out);
  p.status = L.status;
  p.bar_count = L.status + kBarrierCountWord;
  p.bar_gen = L.status + kBarrierGenWord;
  p.exit_count = L.status + kExitCountWord;
  p.timeout_ns = L.timeout_ns;

  // As many pairs as the larger GEMM phase has tiles at most (every expert
  // active, one token chunk each): a small layer waits at its grid barriers
  // for fewer CTAs.
  const long long tiles = static_cast<long long>(L.E) * std::max(gu.slabs, dn.slabs);
  const int pairs = static_cast<int>(std::max(1LL, std::min<long long>(shape.pairs, tiles)));
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * pairs);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = shape.smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  KernelScope scope(s, "moe_decode_fused");
  return cudaLaunchKernelEx(&cfg, moe_decode_fused_kernel, p);
}

}  // namespace moe
