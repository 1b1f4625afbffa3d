// The whole MoE layer in one kernel launch, for decode-sized batches.
//
// 'Hosting Qwen on Blackwell', "Expert parallelism": for decode the dispatch,
// the expert GEMMs and the combine run as one kernel, while prefill splits
// them.  Here one persistent cooperative launch (every CTA resident at once)
// runs the layer's steps as phases separated by grid-wide barriers:
//
//   1. router logits: fp32 partial sums of x W_r^T over 128-wide ranges of d,
//      warp-level tensor-core MMAs (16 experts x 8 tokens per MMA tile);
//   2. top-k and gates: one warp per token adds the ranges in range order
//      (the same warp code as the standalone router);
//   3. grouping: counts, offsets and the stable permutation, by one CTA;
//   4. gate_up with the SwiGLU epilogue and 5. down: the small-M grouped
//      GEMMs (warp-level MMAs, weights streamed through per-warp cp.async
//      rings), token rows taken from x through the permutation;
//   6. combine: fp32 sum of each token's k rows in slot order, one bf16
//      rounding.
//
// A grid-wide barrier is an arrival counter and a generation word in the
// workspace's status region; thread 0 of each CTA arrives and waits for the
// generation to move, bounded by %globaltimer.  A wait that runs out records
// MOE_ERR_TIMEOUT and its CTA skips the rest of the layer (the others then
// run out too), so a missing CTA cannot hang the GPU.  The last CTA to leave
// resets the counters, so the next launch starts clean even after a timeout.
// Data one phase writes and a later phase reads goes through L2 (ld_in with
// COHERENT = true).

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>
#include <mutex>

#include "moe_device.cuh"
#include "moe_internal.h"
#include "moe_permute.cuh"
#include "moe_router.cuh"
#include "moe_smallm.cuh"

namespace moe {
namespace {

constexpr int kRouterRange = 128;  // the router's partial sums: 128-wide ranges of d

struct FusedParams {
  const __nv_bfloat16* x;         // [T, d]
  const __nv_bfloat16* w_router;  // [E, d]
  const float* bias;              // [E] or null
  int sel_only;
  int T, d, E, k;
  float* partial;                 // [d / 128][T][npad]
  int npad;
  int32_t *ids, *counts, *offsets, *perm, *slot_pos;
  float* gates;
  SmParams gu, dn;                // the two grouped GEMMs
  const __half* y;                // [T k, d] (dn.out)
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

// Grid-wide barrier (every thread of every CTA).  Returns false when the wait
// ran out; the caller then skips the rest of the layer.
__device__ __forceinline__ bool grid_sync(const FusedParams& p) {
  __shared__ int s_ok;
  __syncthreads();
  if (threadIdx.x == 0) {
    int ok = 1;
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
          ok = 0;
          break;
        }
      }
    }
    __threadfence();
    s_ok = ok;
  }
  __syncthreads();
  return s_ok != 0;
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
  const int W = gridDim.x * kSmWarps;
  for (int tau = blockIdx.x * kSmWarps + (threadIdx.x >> 5); tau < total; tau += W) {
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

__global__ void __launch_bounds__(kSmThreads, 2) moe_decode_fused_kernel(const FusedParams p) {
  extern __shared__ __align__(16) uint8_t sm_raw[];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  router_partials(p);
  bool alive = grid_sync(p);

  if (alive) {
    const int splits = p.d / kRouterRange;
    for (int t = blockIdx.x * kSmWarps + warp; t < p.T; t += gridDim.x * kSmWarps) {
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
    alive = grid_sync(p);
  }
  if (alive) {
    if (blockIdx.x == 0)
      permute_small_block<kSmWarps, true>(p.ids, p.T * p.k, p.E, p.counts, p.offsets, p.perm,
                                          p.slot_pos, p.status);
    alive = grid_sync(p);
  }
  if (alive) {
    sm_phase<kSmBf16, kSmGateUp, true>(p.gu, sm_raw);
    alive = grid_sync(p);
  }
  if (alive) {
    sm_phase<kSmBf16, kSmDown, true>(p.dn, sm_raw);
    alive = grid_sync(p);
  }
  if (alive) {
    const int cpr = p.d / 8;  // 8-column groups per token
    const int n = p.T * cpr;
    for (int i = blockIdx.x * kSmThreads + threadIdx.x; i < n; i += gridDim.x * kSmThreads) {
      const int t = i / cpr;
      combine_cols<true>(p.y, p.slot_pos, p.gates, nullptr, p.d, p.k, p.T * p.k, t,
                         (i - t * cpr) * 8, p.out, p.status);
    }
  }

  // The last CTA to leave resets the arrival counter (after a timeout it may
  // hold stale arrivals) for the next launch.
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(p.exit_count, 1u) == gridDim.x - 1) {
      atomicExch(p.bar_count, 0u);
      atomicExch(p.exit_count, 0u);
      __threadfence();
    }
  }
}

// CTAs per SM that can be resident with the kernel's shared memory (0 on error).
int fused_blocks_per_sm() {
  static std::once_flag once[64];
  static int blocks[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  std::call_once(once[dev], [&] {
    constexpr int smem = sm_smem_bytes<kSmBf16>();
    int n = 0;
    if (cudaFuncSetAttribute(moe_decode_fused_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             smem) == cudaSuccess &&
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, moe_decode_fused_kernel, kSmThreads,
                                                      smem) == cudaSuccess)
      blocks[dev] = std::min(n, 2);
    else
      cudaGetLastError();
  });
  return blocks[dev];
}

}  // namespace

size_t fused_partial_bytes(int T, int d, int E) {
  return static_cast<size_t>(d / kRouterRange) * T * router_npad(E) * sizeof(float);
}

cudaError_t launch_decode_fused(cudaStream_t s, const FusedLayer& L) {
  if (L.d % kRouterRange || L.I % kRouterRange || L.E > kMaxExperts || L.k > kMaxTopK ||
      L.T * L.k > kPermuteSmallMax)
    return cudaErrorInvalidValue;
  const int per_sm = fused_blocks_per_sm();
  if (per_sm <= 0) return cudaErrorInvalidConfiguration;
  const int rows = L.T * L.k;
  FusedParams p{};
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
  SmParams& gu = p.gu;
  gu.w = static_cast<const uint8_t*>(L.w_gate_up);
  gu.row_bytes = static_cast<long long>(L.d) * 2;
  gu.K = L.d;
  gu.n_out = L.I;
  gu.w_rows_per_expert = 2 * L.I;
  gu.up_offset = L.I;
  gu.E = L.E;
  gu.offsets = L.offsets;
  gu.total_rows = rows;
  gu.b = p.x;
  gu.b_rows = L.T;
  gu.perm = L.perm;
  gu.div = L.k;
  gu.out = L.h;
  gu.ld_out = L.I;
  gu.status = L.status;
  SmParams& dn = p.dn;
  dn = gu;
  dn.w = static_cast<const uint8_t*>(L.w_down);
  dn.row_bytes = static_cast<long long>(L.I) * 2;
  dn.K = L.I;
  dn.n_out = L.d;
  dn.w_rows_per_expert = L.d;
  dn.up_offset = 0;
  dn.b = static_cast<const __nv_bfloat16*>(L.h);
  dn.b_rows = rows;
  dn.perm = nullptr;
  dn.div = 1;
  dn.out = L.y;
  dn.ld_out = L.d;
  p.y = static_cast<const __half*>(L.y);
  p.out = static_cast<__nv_bfloat16*>(L.out);
  p.status = L.status;
  p.bar_count = L.status + kBarrierCountWord;
  p.bar_gen = L.status + kBarrierGenWord;
  p.exit_count = L.status + kExitCountWord;
  p.timeout_ns = L.timeout_ns;

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(per_sm * device_sm_count());
  cfg.blockDim = dim3(kSmThreads);
  cfg.dynamicSmemBytes = sm_smem_bytes<kSmBf16>();
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
