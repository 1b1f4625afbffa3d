// Router logits on the tensor cores (sm_103a): x [T, d] times W_r [E, d]^T in
// fp32, as partial sums over 512-wide ranges of d (one range per work tile),
// written to partial [range][T][E rounded up to 16].  The top-k kernel
// (moe_router.cu) adds the ranges in order, so the number of ranges depends
// on d only and a token's logits do not depend on the rest of the batch.
//
// A persistent tcgen05 GEMM: warp 0 issues TMA loads into a 4-stage ring of
// {x: 128 x 64, W_r: up to 256 x 64} bf16 tiles (128-byte swizzle); one
// thread of warp 1 issues tcgen05.mma (M = 128, N = E rounded up to 16; W_r
// rows past E read as zero) into one of two TMEM accumulators; warps 2-5
// read the other accumulator with tcgen05.ld and store it.  Token rows past
// T read as zero and are not stored.  Every wait is bounded; on timeout the
// kernel records it in the status word, drains its copies and MMAs in flight,
// frees tensor memory and returns.
//
// This file also holds the tensor-map helper shared with the expert GEMMs.

#include <algorithm>
#include <mutex>

#include "moe_device.cuh"
#include "moe_internal.h"

namespace moe {
namespace {

constexpr int kBM = 128;  // tokens per tile = MMA M
constexpr int kBK = 64;   // K per stage: one 128-byte swizzle row of bf16
constexpr int kStages = 4;
constexpr int kMaxN = 256;
constexpr int kABytes = kBM * kBK * 2;    // 16 KB
constexpr int kBBytes = kMaxN * kBK * 2;  // 32 KB
constexpr int kSmemBytes = kStages * (kABytes + kBBytes) + 1024;
constexpr int kThreads = 192;
constexpr int kEpiThreads = 128;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAccCols = 256;

struct RouterParams {
  int T, K;            // tokens, reduction length (d)
  int mma_n;           // E rounded up to 16
  int k_splits;        // 512-wide ranges of d
  int kb_per_split;    // 64-wide K blocks per range
  float* partial;      // [k_splits][T][mma_n]
  unsigned* status;
  unsigned long long timeout_ns;
};

__global__ void __launch_bounds__(kThreads, 1)
    moe_router_logits_kernel(const __grid_constant__ CUtensorMap tmap_x,
                             const __grid_constant__ CUtensorMap tmap_w, const RouterParams p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ alignas(8) uint64_t s_bar[2 * kStages + 5];
  __shared__ uint32_t s_tmem_base;
  __shared__ int s_abort;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t a_base = base;
  const uint32_t b_base = base + kStages * kABytes;
  const uint32_t full_bar = smem_u32(&s_bar[0]);
  const uint32_t empty_bar = smem_u32(&s_bar[kStages]);
  const uint32_t tfull_bar = smem_u32(&s_bar[2 * kStages]);
  const uint32_t tempty_bar = smem_u32(&s_bar[2 * kStages + 2]);
  const uint32_t drain_bar = smem_u32(&s_bar[2 * kStages + 4]);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full_bar + 8 * s, 1);
      mbar_init(empty_bar + 8 * s, 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull_bar + 8 * a, 1);
      mbar_init(tempty_bar + 8 * a, kEpiThreads);
    }
    mbar_init(drain_bar, 1);
    s_abort = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmap_x);
    tma_prefetch_desc(&tmap_w);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&s_tmem_base), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  pdl_wait_and_release();

  const uint32_t tmem_base = s_tmem_base;
  const int m_tiles = (p.T + kBM - 1) / kBM;
  const int total_tiles = m_tiles * p.k_splits;
  const int num_kb = p.K / kBK;
  const WaitCtx wc{p.timeout_ns, p.status, &s_abort};

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer
      const uint32_t tx_bytes = kABytes + static_cast<uint32_t>(p.mma_n) * kBK * 2;
      int stage = 0;
      uint32_t phase = 0;
      int issued = 0;
      bool ok = true;
      for (int tau = blockIdx.x; tau < total_tiles && ok; tau += gridDim.x) {
        const int row0 = (tau / p.k_splits) * kBM;
        const int kb0 = (tau % p.k_splits) * p.kb_per_split;
        const int kb1 = min(num_kb, kb0 + p.kb_per_split);
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait(empty_bar + 8 * stage, phase ^ 1u, wc)) { ok = false; break; }
          const uint32_t fb = full_bar + 8 * stage;
          mbar_arrive_expect_tx(fb, tx_bytes);
          tma_load_2d(a_base + stage * kABytes, &tmap_x, fb, kb * kBK, row0);
          tma_load_2d(b_base + stage * kBBytes, &tmap_w, fb, kb * kBK, 0);
          ++issued;
          if (++stage == kStages) { stage = 0; phase ^= 1u; }
        }
      }
      // Drain: the last (up to kStages) loads may still be landing.
      for (int i = max(0, issued - kStages); i < issued; ++i)
        mbar_wait_drain(full_bar + 8 * (i % kStages), (i / kStages) & 1, p.status);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer
      const uint32_t idesc = idesc_bf16_f32(kBM, p.mma_n);
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int tau = blockIdx.x; tau < total_tiles && ok; tau += gridDim.x) {
        if (!mbar_wait(tempty_bar + 8 * acc, acc_phase ^ 1u, wc)) { ok = false; break; }
        tc_fence_after_sync();
        const uint32_t d_tmem = tmem_base + acc * kAccCols;
        const int kb0 = (tau % p.k_splits) * p.kb_per_split;
        const int kb1 = min(num_kb, kb0 + p.kb_per_split);
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait(full_bar + 8 * stage, phase, wc)) { ok = false; break; }
          tc_fence_after_sync();
          const uint32_t a_addr = a_base + stage * kABytes;
          const uint32_t b_addr = b_base + stage * kBBytes;
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k)
            mma_bf16_ss(d_tmem, smem_desc_sw128(a_addr + k * 32), smem_desc_sw128(b_addr + k * 32),
                        idesc, (kb != kb0 || k != 0) ? 1u : 0u);
          mma_commit(empty_bar + 8 * stage);  // frees the stage once these MMAs finish
          if (++stage == kStages) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        mma_commit(tfull_bar + 8 * acc);      // accumulator ready for the epilogue
        if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
      }
      // Drain: every MMA this thread issued completes before TMEM is freed.
      mma_commit(drain_bar);
      mbar_wait_drain(drain_bar, 0, p.status);
    }
  } else {
    // ---------------- epilogue: warps 2..5 cover TMEM lanes by (warp % 4)
    const int q = warp & 3;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int tau = blockIdx.x; tau < total_tiles; tau += gridDim.x) {
      const bool ok = mbar_wait(tfull_bar + 8 * acc, acc_phase, wc);
      if (!__all_sync(0xffffffffu, ok)) break;
      tc_fence_after_sync();
      const int row = (tau / p.k_splits) * kBM + q * 32 + lane;
      const int split = tau % p.k_splits;
      const uint32_t t_row = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * kAccCols;
      float* dst = p.partial + ((size_t)split * p.T + row) * p.mma_n;
#pragma unroll 1
      for (int c = 0; c < p.mma_n; c += 16) {
        uint32_t v[16];
        tmem_ld_32x32b_x16(t_row + c, v);
        tmem_ld_wait();
        if (row < p.T) {
          uint4* d4 = reinterpret_cast<uint4*>(dst + c);
#pragma unroll
          for (int i = 0; i < 4; ++i) d4[i] = make_uint4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
        }
      }
      tc_fence_before_sync();
      mbar_arrive(tempty_bar + 8 * acc);
      if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

// The same logits for large batches in one pass per tile: a tile is 128
// tokens by a chunk of at most 128 experts, and it runs over all 512-wide
// ranges of d.  Each range is accumulated into one of two TMEM accumulators
// (so the next range's MMAs overlap the epilogue of this one); the epilogue
// threads (one token row each) add the ranges into a running sum in
// registers, starting from +0 and in range order, exactly as the top-k
// kernel adds the partial sums, so the logits are bit for bit those of the
// split kernel above.  Only the final sums are written (one range of
// partial), so the top-k kernel reads T x E values instead of splits times as
// many.
constexpr int kAccMaxN = 128;  // experts per tile
constexpr int kAccBBytes = kAccMaxN * kBK * 2;  // 16 KB
constexpr int kAccStages = 6;  // 6 x 32 KB: the split kernel's shared memory
static_assert(kAccStages * (kABytes + kAccBBytes) + 1024 <= kSmemBytes, "fits the same allocation");

struct RouterAccParams {
  int T, K;
  int n_per;           // experts per tile (multiple of 16, <= kAccMaxN)
  int n_chunks;        // expert chunks: tiles = m tiles x n_chunks
  int npad;            // row length of partial (E rounded up to 16)
  int k_splits;        // 512-wide ranges of d
  int kb_per_split;    // 64-wide K blocks per range
  float* partial;      // [T][npad]: the logits
  unsigned* status;
  unsigned long long timeout_ns;
};

__global__ void __launch_bounds__(kThreads, 1)
    moe_router_logits_accum_kernel(const __grid_constant__ CUtensorMap tmap_x,
                                   const __grid_constant__ CUtensorMap tmap_w,
                                   const RouterAccParams p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ alignas(8) uint64_t s_bar[2 * kAccStages + 5];
  __shared__ uint32_t s_tmem_base;
  __shared__ int s_abort;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t a_base = base;
  const uint32_t b_base = base + kAccStages * kABytes;
  const uint32_t full_bar = smem_u32(&s_bar[0]);
  const uint32_t empty_bar = smem_u32(&s_bar[kAccStages]);
  const uint32_t tfull_bar = smem_u32(&s_bar[2 * kAccStages]);
  const uint32_t tempty_bar = smem_u32(&s_bar[2 * kAccStages + 2]);
  const uint32_t drain_bar = smem_u32(&s_bar[2 * kAccStages + 4]);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kAccStages; ++s) {
      mbar_init(full_bar + 8 * s, 1);
      mbar_init(empty_bar + 8 * s, 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull_bar + 8 * a, 1);
      mbar_init(tempty_bar + 8 * a, kEpiThreads);
    }
    mbar_init(drain_bar, 1);
    s_abort = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmap_x);
    tma_prefetch_desc(&tmap_w);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&s_tmem_base), 2 * kAccMaxN);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  pdl_wait_and_release();

  const uint32_t tmem_base = s_tmem_base;
  const int m_tiles = (p.T + kBM - 1) / kBM;
  const int total_tiles = m_tiles * p.n_chunks;
  const int num_kb = p.K / kBK;
  const WaitCtx wc{p.timeout_ns, p.status, &s_abort};

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer: every K block of the tile, in order
      const uint32_t tx_bytes = kABytes + static_cast<uint32_t>(p.n_per) * kBK * 2;
      int stage = 0;
      uint32_t phase = 0;
      int issued = 0;
      bool ok = true;
      for (int tau = blockIdx.x; tau < total_tiles && ok; tau += gridDim.x) {
        const int row0 = (tau / p.n_chunks) * kBM;
        const int e0 = (tau % p.n_chunks) * p.n_per;
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!mbar_wait(empty_bar + 8 * stage, phase ^ 1u, wc)) { ok = false; break; }
          const uint32_t fb = full_bar + 8 * stage;
          mbar_arrive_expect_tx(fb, tx_bytes);
          tma_load_2d(a_base + stage * kABytes, &tmap_x, fb, kb * kBK, row0);
          tma_load_2d(b_base + stage * kAccBBytes, &tmap_w, fb, kb * kBK, e0);
          ++issued;
          if (++stage == kAccStages) { stage = 0; phase ^= 1u; }
        }
      }
      for (int i = max(0, issued - kAccStages); i < issued; ++i)
        mbar_wait_drain(full_bar + 8 * (i % kAccStages), (i / kAccStages) & 1, p.status);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer: one accumulation per range
      const uint32_t idesc = idesc_bf16_f32(kBM, p.n_per);
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int tau = blockIdx.x; tau < total_tiles && ok; tau += gridDim.x) {
        for (int sp = 0; sp < p.k_splits && ok; ++sp) {
          if (!mbar_wait(tempty_bar + 8 * acc, acc_phase ^ 1u, wc)) { ok = false; break; }
          tc_fence_after_sync();
          const uint32_t d_tmem = tmem_base + acc * kAccMaxN;
          const int kb0 = sp * p.kb_per_split;
          const int kb1 = min(num_kb, kb0 + p.kb_per_split);
          for (int kb = kb0; kb < kb1; ++kb) {
            if (!mbar_wait(full_bar + 8 * stage, phase, wc)) { ok = false; break; }
            tc_fence_after_sync();
            const uint32_t a_addr = a_base + stage * kABytes;
            const uint32_t b_addr = b_base + stage * kAccBBytes;
#pragma unroll
            for (int k = 0; k < kBK / 16; ++k)
              mma_bf16_ss(d_tmem, smem_desc_sw128(a_addr + k * 32),
                          smem_desc_sw128(b_addr + k * 32), idesc,
                          (kb != kb0 || k != 0) ? 1u : 0u);
            mma_commit(empty_bar + 8 * stage);
            if (++stage == kAccStages) { stage = 0; phase ^= 1u; }
          }
          if (!ok) break;
          mma_commit(tfull_bar + 8 * acc);  // this range's sums ready for the epilogue
          if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
        }
      }
      mma_commit(drain_bar);
      mbar_wait_drain(drain_bar, 0, p.status);
    }
  } else {
    // ---------------- epilogue: warps 2..5, TMEM lane = token row of the tile
    const int q = warp & 3;
    int acc = 0;
    uint32_t acc_phase = 0;
    bool live = true;
    for (int tau = blockIdx.x; tau < total_tiles && live; tau += gridDim.x) {
      const int row = (tau / p.n_chunks) * kBM + q * 32 + lane;
      const int e0 = (tau % p.n_chunks) * p.n_per;
      float sum[kAccMaxN];
#pragma unroll
      for (int i = 0; i < kAccMaxN; ++i) sum[i] = 0.0f;
      for (int sp = 0; sp < p.k_splits; ++sp) {
        const bool ok = mbar_wait(tfull_bar + 8 * acc, acc_phase, wc);
        if (!__all_sync(0xffffffffu, ok)) { live = false; break; }
        tc_fence_after_sync();
        const uint32_t t_row = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * kAccMaxN;
#pragma unroll
        for (int c = 0; c < kAccMaxN; c += 16) {
          if (c < p.n_per) {
            uint32_t v[16];
            tmem_ld_32x32b_x16(t_row + c, v);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 16; ++i) sum[c + i] += __uint_as_float(v[i]);
          }
        }
        tc_fence_before_sync();
        mbar_arrive(tempty_bar + 8 * acc);
        if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
      }
      if (live && row < p.T) {
        // the last chunk may reach past the row's npad columns: not stored
        const int n_valid = min(p.n_per, p.npad - e0);
        float* dst = p.partial + (size_t)row * p.npad + e0;
#pragma unroll
        for (int c = 0; c < kAccMaxN; c += 16) {
          if (c < n_valid) {
            uint4* d4 = reinterpret_cast<uint4*>(dst + c);
#pragma unroll
            for (int i = 0; i < 4; ++i)
              d4[i] = make_uint4(__float_as_uint(sum[c + 4 * i]), __float_as_uint(sum[c + 4 * i + 1]),
                                 __float_as_uint(sum[c + 4 * i + 2]),
                                 __float_as_uint(sum[c + 4 * i + 3]));
          }
        }
      }
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, 2 * kAccMaxN);
  }
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  return fn;
}

cudaError_t ensure_router_smem_attr() {
  static std::mutex mu;
  static unsigned done_mask = 0;  // one bit per device
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  if (dev < 32 && (done_mask >> dev) & 1u) return cudaSuccess;
  e = cudaFuncSetAttribute(moe_router_logits_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           kSmemBytes);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(moe_router_logits_accum_kernel,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e == cudaSuccess && dev < 32) done_mask |= 1u << dev;
  return e;
}

}  // namespace

cudaError_t make_bf16_map(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols,
                          uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return cudaErrorNotSupported;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 2};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(kBK), box_rows};
  const cuuint32_t estride[2] = {1, 1};
  const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims,
                        strides, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t make_bf16_map_nd(CUtensorMap* m, const void* base, int rank, const uint64_t* dims,
                             const uint64_t* strides_bytes, const uint32_t* box) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return cudaErrorNotSupported;
  cuuint64_t d[5], st[4];
  cuuint32_t b[5], es[5];
  for (int i = 0; i < rank; ++i) {
    d[i] = dims[i];
    b[i] = box[i];
    es[i] = 1;
    if (i + 1 < rank) st[i] = strides_bytes[i];
  }
  const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(base), d, st,
                        b, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t make_u8_map_nd(CUtensorMap* m, const void* base, int rank, const uint64_t* dims,
                           const uint64_t* strides_bytes, const uint32_t* box) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return cudaErrorNotSupported;
  cuuint64_t d[5], st[4];
  cuuint32_t b[5], es[5];
  for (int i = 0; i < rank; ++i) {
    d[i] = dims[i];
    b[i] = box[i];
    es[i] = 1;
    if (i + 1 < rank) st[i] = strides_bytes[i];
  }
  const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, rank, const_cast<void*>(base), d, st, b,
                        es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// One pass per tile over all ranges (moe_router_logits_accum) when the batch
// has at least 16 token tiles and the partial sums of the split kernel would
// move (written, then read) more than 1.5 times the bytes of x; otherwise one
// tile per range, which spreads a tile's K over many SMs.  Both give the same
// logits.  Measured (router logits + top-k): the DeepSeek-like layer (d = 7168,
// 14 ranges, E = 256) 64 against 108 us; the 6000-token Qwen3 prefill (8
// ranges, E = 128) 40 against 37 us, so it keeps the split kernel.
constexpr int kAccumMinTiles = 16;

int router_ranges_written(int T, int d, int E) {
  const long long partial_bytes = 8LL * router_splits(d) * router_npad(E);  // per token
  const long long x_bytes = 2LL * d;
  const bool accum = (T + kBM - 1) / kBM >= kAccumMinTiles && 2 * partial_bytes > 3 * x_bytes;
  return accum ? 1 : router_splits(d);
}

cudaError_t launch_router_logits(cudaStream_t s, const void* x, const void* w_router, int T,
                                 int d, int E, float* partial, unsigned* status,
                                 unsigned long long timeout_ns) {
  const int m_tiles = (T + kBM - 1) / kBM;
  const int npad = router_npad(E);
  cudaError_t e = ensure_router_smem_attr();
  if (e != cudaSuccess) return e;
  CUtensorMap mx, mw;
  e = make_bf16_map(&mx, x, T, d, kBM);
  if (e != cudaSuccess) return e;
  if (router_ranges_written(T, d, E) == 1) {
    RouterAccParams p{};
    p.T = T;
    p.K = d;
    p.npad = npad;
    p.k_splits = router_splits(d);
    p.kb_per_split = kRouterSplitK / kBK;
    // expert chunks: enough tiles for every SM, at most kAccMaxN experts each
    const int sms = device_sm_count();
    int chunks = std::max((npad + kAccMaxN - 1) / kAccMaxN, std::min(npad / 16, sms / m_tiles));
    p.n_per = ((npad + chunks - 1) / chunks + 15) / 16 * 16;
    p.n_chunks = (npad + p.n_per - 1) / p.n_per;
    p.partial = partial;
    p.status = status;
    p.timeout_ns = timeout_ns;
    e = make_bf16_map(&mw, w_router, E, d, p.n_per);
    if (e != cudaSuccess) return e;
    const long long tiles = static_cast<long long>(m_tiles) * p.n_chunks;
    const long long grid = std::max(1LL, std::min<long long>(sms, tiles));
    KernelScope scope(s, "moe_router_logits");
    cudaError_t le = launch_kernel(moe_router_logits_accum_kernel,
                                   dim3(static_cast<unsigned>(grid)), dim3(kThreads), kSmemBytes,
                                   s, mx, mw, p);
    if (le != cudaSuccess) return le;
    return cudaGetLastError();
  }
  RouterParams p{};
  p.T = T;
  p.K = d;
  p.mma_n = npad;
  p.k_splits = router_splits(d);
  p.kb_per_split = kRouterSplitK / kBK;
  p.partial = partial;
  p.status = status;
  p.timeout_ns = timeout_ns;
  e = make_bf16_map(&mw, w_router, E, d, p.mma_n);
  if (e != cudaSuccess) return e;
  const long long tiles = static_cast<long long>(m_tiles) * p.k_splits;
  const long long grid = std::max(1LL, std::min<long long>(device_sm_count(), tiles));
  KernelScope scope(s, "moe_router_logits");
  cudaError_t le = launch_kernel(moe_router_logits_kernel, dim3(static_cast<unsigned>(grid)),
                                 dim3(kThreads), kSmemBytes, s, mx, mw, p);
  if (le != cudaSuccess) return le;
  return cudaGetLastError();
}

}  // namespace moe
