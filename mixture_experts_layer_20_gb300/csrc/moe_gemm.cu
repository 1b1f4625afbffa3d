// Tensor-core kernels of the MoE layer on sm_103a: one warp-specialised,
// persistent tcgen05 GEMM used three ways.
//
//   router  : partial logits x W_r^T over one 512-wide K range per tile
//             (fp32); the top-k kernel sums the ranges in a fixed order.
//   gate_up : per expert, [G | U] = x_perm W_gu^T with the gate and up rows of
//             the same 128 output columns loaded side by side into one N=256
//             operand; the epilogue computes h = silu(G) * U and rounds it to
//             bf16 ('Chapter 9. Distributed inference', section 9.3.2: three
//             matrices per expert).
//   down    : per expert, y = h W_d^T, stored in fp32.
//
// Grouped M without padding copies ('Chapter 9. Distributed inference',
// section 9.4.3, grouped GEMM): an expert's rows are the contiguous range
// [offsets[e], offsets[e+1]) of the grouped activations.  Its M-tiles start
// at offsets[e] + 128 i; rows past the expert's end are loaded (they belong to
// the next expert, or lie past the tensor and read as zero) but never stored.
// Tiles are ordered (expert, n-tile, m-tile) so that the CTAs working at the
// same time share weight slabs through L2, and each CTA strides through that
// list (grid = SM count): every tile costs the same, so a static stride
// balances even a skewed expert distribution.
//
// Roles (192 threads): warp 0 issues TMA loads into a 4-stage shared-memory
// ring; warp 1 owns the tensor memory (512 columns = two 128 x 256 fp32
// accumulators) and one of its threads issues tcgen05.mma; warps 2-5 drain
// an accumulator (tcgen05.ld) while the next tile accumulates into the other.
// Every wait is bounded; on timeout the kernel records it in the status word,
// drains its copies and MMAs in flight, frees tensor memory and returns.

#include <algorithm>
#include <climits>
#include <mutex>

#include "moe_device.cuh"
#include "moe_internal.h"

namespace moe {
namespace {

constexpr int kBM = 128;  // rows per tile = MMA M
constexpr int kBK = 64;   // K per stage: one 128-byte swizzle row of bf16
constexpr int kStages = 4;
constexpr int kMaxN = 256;
constexpr int kABytes = kBM * kBK * 2;    // 16 KB
constexpr int kBBytes = kMaxN * kBK * 2;  // 32 KB
// Epilogue staging: per epilogue warp a 32 x 32 block of fp32 (rows padded
// to 36 words) used to turn row-per-lane registers into row-contiguous stores.
constexpr int kEpiStride = 36;
constexpr int kEpiWarpBytes = 32 * kEpiStride * 4;
constexpr int kSmemBytes = kStages * (kABytes + kBBytes) + 4 * kEpiWarpBytes + 1024;
constexpr int kThreads = 192;
constexpr int kEpiThreads = 128;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAccCols = 256;

enum Kind : int { kRouter = 0, kGateUp = 1, kDown = 2 };

struct GemmParams {
  int K;                 // reduction length, a multiple of 64
  int n_out;             // valid output columns: E, I or d
  int n_tiles;           // output tiles along N per M-tile
  int n_step;            // weight rows advanced per N-tile (gate_up 128, down 256)
  int b_rows_per_group;  // weight rows per expert in the B tensor map
  int b_box_rows;        // rows of one B box (gate_up: two boxes per stage)
  int up_offset;         // gate_up: row offset of the up half inside an expert
  int mma_n;             // MMA N
  int groups;            // experts, or 1 when offsets == nullptr
  const int32_t* offsets;
  int total_rows;        // rows of the A operand
  void* out;             // router: ids int32 [T,k]; gate_up: h bf16; down: y fp32
  float* out_gates;      // router: gates [T,k]
  const float* bias;     // router: [E] or nullptr
  int top_k;
  long long ld_out;      // output row stride in elements
  unsigned* status;
  unsigned long long timeout_ns;
  int k_splits;          // K ranges per output tile (router: d / 512; else 1)
  int kb_per_split;      // 64-wide K blocks per range
};

__device__ __forceinline__ void decode_tile(int tau, int n_tiles, int groups, const int* s_mt,
                                            const int* s_off, int& g, int& n, int& row0,
                                            int& row_end) {
  int lo = 0, hi = groups - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (s_mt[mid] * n_tiles <= tau) lo = mid; else hi = mid - 1;
  }
  g = lo;
  const int mt = s_mt[g + 1] - s_mt[g];
  const int local = tau - s_mt[g] * n_tiles;
  n = local / mt;
  row0 = s_off[g] + (local - n * mt) * kBM;
  row_end = s_off[g + 1];
}

// The epilogue of one tile for one warp.  Thread `lane` owns accumulator row
// row_base + lane (TMEM lane q*32 + lane).  Results go through `stage`, the
// warp's padded shared-memory block, so that global stores run along rows:
// each store instruction writes whole 64- or 128-byte row segments instead of
// 32 separate 16-byte pieces.  Rows at or past row_end are not stored.
template <int KIND>
__device__ __forceinline__ void epilogue_tile(const GemmParams& p, uint32_t t_row, int row_base,
                                              int row_end, int n, int split, uint32_t* stage) {
  const int lane = threadIdx.x & 31;
  if constexpr (KIND == kGateUp) {
    const int col0 = n * 128;
    __nv_bfloat16* h = static_cast<__nv_bfloat16*>(p.out);
#pragma unroll 1
    for (int c = 0; c < 128; c += 32) {
      uint32_t g[32], u[32];
      tmem_ld_32x32b_x32(t_row + c, g);
      tmem_ld_32x32b_x32(t_row + 128 + c, u);
      tmem_ld_wait();
      if (col0 + c >= p.n_out) continue;  // uniform across the warp
      uint32_t packed[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const float g0 = __uint_as_float(g[2 * j]), g1 = __uint_as_float(g[2 * j + 1]);
        const float u0 = __uint_as_float(u[2 * j]), u1 = __uint_as_float(u[2 * j + 1]);
        const float h0 = g0 / (1.0f + expf(-g0)) * u0;
        const float h1 = g1 / (1.0f + expf(-g1)) * u1;
        packed[j] = pack_bf16x2(h0, h1);
      }
      // 32 rows x 64 bytes, row pitch 20 words (80 bytes)
      uint4* w = reinterpret_cast<uint4*>(stage + lane * 20);
#pragma unroll
      for (int i = 0; i < 4; ++i)
        w[i] = make_uint4(packed[4 * i], packed[4 * i + 1], packed[4 * i + 2], packed[4 * i + 3]);
      __syncwarp();
#pragma unroll
      for (int r = 0; r < 32; r += 8) {
        const int rr = r + (lane >> 2);
        const uint4 v = *reinterpret_cast<const uint4*>(stage + rr * 20 + (lane & 3) * 4);
        const int row = row_base + rr;
        if (row < row_end)
          *reinterpret_cast<uint4*>(h + (size_t)row * p.ld_out + col0 + c + (lane & 3) * 8) = v;
      }
      __syncwarp();
    }
  } else if constexpr (KIND == kDown) {
    const int col0 = n * 256;
    float* y = static_cast<float*>(p.out);
#pragma unroll 1
    for (int c = 0; c < 256; c += 32) {
      uint32_t v[32];
      tmem_ld_32x32b_x32(t_row + c, v);
      tmem_ld_wait();
      if (col0 + c >= p.n_out) continue;  // uniform across the warp
      // 32 rows x 128 bytes, row pitch 36 words (144 bytes)
      uint4* w = reinterpret_cast<uint4*>(stage + lane * kEpiStride);
#pragma unroll
      for (int i = 0; i < 8; ++i) w[i] = make_uint4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
      __syncwarp();
#pragma unroll
      for (int r = 0; r < 32; r += 4) {
        const int rr = r + (lane >> 3);
        const uint4 val = *reinterpret_cast<const uint4*>(stage + rr * kEpiStride + (lane & 7) * 4);
        const int row = row_base + rr;
        if (row < row_end)
          *reinterpret_cast<uint4*>(y + (size_t)row * p.ld_out + col0 + c + (lane & 7) * 4) = val;
      }
      __syncwarp();
    }
  } else {  // router: this K range's partial logits, fp32 [split][row][mma_n]
    const int row = row_base + lane;
    const bool valid = row < row_end;
    float* dst = static_cast<float*>(p.out) + ((size_t)split * p.total_rows + row) * p.ld_out;
#pragma unroll 1
    for (int c = 0; c < p.mma_n; c += 16) {
      uint32_t v[16];
      tmem_ld_32x32b_x16(t_row + c, v);
      tmem_ld_wait();
      if (valid) {
        uint4* d4 = reinterpret_cast<uint4*>(dst + c);
#pragma unroll
        for (int i = 0; i < 4; ++i) d4[i] = make_uint4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
      }
    }
  }
}

template <int KIND>
__device__ __forceinline__ void gemm_body(const CUtensorMap& tmap_a, const CUtensorMap& tmap_b,
                                          const GemmParams& p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ int s_off[kMaxExperts + 1];
  __shared__ int s_mt[kMaxExperts + 1];
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
    tma_prefetch_desc(&tmap_a);
    tma_prefetch_desc(&tmap_b);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&s_tmem_base), kTmemCols);
    tmem_relinquish();
  }

  // Tile schedule: per-expert M-tile counts and their exclusive prefix.
  const int G = p.groups;
  for (int i = threadIdx.x; i <= G; i += blockDim.x)
    s_off[i] = p.offsets ? __ldg(p.offsets + i) : (i == 0 ? 0 : p.total_rows);
  __syncthreads();
  if (warp == 0) {
    const int per = (G + 31) / 32;
    int local = 0;
    bool bad = false;
    for (int j = 0; j < per; ++j) {
      const int g = lane * per + j;
      if (g < G) {
        const int m = s_off[g + 1] - s_off[g];
        bad |= m < 0;
        local += m > 0 ? (m + kBM - 1) / kBM : 0;
      }
    }
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    int run = incl - local;
    for (int j = 0; j < per; ++j) {
      const int g = lane * per + j;
      if (g < G) {
        s_mt[g] = run;
        const int m = s_off[g + 1] - s_off[g];
        run += m > 0 ? (m + kBM - 1) / kBM : 0;
      }
    }
    bad |= (s_off[0] != 0) || (s_off[G] != p.total_rows);
    bad = __any_sync(0xffffffffu, bad);
    __syncwarp();
    if (lane == 31) s_mt[G] = bad ? 0 : incl;
    if (bad && lane == 0 && blockIdx.x == 0) atomicOr(p.status, kStatusDeviceCheck);
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();

  const uint32_t tmem_base = s_tmem_base;
  const int total_tiles = s_mt[G] * p.n_tiles * p.k_splits;
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
        int g, n, row0, row_end;
        decode_tile(tau / p.k_splits, p.n_tiles, G, s_mt, s_off, g, n, row0, row_end);
        const int brow = g * p.b_rows_per_group + n * p.n_step;
        const int kb0 = (tau % p.k_splits) * p.kb_per_split;
        const int kb1 = min(num_kb, kb0 + p.kb_per_split);
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait(empty_bar + 8 * stage, phase ^ 1u, wc)) { ok = false; break; }
          const uint32_t fb = full_bar + 8 * stage;
          mbar_arrive_expect_tx(fb, tx_bytes);
          const uint32_t a_dst = a_base + stage * kABytes;
          const uint32_t b_dst = b_base + stage * kBBytes;
          tma_load_2d(a_dst, &tmap_a, fb, kb * kBK, row0);
          tma_load_2d(b_dst, &tmap_b, fb, kb * kBK, brow);
          if (KIND == kGateUp)
            tma_load_2d(b_dst + p.b_box_rows * kBK * 2, &tmap_b, fb, kb * kBK, brow + p.up_offset);
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
          for (int k = 0; k < kBK / 16; ++k) {
            mma_bf16_ss(d_tmem, smem_desc_sw128(a_addr + k * 32), smem_desc_sw128(b_addr + k * 32),
                        idesc, (kb != kb0 || k != 0) ? 1u : 0u);
          }
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
    uint32_t* epi_stage = reinterpret_cast<uint32_t*>(
        smem_raw + (base - smem_u32(smem_raw)) + kStages * (kABytes + kBBytes) + q * kEpiWarpBytes);
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int tau = blockIdx.x; tau < total_tiles; tau += gridDim.x) {
      int g, n, row0, row_end;
      decode_tile(tau / p.k_splits, p.n_tiles, G, s_mt, s_off, g, n, row0, row_end);
      const bool ok = mbar_wait(tfull_bar + 8 * acc, acc_phase, wc);
      if (!__all_sync(0xffffffffu, ok)) break;
      tc_fence_after_sync();
      const uint32_t t_row = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * kAccCols;
      epilogue_tile<KIND>(p, t_row, row0 + q * 32, row_end, n, tau % p.k_splits, epi_stage);
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

__global__ void __launch_bounds__(kThreads, 1)
    moe_router_logits_kernel(const __grid_constant__ CUtensorMap tmap_a,
                           const __grid_constant__ CUtensorMap tmap_b, const GemmParams p) {
  gemm_body<kRouter>(tmap_a, tmap_b, p);
}

__global__ void __launch_bounds__(kThreads, 1)
    moe_gate_up_swiglu_kernel(const __grid_constant__ CUtensorMap tmap_a,
                              const __grid_constant__ CUtensorMap tmap_b, const GemmParams p) {
  gemm_body<kGateUp>(tmap_a, tmap_b, p);
}

__global__ void __launch_bounds__(kThreads, 1)
    moe_down_kernel(const __grid_constant__ CUtensorMap tmap_a,
                    const __grid_constant__ CUtensorMap tmap_b, const GemmParams p) {
  gemm_body<kDown>(tmap_a, tmap_b, p);
}

typedef void (*GemmKernel)(const CUtensorMap, const CUtensorMap, const GemmParams);

template <int KIND>
constexpr GemmKernel kernel_of() {
  return KIND == kRouter ? moe_router_logits_kernel
                         : (KIND == kGateUp ? moe_gate_up_swiglu_kernel : moe_down_kernel);
}

// ------------------------------------------------------------------ host

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

// Row-major bf16 matrix [rows, cols] as a 2-D tensor map with a box of
// 64 columns x box_rows rows and 128-byte swizzling.
cudaError_t make_map(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols,
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

template <int KIND>
cudaError_t ensure_smem_attr() {
  static std::mutex mu;
  static unsigned done_mask = 0;  // one bit per device
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  if (dev < 32 && (done_mask >> dev) & 1u) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel_of<KIND>(), cudaFuncAttributeMaxDynamicSharedMemorySize,
                           kSmemBytes);
  if (e == cudaSuccess && dev < 32) done_mask |= 1u << dev;
  return e;
}

template <int KIND>
cudaError_t launch(cudaStream_t s, const char* name, const CUtensorMap& ma, const CUtensorMap& mb,
                   const GemmParams& p, long long tiles_bound) {
  cudaError_t e = ensure_smem_attr<KIND>();
  if (e != cudaSuccess) return e;
  const long long grid = std::max(1LL, std::min<long long>(device_sm_count(), tiles_bound));
  KernelScope scope(s, name);
  kernel_of<KIND>()<<<static_cast<unsigned>(grid), kThreads, kSmemBytes, s>>>(ma, mb, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_router_logits(cudaStream_t s, const void* x, const void* w_router, int T,
                                 int d, int E, float* partial, unsigned* status,
                                 unsigned long long timeout_ns) {
  const int mma_n = router_npad(E);
  CUtensorMap ma, mb;
  cudaError_t e = make_map(&ma, x, T, d, kBM);
  if (e == cudaSuccess) e = make_map(&mb, w_router, E, d, mma_n);
  if (e != cudaSuccess) return e;
  GemmParams p{};
  p.K = d;
  p.n_out = E;
  p.n_tiles = 1;
  p.n_step = 0;
  p.b_rows_per_group = 0;
  p.b_box_rows = mma_n;
  p.mma_n = mma_n;
  p.groups = 1;
  p.offsets = nullptr;
  p.total_rows = T;
  p.out = partial;
  p.ld_out = mma_n;
  p.status = status;
  p.timeout_ns = timeout_ns;
  p.k_splits = router_splits(d);
  p.kb_per_split = kRouterSplitK / kBK;
  return launch<kRouter>(s, "moe_router_logits", ma, mb, p,
                         static_cast<long long>((T + kBM - 1) / kBM) * p.k_splits);
}

cudaError_t launch_grouped_ffn(cudaStream_t s, const void* a, const int32_t* offsets, int rows,
                               int d, int E, int I, const void* w_gate_up, const void* w_down,
                               void* h, float* y, unsigned* status,
                               unsigned long long timeout_ns) {
  const int groups = offsets ? E : 1;
  const long long mtiles_bound =
      offsets ? rows / kBM + std::min(E, rows) : (rows + kBM - 1) / kBM;

  CUtensorMap ma, mb;
  cudaError_t e = make_map(&ma, a, rows, d, kBM);
  if (e == cudaSuccess) e = make_map(&mb, w_gate_up, static_cast<uint64_t>(groups) * 2 * I, d, 128);
  if (e != cudaSuccess) return e;
  GemmParams p{};
  p.K = d;
  p.n_out = I;
  p.n_tiles = (I + 127) / 128;
  p.n_step = 128;
  p.b_rows_per_group = 2 * I;
  p.b_box_rows = 128;
  p.up_offset = I;
  p.mma_n = 256;
  p.groups = groups;
  p.offsets = offsets;
  p.total_rows = rows;
  p.out = h;
  p.ld_out = I;
  p.status = status;
  p.timeout_ns = timeout_ns;
  p.k_splits = 1;
  p.kb_per_split = d / kBK;
  e = launch<kGateUp>(s, offsets ? "moe_gate_up_swiglu" : "moe_shared_gate_up_swiglu", ma, mb, p,
                      mtiles_bound * p.n_tiles);
  if (e != cudaSuccess) return e;

  CUtensorMap ma2, mb2;
  e = make_map(&ma2, h, rows, I, kBM);
  if (e == cudaSuccess) e = make_map(&mb2, w_down, static_cast<uint64_t>(groups) * d, I, 256);
  if (e != cudaSuccess) return e;
  GemmParams q{};
  q.K = I;
  q.n_out = d;
  q.n_tiles = (d + 255) / 256;
  q.n_step = 256;
  q.b_rows_per_group = d;
  q.b_box_rows = 256;
  q.mma_n = 256;
  q.groups = groups;
  q.offsets = offsets;
  q.total_rows = rows;
  q.out = y;
  q.ld_out = d;
  q.status = status;
  q.timeout_ns = timeout_ns;
  q.k_splits = 1;
  q.kb_per_split = I / kBK;
  return launch<kDown>(s, offsets ? "moe_down" : "moe_shared_down", ma2, mb2, q,
                       mtiles_bound * q.n_tiles);
}

}  // namespace moe
