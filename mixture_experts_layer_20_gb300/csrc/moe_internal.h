// Host-side declarations shared by the library's translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstddef>
#include <cstdint>
#include <string>
#include <utility>

namespace moe {

constexpr int kMaxExperts = 256;
constexpr int kMaxTopK = 8;
constexpr int kPermuteChunk = 1024;     // assignments per count / scatter CTA
constexpr int kPermuteSmallMax = 4096;  // up to this many, one CTA groups them all

// The router's logits are sums over K ranges of 512 on the tensor cores,
// added in range order starting from +0 (by the top-k kernel, or, for large
// batches, already by the logits kernel, which then writes one range).  The
// number of ranges depends on d only, so a token's logits do not depend on
// the batch.
constexpr int kRouterSplitK = 512;
inline int router_splits(int d) { return (d + kRouterSplitK - 1) / kRouterSplitK; }
inline int router_npad(int E) { return (E + 15) / 16 * 16; }
inline size_t router_partial_bytes(int T, int d, int E) {
  return static_cast<size_t>(router_splits(d)) * T * router_npad(E) * sizeof(float);
}
// Ranges the logits kernel writes for a batch of T tokens (moe_gemm.cu).
int router_ranges_written(int T, int d, int E);

// Words of the workspace's 256-byte status region: word 0 is the status word;
// the single-launch decode kernel keeps its grid-barrier counters in three
// more, each on its own 64-byte line (moe_workspace_init zeroes all of them).
constexpr int kBarrierCountWord = 16;
constexpr int kBarrierGenWord = 32;
constexpr int kExitCountWord = 48;
// The bf16 expert GEMMs' tile counter and exit counter (dynamic schedule):
// the next tile to hand out, and the CTAs that have left (the last one resets
// both to zero for the next launch).
constexpr int kTileCounterWord = 24;
constexpr int kTileExitWord = 40;

// Bits of the workspace's device status word.
constexpr unsigned kStatusTimeout = 1u;
constexpr unsigned kStatusDeviceCheck = 2u;
constexpr unsigned kStatusRange = 4u;  // an expert output outside the fp16 range of y

// Programmatic dependent launch.  Every kernel of the layer is launched with
// programmatic stream serialisation, so it may be scheduled while the kernel
// before it in the stream is still finishing.  Before its first global-memory
// access each kernel waits for that kernel to complete (griddepcontrol.wait;
// a no-op for a normal launch) and then lets the next kernel be scheduled:
// its launch latency and prologue (barrier init, tensor-memory allocation)
// overlap the tail of this one, and at most one kernel waits at a time.
#ifndef MOE_PDL
#define MOE_PDL 1
#endif
#ifdef __CUDACC__
__device__ __forceinline__ void pdl_wait_and_release() {
#if MOE_PDL
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
#endif
}

// A load of data the kernel only reads.  COHERENT = false: written by an
// earlier kernel (the read-only path, __ldg).  COHERENT = true: written by
// another CTA of the same kernel before a grid-wide barrier, so it is read
// from L2 (__ldcg), never from a possibly stale L1 line.
template <bool COHERENT, typename T>
__device__ __forceinline__ T ld_in(const T* p) {
  if constexpr (COHERENT) return __ldcg(p);
  else return __ldg(p);
}

template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                          cudaStream_t s, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = MOE_PDL;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}
#endif

// Records the kernel name, counts the launch and, while tracing is on,
// brackets it with CUDA events on `stream`.  Defined in moe_api.cu.
class KernelScope {
 public:
  KernelScope(cudaStream_t stream, const char* name);
  ~KernelScope();
  KernelScope(const KernelScope&) = delete;
  KernelScope& operator=(const KernelScope&) = delete;

 private:
  cudaStream_t stream_;
  int slot_;
};

int device_sm_count();

// Message returned by moe_last_error() on this thread.  Defined in moe_api.cu.
void set_last_error(const std::string& msg);

// Row-major bf16 matrix [rows, cols] as a 2-D TMA tensor map with a box of
// 64 columns x box_rows rows and 128-byte swizzling (moe_gemm.cu).
cudaError_t make_bf16_map(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                          uint32_t box_rows);

// bf16 tensor of rank 2..5 (dims innermost first, in elements; strides of
// dims 1.. in bytes) as a TMA tensor map with 128-byte swizzling; box[0] must
// be 64 (one 128-byte row).
cudaError_t make_bf16_map_nd(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                             const uint64_t* strides_bytes, const uint32_t* box);
// The same for a uint8 tensor (MXFP8 codes), 128-byte swizzle.
cudaError_t make_u8_map_nd(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                           const uint64_t* strides_bytes, const uint32_t* box);

// ---- tcgen05 GEMM launchers.  Return a CUDA error code.

// Router logits of x [T,d] against w_router [E,d] on the tensor cores:
// partial [router_ranges_written(T, d, E)][T][npad] fp32 (the partial sums over
// each 512-wide K range, or, for large batches, their in-order sum).
cudaError_t launch_router_logits(cudaStream_t s, const void* x, const void* w_router, int T,
                                 int d, int E, float* partial, unsigned* status,
                                 unsigned long long timeout_ns);

// Router: logits (via the partials in `partial`), bias, top-k with the
// lowest-index tie-break, renormalised gates (moe_router.cu).  With
// bias_selection_only the bias picks the experts and the gates come from the
// unbiased logits.
cudaError_t launch_router(cudaStream_t s, const void* x, const void* w_router, const float* bias,
                          int bias_selection_only, int T, int d, int E, int top_k, int32_t* ids,
                          float* gates, float* partial, unsigned* status,
                          unsigned long long timeout_ns);

// Gate_up's token rows taken straight from the unpermuted tokens: row pos of
// the grouped operand is src[perm[pos] / div] (src: [src_rows, d] bf16).
struct TokenGather {
  const void* src;
  const int32_t* perm;
  int div;
  int src_rows;
};

// Grouped SwiGLU FFN (moe_expert_gemm.cu).  Rows [offsets[e], offsets[e+1])
// of a [rows, d] go through expert e (weights per expert: w_gate_up [2I, d],
// w_down [d, I]).  offsets == nullptr: a single expert on all `rows` rows.
// With `gather`, a is not read: gate_up gathers its rows (see TokenGather).
// Writes h [rows, I] bf16 (scratch) and y [rows, d] fp16 (fp32 with y_fp32).
// sched_words: the workspace's status region (its tile and exit counters, at
// zero); the kernels then hand their tiles out in order through the counter
// instead of by a static stride.  Null: the static stride.
cudaError_t launch_grouped_ffn(cudaStream_t s, const void* a, const int32_t* offsets, int rows,
                               int d, int E, int I, const void* w_gate_up, const void* w_down,
                               void* h, void* y, unsigned* status,
                               unsigned long long timeout_ns,
                               const TokenGather* gather = nullptr, bool y_fp32 = false,
                               unsigned* sched_words = nullptr);

// The same with quantised expert weights (fmt 0: MXFP8, fmt 1: NVFP4):
// codes [E, 2I, d] / [E, d, I] (one byte per value for MXFP8, two values per
// byte for NVFP4) and block scales [K/128][rows][4] E8M0 (MXFP8) or
// [K/256][rows][16] E4M3 (NVFP4), rows = E*2I (gate_up) or E*d (down); NVFP4
// also a tensor scale per expert and matrix.  d and I multiples of 128
// (MXFP8) or 256 (NVFP4).
cudaError_t launch_grouped_ffn_quant(cudaStream_t s, int fmt, const void* a,
                                     const int32_t* offsets, int rows, int d, int E, int I,
                                     const uint8_t* codes_gate_up, const uint8_t* scales_gate_up,
                                     const float* tscale_gate_up, const uint8_t* codes_down,
                                     const uint8_t* scales_down, const float* tscale_down,
                                     void* h, void* y, unsigned* status,
                                     unsigned long long timeout_ns, bool y_fp32 = false);

// Grouped SwiGLU FFN for few token rows per expert (decode): warp-level
// tensor-core MMAs, weights decoded in registers (moe_smallm.cu).  fmt 1:
// MXFP8, 2: NVFP4 (scales and tensor scales as for launch_grouped_ffn_quant).
// Gate_up's token rows are a[perm[pos] / div] (perm != nullptr) or a[pos];
// d and I multiples of 256.
// Writes h [rows, I] bf16 and y [rows, d] fp16 (fp32 with y_fp32).
cudaError_t launch_grouped_ffn_smallm(cudaStream_t s, int fmt, const void* a,
                                      const int32_t* perm, int div, const int32_t* offsets,
                                      int rows, int d, int E, int I, const void* w_gate_up,
                                      const uint8_t* scales_gate_up, const float* tscale_gate_up,
                                      const void* w_down, const uint8_t* scales_down,
                                      const float* tscale_down, void* h, void* y,
                                      unsigned* status, bool y_fp32 = false);

// The same with MXFP8 tokens too (W8A8): x [T, d] is quantised into xq / xs
// ([T, d] codes, [T, d / 32] scales), h into hq / hs ([rows, I], [rows, I / 32])
// by launch_act_mxfp8; MXFP8 weights only.
cudaError_t launch_grouped_ffn_smallm_a8(cudaStream_t s, const void* x, int T,
                                         const int32_t* perm, int div, const int32_t* offsets,
                                         int rows, int d, int E, int I, const void* w_gate_up,
                                         const uint8_t* scales_gate_up, const void* w_down,
                                         const uint8_t* scales_down, uint8_t* xq, uint8_t* xs,
                                         void* h, uint8_t* hq, uint8_t* hs, void* y,
                                         unsigned* status, bool y_fp32 = false);

// The whole layer in one cooperative launch, for decode-sized batches with
// bf16 expert weights and no shared expert (moe_fused.cu).  Requires d and I
// multiples of 128, E <= 256 and T * k <= kPermuteSmallMax; partial holds
// fused_partial_bytes(T, d, E) bytes; status points at the workspace's status
// region (its barrier words must start at zero).
struct FusedLayer {
  const void* x;
  const void* w_router;
  const float* bias;
  int bias_selection_only;
  const void* w_gate_up;
  const void* w_down;
  int T, d, E, I, k;
  float* partial;
  int32_t* ids;
  float* gates;
  int32_t *counts, *offsets, *perm, *slot_pos;
  void* h;    // [T k, I] bf16
  void* y;    // [T k, d] fp16
  void* out;  // [T, d] bf16
  unsigned* status;
  unsigned long long timeout_ns;
};
size_t fused_partial_bytes(int T, int d, int E);
cudaError_t launch_decode_fused(cudaStream_t s, const FusedLayer& L);

// NVFP4 quantisation of `groups` matrices [rows_per_group, K] (K a multiple of
// 256) in one bf16 array: codes, scales as above, one tensor scale per matrix.
cudaError_t launch_nvfp4_quantize(cudaStream_t s, const void* w, int groups,
                                  long long rows_per_group, int K, uint8_t* codes,
                                  uint8_t* scales, float* tensor_scales);

// ---- grouping and combine (moe_permute.cu)

cudaError_t launch_permute(cudaStream_t s, const int32_t* ids, const void* x, int T, int d, int E,
                           int top_k, int32_t* counts, int32_t* offsets, int32_t* perm,
                           int32_t* slot_pos, void* x_perm, int32_t* chunk_table,
                           unsigned* status);

// y (and y_shared) fp16, or fp32 with y_fp32.
cudaError_t launch_combine(cudaStream_t s, const void* y, const int32_t* slot_pos,
                           const float* gates, const void* y_shared, int T, int d, int top_k,
                           void* out, unsigned* status, bool y_fp32 = false);

// ---- MXFP8 weights (moe_mxfp8.cu)

// bf16 [rows, K] (K a multiple of 128) -> E4M3 codes [rows, K] and E8M0
// scales [K / 128][rows][4].
cudaError_t launch_mxfp8_quantize(cudaStream_t s, const void* w, long long rows, int K,
                                  uint8_t* codes, uint8_t* scales);

// bf16 activations [rows, K] (K a multiple of 256) -> MXFP8 codes [rows, K],
// each 256-wide chunk in the small-M W8A8 GEMMs' order (byte 64 t + 8 r + j
// of a chunk: value 32 r + 4 t + (j & 3) + 16 (j >> 2)), and scales
// [rows][K / 32].
cudaError_t launch_act_mxfp8(cudaStream_t s, const void* a, long long rows, int K, uint8_t* codes,
                             uint8_t* scales);

}  // namespace moe
