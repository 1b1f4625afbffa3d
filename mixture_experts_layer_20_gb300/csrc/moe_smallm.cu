// Small-M expert GEMMs: the grouped SwiGLU FFN when experts receive few token
// rows (decode batches), for MXFP8 and NVFP4 expert weights.
//
// At decode every active expert sees a handful of tokens, so the layer is
// bound by streaming the expert weights from HBM ('Hosting Qwen on
// Blackwell', "Decoders"; 'Chapter 9. Distributed inference', section 9.3.3:
// 64 tokens x top-8 touch ~126 of 128 experts).  Here each warp owns 16
// weight rows of one expert over the whole reduction and multiplies them by
// that expert's tokens with warp-level tensor-core MMAs (mma.sync m16n8k16,
// bf16 in, fp32 accumulate): every warp issues its own MMAs, so nothing
// serialises on one issuing thread, and the quantised weights are decoded to
// bf16 in registers right before their MMA.  No reduction over K is split,
// so every output is one fixed-order fp32 sum.
//
//   gate_up : a warp's 16 rows are gate rows c0..c0+7 of the expert and the
//             matching up rows, so the accumulator fragment of each lane holds
//             gate and up of the same h column and token: h = silu(g) * u is
//             formed in registers and stored as bf16.
//   down    : 16 consecutive rows of W_down (16 y columns); y stored in fp16
//             with the same range rule as the large-M kernels.
//
// The reduction is consumed in chunks of 256 values.  Lane (g, t) of a warp
// (g = lane / 4, t = lane % 4) loads 16-byte units of its rows g and g + 8 at
// byte offsets 64 i + 16 t of the row's chunk, so four lanes read 64
// contiguous bytes of a row per instruction.  A unit holds V values (16 E4M3
// or 32 E2M1 codes) at reduction indices V (4 i + t) + [0, V).  MXFP8: the
// MMA whose fragment k-positions {2t, 2t+1, 2t+8, 2t+9} stand for indices
// V (4 i + t) + 4 j + {0, 1, 2, 3} takes the same indices of the tokens.
// NVFP4: the two MMAs of 32-bit word m of a unit stand for V (4 i + t) +
// 8 m + {0, 4, 1, 5} and {2, 6, 3, 7}: codes 16 bits apart share a bf16 pair,
// so one shift places both (e2m1x8_to_bf16_pairs), and one byte permute per
// pair pairs the token values alike.  Either way a fixed permutation of the
// reduction, applied to both operands, leaves the sum unchanged.
//
// Decoding E2M1 codes bounds the NVFP4 kernels (integer and bf16 multiply
// pipes, not HBM): the codes' magnitude bits go straight into bf16 exponent
// and mantissa fields (the weight times 2^-8 after the block-scale multiply;
// the fp32 sums are multiplied by 2^8 with the tensor scale), so a code costs
// about two instructions.
//
// W8A8 (MXFP8 weights and MXFP8 token rows, an option of the MXFP8 layer):
// the tokens are quantised like the weights (launch_act_mxfp8: x before
// gate_up, h before down), and each 32-value run is one mma.sync m16n8k32
// E4M3 x E4M3 -> fp32 with no accumulator input, whose four sums the lane
// scales by the runs' weight and token scales (exact powers of two) and adds
// to its fp32 accumulators in run order.  No code is decoded: the codes go
// from shared memory (weights) and global memory (tokens) into the MMA.
//
// Weights (and their block scales) reach shared memory through a per-warp
// ring of cp.async copies several chunks ahead, across task boundaries; each
// lane copies and later reads only its own units, so a lane's own
// cp.async.wait_group is all the synchronisation the ring needs.  Token rows
// are read straight from global memory (they are shared by the CTA's warps,
// which work on the same expert, and stay in L1 / L2).

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>
#include <mutex>

#include "moe_internal.h"
#include "moe_smallm.cuh"

namespace moe {
namespace {

template <int FMT, int KIND>
__global__ void __launch_bounds__(kSmThreads, 2) moe_smallm_kernel(const SmParams p) {
  extern __shared__ __align__(16) uint8_t sm_raw[];
  pdl_wait_and_release();
  sm_phase<FMT, KIND>(p, sm_raw);
}

typedef void (*SmKernel)(const SmParams);

template <int FMT, int KIND>
cudaError_t sm_launch(cudaStream_t s, const char* name, const SmParams& p) {
  SmKernel k = moe_smallm_kernel<FMT, KIND>;
  constexpr int smem = sm_smem_bytes<FMT>();
  static std::once_flag once[64];
  static cudaError_t attr_err[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::call_once(once[dev], [&] {
    attr_err[dev] = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  });
  if (attr_err[dev] != cudaSuccess) return attr_err[dev];
  KernelScope scope(s, name);
  return launch_kernel(k, dim3(2 * device_sm_count()), dim3(kSmThreads), smem, s, p);
}

template <int FMT>
cudaError_t sm_ffn(cudaStream_t s, const char* gu_name, const char* dn_name, const void* a,
                   const int32_t* perm, int div, const int32_t* offsets, int rows, int d, int E,
                   int I, const uint8_t* w_gate_up, const uint8_t* s_gate_up,
                   const float* t_gate_up, const uint8_t* w_down, const uint8_t* s_down,
                   const float* t_down, void* h, void* y, unsigned* status, bool y_fp32) {
  using F = SmF<FMT>;
  if (d % sm_chunk_k<FMT>() || I % sm_chunk_k<FMT>()) return cudaErrorInvalidValue;
  SmParams p{};
  p.w = w_gate_up;
  p.scales = s_gate_up;
  p.tscale = t_gate_up;
  p.scale_rows = 2LL * I * E;
  p.row_bytes = static_cast<long long>(d) * F::kBytesX2 / 2;
  p.K = d;
  p.n_out = I;
  p.w_rows_per_expert = 2 * I;
  p.up_offset = I;
  p.E = E;
  p.offsets = offsets;
  p.total_rows = rows;
  p.b = static_cast<const __nv_bfloat16*>(a);
  p.b_rows = perm ? (rows + div - 1) / div : rows;
  p.perm = perm;
  p.div = div;
  p.out = h;
  p.ld_out = I;
  p.status = status;
  cudaError_t e = sm_launch<FMT, kSmGateUp>(s, gu_name, p);
  if (e != cudaSuccess) return e;
  SmParams q = p;
  q.w = w_down;
  q.scales = s_down;
  q.tscale = t_down;
  q.scale_rows = static_cast<long long>(E) * d;
  q.row_bytes = static_cast<long long>(I) * F::kBytesX2 / 2;
  q.K = I;
  q.n_out = d;
  q.w_rows_per_expert = d;
  q.up_offset = 0;
  q.b = static_cast<const __nv_bfloat16*>(h);
  q.b_rows = rows;
  q.perm = nullptr;
  q.div = 1;
  q.out = y;
  q.ld_out = d;
  q.y_fp32 = y_fp32 ? 1 : 0;
  return sm_launch<FMT, kSmDown>(s, dn_name, q);
}

// W8A8: x (the T unpermuted tokens) and then h quantised to MXFP8 by
// launch_act_mxfp8, each GEMM reading the codes with fp8 warp MMAs.
cudaError_t sm_ffn_a8(cudaStream_t s, const void* x, int T, const int32_t* perm, int div,
                      const int32_t* offsets, int rows, int d, int E, int I,
                      const uint8_t* w_gate_up, const uint8_t* s_gate_up, const uint8_t* w_down,
                      const uint8_t* s_down, uint8_t* xq, uint8_t* xs, void* h, uint8_t* hq,
                      uint8_t* hs, void* y, unsigned* status, bool y_fp32) {
  constexpr int F = kSmMx8A8;
  if (d % sm_chunk_k<F>() || I % sm_chunk_k<F>()) return cudaErrorInvalidValue;
  cudaError_t e = launch_act_mxfp8(s, x, T, d, xq, xs);
  if (e != cudaSuccess) return e;
  SmParams p{};
  p.w = w_gate_up;
  p.scales = s_gate_up;
  p.scale_rows = 2LL * I * E;
  p.row_bytes = d;
  p.K = d;
  p.n_out = I;
  p.w_rows_per_expert = 2 * I;
  p.up_offset = I;
  p.E = E;
  p.offsets = offsets;
  p.total_rows = rows;
  p.bq = xq;
  p.bs = xs;
  p.b_rows = T;
  p.perm = perm;
  p.div = div;
  p.out = h;
  p.ld_out = I;
  p.status = status;
  e = sm_launch<F, kSmGateUp>(s, "moe_gate_up_swiglu_mxfp8_a8_smallm", p);
  if (e == cudaSuccess) e = launch_act_mxfp8(s, h, rows, I, hq, hs);
  if (e != cudaSuccess) return e;
  SmParams q = p;
  q.w = w_down;
  q.scales = s_down;
  q.scale_rows = static_cast<long long>(E) * d;
  q.row_bytes = I;
  q.K = I;
  q.n_out = d;
  q.w_rows_per_expert = d;
  q.up_offset = 0;
  q.bq = hq;
  q.bs = hs;
  q.b_rows = rows;
  q.perm = nullptr;
  q.div = 1;
  q.out = y;
  q.ld_out = d;
  q.y_fp32 = y_fp32 ? 1 : 0;
  return sm_launch<F, kSmDown>(s, "moe_down_mxfp8_a8_smallm", q);
}

}  // namespace

cudaError_t launch_grouped_ffn_smallm_a8(cudaStream_t s, const void* x, int T,
                                         const int32_t* perm, int div, const int32_t* offsets,
                                         int rows, int d, int E, int I, const void* w_gate_up,
                                         const uint8_t* scales_gate_up, const void* w_down,
                                         const uint8_t* scales_down, uint8_t* xq, uint8_t* xs,
                                         void* h, uint8_t* hq, uint8_t* hs, void* y,
                                         unsigned* status, bool y_fp32) {
  if (E > kMaxExperts) return cudaErrorInvalidValue;
  return sm_ffn_a8(s, x, T, perm, div, offsets, rows, d, E, I,
                   static_cast<const uint8_t*>(w_gate_up), scales_gate_up,
                   static_cast<const uint8_t*>(w_down), scales_down, xq, xs, h, hq, hs, y, status,
                   y_fp32);
}

cudaError_t launch_grouped_ffn_smallm(cudaStream_t s, int fmt, const void* a,
                                      const int32_t* perm, int div, const int32_t* offsets,
                                      int rows, int d, int E, int I, const void* w_gate_up,
                                      const uint8_t* scales_gate_up, const float* tscale_gate_up,
                                      const void* w_down, const uint8_t* scales_down,
                                      const float* tscale_down, void* h, void* y,
                                      unsigned* status, bool y_fp32) {
  if (E > kMaxExperts) return cudaErrorInvalidValue;
  const uint8_t* wg = static_cast<const uint8_t*>(w_gate_up);
  const uint8_t* wd = static_cast<const uint8_t*>(w_down);
  switch (fmt) {
    case 1:
      return sm_ffn<kSmMx8>(s, "moe_gate_up_swiglu_mxfp8_smallm", "moe_down_mxfp8_smallm", a,
                            perm, div, offsets, rows, d, E, I, wg, scales_gate_up, nullptr, wd,
                            scales_down, nullptr, h, y, status, y_fp32);
    case 2:
      return sm_ffn<kSmNv4>(s, "moe_gate_up_swiglu_nvfp4_smallm", "moe_down_nvfp4_smallm", a,
                            perm, div, offsets, rows, d, E, I, wg, scales_gate_up, tscale_gate_up,
                            wd, scales_down, tscale_down, h, y, status, y_fp32);
  }
  return cudaErrorInvalidValue;
}

}  // namespace moe
