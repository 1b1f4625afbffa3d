// NVFP4 expert weights ('PagedAttention, speculative decoding, MoE and
// Blackwell', section 3: blocks of 16 values with their own FP8 scale plus
// one FP32 scale for the whole tensor).  Elements are FP4 E2M1 (0, 0.5, 1,
// 1.5, 2, 3, 4, 6 and negatives).  Scales, one tensor = one expert matrix:
// g = amax / (448 * 6) (1 for an all-zero matrix); a block's scale is
// E4M3((amax_block / 6) / g); an element is E2M1(w / (scale * g)), round to
// nearest even, saturating at 6, -0 stored as +0.  Every step is an fp32
// operation with round to nearest, in that order.
//
// Layouts (chosen for the NVFP4 expert GEMMs): codes [rows, K / 2] bytes,
// value 2i of a row in the low nibble of byte i and value 2i + 1 in the high
// nibble; block scales [K / 256][rows][16] bytes, so a 256-wide K stage's 16
// scales of a row are 16 contiguous bytes and a stage's scales for a range of
// weight rows are one contiguous run; tensor scales [groups] fp32.

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp4.h>
#include <cuda_fp8.h>

#include <algorithm>

#include "moe_internal.h"

namespace moe {
namespace {

constexpr float kTensorDiv = 448.0f * 6.0f;

// Largest |w| of each group's matrix, as the bits of a non-negative float
// (ordered like unsigned integers) accumulated with atomicMax into amax_bits,
// which the caller zeroes.
__global__ void __launch_bounds__(256) moe_nvfp4_amax_kernel(const __nv_bfloat16* __restrict__ w,
                                                         long long per_group,
                                                         unsigned* __restrict__ amax_bits) {
  pdl_wait_and_release();
  const int group = blockIdx.y;
  const uint4* src = reinterpret_cast<const uint4*>(w + static_cast<size_t>(group) * per_group);
  const long long n = per_group / 8;  // 8 bf16 per 16-byte load
  float m = 0.0f;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const uint4 r = __ldg(src + i);
    const uint32_t words[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      m = fmaxf(m, fabsf(__uint_as_float(words[j] << 16)));
      m = fmaxf(m, fabsf(__uint_as_float(words[j] & 0xffff0000u)));
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((threadIdx.x & 31) == 0) atomicMax(amax_bits + group, __float_as_uint(m));
}

__device__ __forceinline__ float e4m3_value(uint8_t code) {
  const __half_raw h = __nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(code), __NV_E4M3);
  return __half2float(*reinterpret_cast<const __half*>(&h));
}

// One warp per (row, 256-wide K stage): lane l holds values 8l .. 8l + 7, lanes
// 2b and 2b + 1 one 16-value block.
__global__ void __launch_bounds__(256) moe_nvfp4_quantize_kernel(
    const __nv_bfloat16* __restrict__ w, long long rows_per_group, long long rows, int K,
    const unsigned* __restrict__ amax_bits, uint8_t* __restrict__ codes,
    uint8_t* __restrict__ scales) {
  pdl_wait_and_release();
  const int lane = threadIdx.x & 31;
  const long long stages = K / 256;
  const long long units = rows * stages;
  const long long warps = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
  for (long long u = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
       u < units; u += warps) {
    const long long row = u / stages;
    const int st = static_cast<int>(u - row * stages);
    const float amax_t = __uint_as_float(__ldg(amax_bits + row / rows_per_group));
    const float g = amax_t > 0.0f ? __fdiv_rn(amax_t, kTensorDiv) : 1.0f;
    const uint4 raw = *reinterpret_cast<const uint4*>(
        w + static_cast<size_t>(row) * K + static_cast<size_t>(st) * 256 + lane * 8);
    const uint32_t words[4] = {raw.x, raw.y, raw.z, raw.w};
    float v[8];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      v[2 * j] = __uint_as_float(words[j] << 16);
      v[2 * j + 1] = __uint_as_float(words[j] & 0xffff0000u);
    }
    float amax_b = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) amax_b = fmaxf(amax_b, fabsf(v[i]));
    amax_b = fmaxf(amax_b, __shfl_xor_sync(0xffffffffu, amax_b, 1));
    const float s = __fdiv_rn(__fdiv_rn(amax_b, 6.0f), g);
    const uint8_t s_code = static_cast<uint8_t>(__nv_cvt_float_to_fp8(s, __NV_SATFINITE, __NV_E4M3));
    const float denom = __fmul_rn(e4m3_value(s_code), g);
    uint32_t packed = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float x = denom > 0.0f ? __fdiv_rn(v[i], denom) : 0.0f;
      uint32_t c = static_cast<uint32_t>(__nv_cvt_float_to_fp4(x, __NV_E2M1, cudaRoundNearest)) & 0xfu;
      if ((c & 0x7u) == 0u) c = 0u;  // -0 stored as +0
      packed |= c << (4 * i);
    }
    *reinterpret_cast<uint32_t*>(codes + static_cast<size_t>(row) * (K / 2) +
                                 static_cast<size_t>(st) * 128 + lane * 4) = packed;
    if ((lane & 1) == 0)
      scales[(static_cast<size_t>(st) * rows + row) * 16 + (lane >> 1)] = s_code;
  }
}

// amax bits -> tensor scale, in place.
__global__ void moe_nvfp4_tensor_scale_kernel(unsigned* __restrict__ amax_bits, int groups) {
  pdl_wait_and_release();
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= groups) return;
  const float amax = __uint_as_float(amax_bits[i]);
  reinterpret_cast<float*>(amax_bits)[i] = amax > 0.0f ? __fdiv_rn(amax, kTensorDiv) : 1.0f;
}

}  // namespace

cudaError_t launch_nvfp4_quantize(cudaStream_t s, const void* w, int groups,
                                  long long rows_per_group, int K, uint8_t* codes,
                                  uint8_t* scales, float* tensor_scales) {
  unsigned* amax_bits = reinterpret_cast<unsigned*>(tensor_scales);
  cudaError_t e = cudaMemsetAsync(amax_bits, 0, sizeof(unsigned) * groups, s);
  if (e != cudaSuccess) return e;
  const long long per_group = rows_per_group * K;
  {
    const int blocks = static_cast<int>(std::max(1LL, std::min<long long>(
        (per_group / 8 + 255) / 256, (4LL * device_sm_count() + groups - 1) / groups)));
    KernelScope scope(s, "moe_nvfp4_amax");
    e = launch_kernel(moe_nvfp4_amax_kernel, dim3(blocks, groups), dim3(256), 0, s,
                      static_cast<const __nv_bfloat16*>(w), per_group, amax_bits);
    if (e != cudaSuccess) return e;
  }
  const long long rows = rows_per_group * groups;
  const long long units = rows * (K / 256);
  {
    const long long grid = std::min<long long>((units + 7) / 8, 4LL * device_sm_count() * 8);
    KernelScope scope(s, "moe_nvfp4_quantize");
    e = launch_kernel(moe_nvfp4_quantize_kernel, dim3(static_cast<unsigned>(std::max(1LL, grid))),
                      dim3(256), 0, s, static_cast<const __nv_bfloat16*>(w), rows_per_group, rows,
                      K, static_cast<const unsigned*>(amax_bits), codes, scales);
    if (e != cudaSuccess) return e;
  }
  KernelScope scope(s, "moe_nvfp4_tensor_scale");
  return launch_kernel(moe_nvfp4_tensor_scale_kernel, dim3((groups + 255) / 256), dim3(256), 0, s,
                       amax_bits, groups);
}

}  // namespace moe
