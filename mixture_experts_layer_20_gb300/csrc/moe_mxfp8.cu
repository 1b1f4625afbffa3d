// MXFP8 expert weights ('Hosting Qwen on Blackwell', "Quantization": the
// weights are converted to MXFP8 statically after training).  MXFP8 is the
// OCP microscaling format with FP8 E4M3 elements: each run of 32 consecutive
// values along K shares one power-of-two scale, an E8M0 byte X + 127 with
// X = floor(log2(max |v|)) - 8 (the run's largest magnitude lands in E4M3's
// top binade); elements are v / 2^X rounded to nearest even and clamped to
// +-448.  An all-zero run stores the byte 0.
//
// Layouts (chosen for the MXFP8 expert GEMMs): codes [rows, K] uint8, the
// same row-major order as the bf16 matrix; scales [K / 128][rows][4] uint8,
// so the four scales of one 128-wide K block of a row are one 32-bit word and
// a pipeline stage's scales for a contiguous range of weight rows are one
// contiguous run.

#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include <algorithm>

#include "moe_internal.h"

namespace moe {
namespace {

// One warp per (row, 128-wide K block): lane l holds elements 4l .. 4l + 3,
// lanes 8j .. 8j + 7 one 32-value run.
__global__ void __launch_bounds__(256) moe_mxfp8_quantize_kernel(const __nv_bfloat16* __restrict__ w,
                                                             long long rows, int K,
                                                             uint8_t* __restrict__ codes,
                                                             uint8_t* __restrict__ scales) {
  pdl_wait_and_release();
  const int lane = threadIdx.x & 31;
  const long long kblocks = K / 128;
  const long long units = rows * kblocks;
  const long long warps = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
  for (long long u = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
       u < units; u += warps) {
    const long long row = u / kblocks;
    const int kb = static_cast<int>(u - row * kblocks);
    const size_t off = static_cast<size_t>(row) * K + static_cast<size_t>(kb) * 128 + lane * 4;
    const uint2 raw = *reinterpret_cast<const uint2*>(w + off);
    float v[4];
    v[0] = __uint_as_float(raw.x << 16);
    v[1] = __uint_as_float(raw.x & 0xffff0000u);
    v[2] = __uint_as_float(raw.y << 16);
    v[3] = __uint_as_float(raw.y & 0xffff0000u);
    float amax = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    int byte = 0;
    if (amax > 0.0f) byte = min(254, max(0, ilogbf(amax) - 8 + 127));
    const int x = byte - 127;
    const __nv_fp8x2_storage_t lo =
        __nv_cvt_float2_to_fp8x2(make_float2(ldexpf(v[0], -x), ldexpf(v[1], -x)), __NV_SATFINITE,
                                 __NV_E4M3);
    const __nv_fp8x2_storage_t hi =
        __nv_cvt_float2_to_fp8x2(make_float2(ldexpf(v[2], -x), ldexpf(v[3], -x)), __NV_SATFINITE,
                                 __NV_E4M3);
    uint32_t packed = static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
    // -0 encodes as +0 (the value is the same)
#pragma unroll
    for (int b = 0; b < 4; ++b)
      if (((packed >> (8 * b)) & 0xffu) == 0x80u) packed &= ~(0xffu << (8 * b));
    *reinterpret_cast<uint32_t*>(codes + off) = packed;
    // the four run scales of this K block, one byte each, from lanes 0, 8, 16, 24
    const int b1 = __shfl_sync(0xffffffffu, byte, 8);
    const int b2 = __shfl_sync(0xffffffffu, byte, 16);
    const int b3 = __shfl_sync(0xffffffffu, byte, 24);
    if (lane == 0)
      *reinterpret_cast<uint32_t*>(scales + (static_cast<size_t>(kb) * rows + row) * 4) =
          static_cast<uint32_t>(byte) | (static_cast<uint32_t>(b1) << 8) |
          (static_cast<uint32_t>(b2) << 16) | (static_cast<uint32_t>(b3) << 24);
  }
}

// Activations: the same format per run of 32 along K, for the W8A8 small-M
// GEMMs.  One warp per (row, 256-wide chunk): lane l holds values 8 l ..
// 8 l + 7 of the chunk (run r = l / 4).  Byte 64 t + 8 r + j of the chunk
// holds value 32 r + 4 t + (j & 3) + 16 (j >> 2): lane t of a small-M warp
// reads its eight bytes of all eight runs as 64 contiguous bytes, values
// 4 t .. 4 t + 3 and 16 + 4 t .. 16 + 4 t + 3 of each run (its MMA
// fragment).  Scales [rows][K / 32], one byte per run in order.
__global__ void __launch_bounds__(256) moe_act_mxfp8_kernel(const __nv_bfloat16* __restrict__ a,
                                                            long long rows, int K,
                                                            uint8_t* __restrict__ codes,
                                                            uint8_t* __restrict__ scales) {
  pdl_wait_and_release();
  const int lane = threadIdx.x & 31;
  const long long chunks = K / 256;
  const long long units = rows * chunks;
  const long long warps = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
  for (long long u = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
       u < units; u += warps) {
    const long long row = u / chunks;
    const int c = static_cast<int>(u - row * chunks);
    const size_t base = static_cast<size_t>(row) * K + static_cast<size_t>(c) * 256;
    const uint4 raw = *reinterpret_cast<const uint4*>(a + base + lane * 8);
    float v[8];
    const uint32_t wv[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      v[2 * i] = __uint_as_float(wv[i] << 16);
      v[2 * i + 1] = __uint_as_float(wv[i] & 0xffff0000u);
    }
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(v[i]));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    int byte = 0;
    if (amax > 0.0f) byte = min(254, max(0, ilogbf(amax) - 8 + 127));
    const int x = byte - 127;
    uint32_t packed[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const __nv_fp8x2_storage_t lo = __nv_cvt_float2_to_fp8x2(
          make_float2(ldexpf(v[4 * h], -x), ldexpf(v[4 * h + 1], -x)), __NV_SATFINITE, __NV_E4M3);
      const __nv_fp8x2_storage_t hi = __nv_cvt_float2_to_fp8x2(
          make_float2(ldexpf(v[4 * h + 2], -x), ldexpf(v[4 * h + 3], -x)), __NV_SATFINITE,
          __NV_E4M3);
      uint32_t w = static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
#pragma unroll
      for (int b = 0; b < 4; ++b)  // -0 encodes as +0 (the value is the same)
        if (((w >> (8 * b)) & 0xffu) == 0x80u) w &= ~(0xffu << (8 * b));
      packed[h] = w;
    }
    // values 8 q + m of run r (q = lane % 4): m = 0..3 go to t = 2 (q % 2),
    // m = 4..7 to t + 1, at byte 4 (q / 2) of the lane's 8 bytes of the run
    const int run = lane >> 2, q = lane & 3;
    const int t0 = 2 * (q & 1), j0 = 4 * (q >> 1);
    *reinterpret_cast<uint32_t*>(codes + base + 64 * t0 + 8 * run + j0) = packed[0];
    *reinterpret_cast<uint32_t*>(codes + base + 64 * (t0 + 1) + 8 * run + j0) = packed[1];
    if (q == 0) scales[static_cast<size_t>(row) * (K / 32) + c * 8 + run] = static_cast<uint8_t>(byte);
  }
}

}  // namespace

cudaError_t launch_act_mxfp8(cudaStream_t s, const void* a, long long rows, int K, uint8_t* codes,
                             uint8_t* scales) {
  if (K % 256) return cudaErrorInvalidValue;
  const long long units = rows * (K / 256);
  const long long grid = std::min<long long>((units + 7) / 8, 4LL * device_sm_count() * 8);
  KernelScope scope(s, "moe_act_mxfp8");
  return launch_kernel(moe_act_mxfp8_kernel, dim3(static_cast<unsigned>(std::max(1LL, grid))),
                       dim3(256), 0, s, static_cast<const __nv_bfloat16*>(a), rows, K, codes,
                       scales);
}

cudaError_t launch_mxfp8_quantize(cudaStream_t s, const void* w, long long rows, int K,
                                  uint8_t* codes, uint8_t* scales) {
  const long long units = rows * (K / 128);
  const long long grid = std::min<long long>((units + 7) / 8, 4LL * device_sm_count() * 8);
  KernelScope scope(s, "moe_mxfp8_quantize");
  return launch_kernel(moe_mxfp8_quantize_kernel, dim3(static_cast<unsigned>(std::max(1LL, grid))),
                       dim3(256), 0, s, static_cast<const __nv_bfloat16*>(w), rows, K, codes,
                       scales);
}

}  // namespace moe
