// Conversions of quantised weight codes to bf16 on sm_103a: E4M3 (MXFP8
// elements), E2M1 (NVFP4 elements) and their block scales.  Every product
// formed here is exact in bf16: an E4M3 code has 4 significant bits, an E2M1
// code 2, and the scales are powers of two (E8M0) or 4-bit values (E4M3).
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

namespace moe {

// 2^(byte - 127) as a float (byte 0: 2^-127, a subnormal).
__device__ __forceinline__ float e8m0_to_float(uint32_t byte) {
  return byte ? __uint_as_float(byte << 23) : __uint_as_float(0x00400000u);
}

// 4 E4M3 codes (a 32-bit word, lowest byte first) times 2^(S - 127) as two
// bf16x2, by bits: a code's seven magnitude bits placed at bf16 bit 4 and its
// sign at bit 15 form the bf16 (normal, or subnormal for a subnormal code)
// whose value is the code's times 2^-120; one exact bf16x2 multiply by
// mul = 2^(S - 7) applies the scale.  Valid while 2^(S - 7) is a finite bf16
// (S <= 134); larger scales take e4m3x8_to_bf16.  The byte permute
// sign-extends each code to 16 bits (prmt selector nibbles with bit 3 set
// replicate the selected byte's sign), so one shift moves the magnitude to
// bits 4-10 and a sign copy to bit 15, and one mask clears the rest.
__device__ __forceinline__ void e4m3x4_to_bf16_bits(uint32_t w, __nv_bfloat162 mul,
                                                    uint32_t* out) {
  uint32_t a, b;
  asm("prmt.b32 %0, %1, 0, 0x9180;" : "=r"(a) : "r"(w));  // sext16(code 0) | sext16(code 1) << 16
  asm("prmt.b32 %0, %1, 0, 0xB3A2;" : "=r"(b) : "r"(w));  // codes 2 and 3
  a = (a << 4) & 0x87F087F0u;
  b = (b << 4) & 0x87F087F0u;
  const __nv_bfloat162 pa = __hmul2(*reinterpret_cast<const __nv_bfloat162*>(&a), mul);
  const __nv_bfloat162 pb = __hmul2(*reinterpret_cast<const __nv_bfloat162*>(&b), mul);
  out[0] = *reinterpret_cast<const uint32_t*>(&pa);
  out[1] = *reinterpret_cast<const uint32_t*>(&pb);
}

// 8 E4M3 codes (a 64-bit word, lowest byte first) times `scale` as 4 bf16x2,
// through the hardware conversions (any scale).
__device__ __forceinline__ void e4m3x8_to_bf16(uint32_t lo, uint32_t hi, float scale,
                                               uint32_t* out) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t w = i < 2 ? lo : hi;
    const __nv_fp8x2_storage_t two =
        static_cast<__nv_fp8x2_storage_t>((w >> (16 * (i & 1))) & 0xffffu);
    const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(two, __NV_E4M3);
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h));
    const __nv_bfloat162 b = __floats2bfloat162_rn(f.x * scale, f.y * scale);
    out[i] = *reinterpret_cast<const uint32_t*>(&b);
  }
}

// 4 E4M3 codes (a 32-bit word, lowest byte first) times `scale` as two
// bf16x2, through the hardware conversions (any scale).
__device__ __forceinline__ void e4m3x4_to_bf16_scaled(uint32_t w, float scale, uint32_t* out) {
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const __nv_fp8x2_storage_t two = static_cast<__nv_fp8x2_storage_t>((w >> (16 * i)) & 0xffffu);
    const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(two, __NV_E4M3);
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h));
    const __nv_bfloat162 b = __floats2bfloat162_rn(f.x * scale, f.y * scale);
    out[i] = *reinterpret_cast<const uint32_t*>(&b);
  }
}

// 4 E2M1 codes (the low 16 bits of w, code i in bits 4i .. 4i + 3) as two
// bf16x2 of code value x scale.  The codes' 3-bit magnitudes index byte
// tables of the bf16 patterns of 0, 0.5, 1, 1.5, 2, 3, 4, 6 with prmt (high
// bytes 00 3F 3F 3F 40 40 40 40, low bytes 00 00 80 C0 00 40 80 C0), two more
// prmt interleave them into bf16 halves, and one exact bf16x2 multiply
// applies the block scale.  Signs: code 2i + 1's sign bit is bit 7 of byte i
// of w and code 2i's is bit 7 of byte i of w << 4, so one sign-replicating
// byte select per pair (selector nibbles 8 | byte) lays them over bits 15
// and 31, and one masked or merges them.
__device__ __forceinline__ void e2m1x4_to_bf16(uint32_t w, __nv_bfloat162 mul, uint32_t* out) {
  const uint32_t sel = w & 0x7777u;
  uint32_t hi, lo, a, b, sa, sb;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(hi) : "r"(0x3F3F3F00u), "r"(0x40404040u), "r"(sel));
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(lo) : "r"(0xC0800000u), "r"(0xC0804000u), "r"(sel));
  asm("prmt.b32 %0, %1, %2, 0x5140;" : "=r"(a) : "r"(lo), "r"(hi));  // values 0, 1
  asm("prmt.b32 %0, %1, %2, 0x7362;" : "=r"(b) : "r"(lo), "r"(hi));  // values 2, 3
  const uint32_t w4 = w << 4;
  asm("prmt.b32 %0, %1, %2, 0xC080;" : "=r"(sa) : "r"(w4), "r"(w));  // signs of codes 0, 1
  asm("prmt.b32 %0, %1, %2, 0xD090;" : "=r"(sb) : "r"(w4), "r"(w));  // signs of codes 2, 3
  a |= sa & 0x80008000u;
  b |= sb & 0x80008000u;
  const __nv_bfloat162 pa = __hmul2(*reinterpret_cast<const __nv_bfloat162*>(&a), mul);
  const __nv_bfloat162 pb = __hmul2(*reinterpret_cast<const __nv_bfloat162*>(&b), mul);
  out[0] = *reinterpret_cast<const uint32_t*>(&pa);
  out[1] = *reinterpret_cast<const uint32_t*>(&pb);
}

// 8 E2M1 codes (a 32-bit word, code q in bits 4q .. 4q + 3) as four bf16x2
// pairs, out[q] = (code q, code q + 4) x mul for q = 0..3: the two codes of a
// pair lie 16 bits apart, so one shift places both.  A code's magnitude bits
// e1 e0 m placed at bf16 bits 8..6 form the bf16 with exponent field e1 e0 and
// mantissa m/2: 2^(e - 127) (1 + m/2) for e > 0 and 2^-126 m/2 (a subnormal)
// for e = 0, i.e. the code's value times 2^-126; its sign goes to bit 15.
// mul is the block scale times 2^118 (e4m3_scale_x2p118), so the products are
// the weights times 2^-8, exact in bf16 (at most 6 significant bits, and
// normal); the caller multiplies its fp32 sums by 2^8.  Ten integer-pipe
// operations (masks, two right shifts), five left shifts that may run as
// integer multiply-adds, and four bf16x2 multiplies per eight codes.
__device__ __forceinline__ void e2m1x8_to_bf16_pairs(uint32_t x, __nv_bfloat162 mul,
                                                     uint32_t* out) {
  uint32_t r[4];
  r[0] = ((x << 6) & 0x01C001C0u) | ((x << 12) & 0x80008000u);  // codes 0, 4
  r[1] = ((x << 2) & 0x01C001C0u) | ((x << 8) & 0x80008000u);   // codes 1, 5
  r[2] = ((x >> 2) & 0x01C001C0u) | ((x << 4) & 0x80008000u);   // codes 2, 6
  r[3] = ((x >> 6) & 0x01C001C0u) | (x & 0x80008000u);          // codes 3, 7
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const __nv_bfloat162 v = __hmul2(*reinterpret_cast<const __nv_bfloat162*>(&r[q]), mul);
    out[q] = *reinterpret_cast<const uint32_t*>(&v);
  }
}

// Byte b (0..3) of an E4M3 scale word as a bf16 pair of value x 2^118, for
// e2m1x8_to_bf16_pairs.  sel = e4m3_scale_sel(b).  The byte, sign-extended
// into both halves by one byte permute and shifted so that its seven
// magnitude bits sit at bf16 bits 10..4, is the bf16 of value x 2^-120
// (normal, or subnormal for a subnormal code; the trick of
// e4m3x4_to_bf16_bits); two exact multiplies by 2^119 give value x 2^118,
// finite for every finite E4M3 value (at most 448 x 2^118 < 2^127).
__host__ __device__ constexpr uint32_t e4m3_scale_sel(uint32_t b) {
  return b | ((b | 8u) << 4) | (b << 8) | ((b | 8u) << 12);
}
__device__ __forceinline__ __nv_bfloat162 e4m3_scale_x2p118(uint32_t word, uint32_t sel) {
  uint32_t t;
  asm("prmt.b32 %0, %1, 0, %2;" : "=r"(t) : "r"(word), "r"(sel));
  t = (t << 4) & 0x87F087F0u;
  const uint32_t k2p119 = 0x7B007B00u;  // bf16 2^119 in both halves
  const __nv_bfloat162 c = *reinterpret_cast<const __nv_bfloat162*>(&k2p119);
  return __hmul2(__hmul2(*reinterpret_cast<const __nv_bfloat162*>(&t), c), c);
}

// An E4M3 block scale as a bf16 pair (exact: 4 significant bits).
__device__ __forceinline__ __nv_bfloat162 e4m3_scale_bf16x2(uint32_t code) {
  const __half_raw h = __nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(code), __NV_E4M3);
  const float f = __half2float(*reinterpret_cast<const __half*>(&h));
  return __floats2bfloat162_rn(f, f);
}

}  // namespace moe
