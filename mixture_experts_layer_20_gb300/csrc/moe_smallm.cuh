// Warp-level small-M expert GEMM (mma.sync m16n8k16) for the decode case of
// the grouped SwiGLU FFN: the device code shared by the standalone small-M
// kernels (moe_smallm.cu) and the single-launch decode kernel.  The design is
// described at the top of moe_smallm.cu.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "moe_convert.cuh"
#include "moe_internal.h"

namespace moe {

enum SmFmt : int { kSmBf16 = 0, kSmMx8 = 1, kSmNv4 = 2 };
enum SmKind : int { kSmGateUp = 1, kSmDown = 2 };

constexpr int kSmWarps = 8;               // warps per CTA
constexpr int kSmThreads = kSmWarps * 32;
constexpr int kSmChunkK = 128;            // reduction values per pipeline step
constexpr int kSmNT = 2;                  // 8-token MMA tiles per pass: 16 tokens
constexpr int kSmTokPass = 8 * kSmNT;
constexpr int kSmScaleSlot = 16;          // bytes of block scales per lane per stage
constexpr float kSmHalfMax = 65504.0f;

// V: values per 16-byte unit; U: units per lane and row per chunk; NS: ring
// stages; SB: scale bytes per weight row per chunk (copied per lane).
template <int FMT> struct SmF;
template <> struct SmF<kSmBf16> {
  static constexpr int V = 8, U = 4, NS = 3, SB = 0, kValBytesX2 = 4;  // 2 bytes / value
};
template <> struct SmF<kSmMx8> {
  static constexpr int V = 16, U = 2, NS = 5, SB = 4, kValBytesX2 = 2;  // 1 byte / value
};
template <> struct SmF<kSmNv4> {
  static constexpr int V = 32, U = 1, NS = 8, SB = 8, kValBytesX2 = 1;  // half a byte / value
};

template <int FMT>
__host__ __device__ constexpr int sm_stage_bytes() {
  return 2 * SmF<FMT>::U * 32 * 16 + (SmF<FMT>::SB ? 32 * kSmScaleSlot : 0);
}
template <int FMT>
__host__ __device__ constexpr int sm_smem_bytes() {
  return kSmWarps * SmF<FMT>::NS * sm_stage_bytes<FMT>();
}

struct SmParams {
  const uint8_t* w;          // weight rows (bf16 values or codes), row_bytes each
  const uint8_t* scales;     // MXFP8 [K/128][scale_rows][4], NVFP4 [K/256][scale_rows][16]
  const float* tscale;       // NVFP4: one scale per expert (null: none)
  long long scale_rows;      // weight rows of the whole tensor
  long long row_bytes;
  int K;                     // reduction length (a multiple of 128)
  int n_out;                 // gate_up: I (h columns); down: d (y columns)
  int w_rows_per_expert;     // 2I or d
  int up_offset;             // gate_up: I
  int E;
  const int32_t* offsets;    // [E + 1] token row offsets of the grouped layout
  int total_rows;
  const __nv_bfloat16* b;    // token rows [b_rows, K]
  int b_rows;
  const int32_t* perm;       // gate_up at decode: B row of slot pos = perm[pos] / div
  int div;
  void* out;                 // gate_up: h bf16 [rows, I]; down: y fp16 [rows, d]
  int ld_out;
  unsigned* status;
};

__device__ __forceinline__ void cp_async_16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_8(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_4(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}

// D (+)= A B with A 16 x 16 bf16 (row-major fragment), B 16 x 8 bf16
// (column-major fragment), D 16 x 8 fp32.
__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t word_of(const uint4& v, int i) {
  return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

// One task: 16 weight rows of one expert (see the file comment) over the
// whole reduction, for all of the expert's tokens (passes of 16).
struct SmTask {
  int e, m, row_off;      // expert, its token rows, first row in the grouped layout
  long long r0, r1;       // weight rows of fragment rows g and g + 8 (this lane)
  int col;                // gate_up: h column c0 + g; down: y column r0 + g
  int npass;
};

template <int KIND>
__device__ __forceinline__ SmTask sm_task(const SmParams& p, const int* s_act, const int* s_off,
                                          int tau, int tpe, int g) {
  SmTask t;
  const int a = tau / tpe;
  const int cg = tau - a * tpe;
  t.e = s_act[a];
  t.row_off = s_off[t.e];
  t.m = s_off[t.e + 1] - t.row_off;
  t.npass = (t.m + kSmTokPass - 1) / kSmTokPass;
  const long long base = static_cast<long long>(t.e) * p.w_rows_per_expert;
  if (KIND == kSmGateUp) {
    t.col = cg * 8 + g;
    t.r0 = base + t.col;
    t.r1 = t.r0 + p.up_offset;
  } else {
    t.col = cg * 16 + g;
    t.r0 = base + t.col;
    t.r1 = t.r0 + 8;
  }
  return t;
}

// Copies of one chunk of a task's weights (and scales) into ring slot `slot`.
template <int FMT>
__device__ __forceinline__ void sm_fetch(const SmParams& p, const SmTask& t, int c, uint32_t slot,
                                         int lane, int tig) {
  using F = SmF<FMT>;
  constexpr int kChunkBytes = kSmChunkK * F::kValBytesX2 / 2;
  const uint8_t* rows[2] = {p.w + t.r0 * p.row_bytes + static_cast<long long>(c) * kChunkBytes,
                            p.w + t.r1 * p.row_bytes + static_cast<long long>(c) * kChunkBytes};
#pragma unroll
  for (int rr = 0; rr < 2; ++rr)
#pragma unroll
    for (int i = 0; i < F::U; ++i)
      cp_async_16(slot + ((rr * F::U + i) * 32 + lane) * 16, rows[rr] + 64 * i + 16 * tig);
  if constexpr (FMT == kSmMx8) {
    const uint32_t s = slot + 2 * F::U * 32 * 16 + lane * kSmScaleSlot;
    const uint8_t* base = p.scales + static_cast<long long>(c) * p.scale_rows * 4;
    cp_async_4(s, base + t.r0 * 4);
    cp_async_4(s + 4, base + t.r1 * 4);
  } else if constexpr (FMT == kSmNv4) {
    const uint32_t s = slot + 2 * F::U * 32 * 16 + lane * kSmScaleSlot;
    const uint8_t* base =
        p.scales + static_cast<long long>(c >> 1) * p.scale_rows * 16 + 8 * (c & 1);
    cp_async_8(s, base + t.r0 * 16);
    cp_async_8(s + 8, base + t.r1 * 16);
  }
}

// One grouped GEMM (gate_up or down) by all warps of the grid.  ring: the
// block's dynamic shared memory (sm_smem_bytes<FMT>()).  COHERENT: the offsets,
// the permutation and (down) the token rows h were written by this kernel
// before a grid-wide barrier (see ld_in).  Ends with every copy landed and a
// block-wide barrier.
template <int FMT, int KIND, bool COHERENT = false>
__device__ __forceinline__ void sm_phase(const SmParams& p, uint8_t* sm_raw) {
  using F = SmF<FMT>;
  constexpr bool kBCoherent = COHERENT && KIND == kSmDown;  // h rows; x is an input
  __shared__ int s_off[kMaxExperts + 1];
  __shared__ int s_act[kMaxExperts];
  __shared__ int s_wcount[kSmWarps];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int g = lane >> 2, tig = lane & 3;

  // Active experts in expert order (the offsets come from the grouping step).
  const int E = p.E;
  for (int i = threadIdx.x; i <= E; i += kSmThreads) s_off[i] = ld_in<COHERENT>(p.offsets + i);
  __syncthreads();
  const int ex = threadIdx.x;  // kSmThreads >= kMaxExperts: one expert per thread
  const int mex = ex < E ? s_off[ex + 1] - s_off[ex] : 0;
  bool bad = mex < 0 || (ex == 0 && (s_off[0] != 0 || s_off[E] != p.total_rows));
  const unsigned ball = __ballot_sync(0xffffffffu, mex > 0);
  if (lane == 0) s_wcount[warp] = __popc(ball);
  bad = __syncthreads_or(bad);
  int before = 0, n_act = 0;
#pragma unroll
  for (int w = 0; w < kSmWarps; ++w) {
    before += w < warp ? s_wcount[w] : 0;
    n_act += s_wcount[w];
  }
  if (mex > 0) s_act[before + __popc(ball & ((1u << lane) - 1u))] = ex;
  __syncthreads();
  if (bad) {
    if (threadIdx.x == 0 && blockIdx.x == 0) atomicOr(p.status, kStatusDeviceCheck);
    return;  // uniform across the block
  }

  const int tpe = KIND == kSmGateUp ? p.n_out / 8 : p.n_out / 16;  // tasks per expert
  const int total = n_act * tpe;
  const int W = gridDim.x * kSmWarps;
  const int nch = p.K / kSmChunkK;
  const uint32_t ring = static_cast<uint32_t>(__cvta_generic_to_shared(sm_raw)) +
                        warp * F::NS * sm_stage_bytes<FMT>();

  // Fetch cursor: runs NS - 1 chunks ahead of the compute cursor over the
  // warp's stream of (task, pass, chunk).
  int f_tau = blockIdx.x * kSmWarps + warp;
  int f_pass = 0, f_c = 0, f_slot = 0;
  SmTask ft;
  if (f_tau < total) ft = sm_task<KIND>(p, s_act, s_off, f_tau, tpe, g);
  auto fetch_next = [&]() {
    if (f_tau < total) {
      sm_fetch<FMT>(p, ft, f_c, ring + f_slot * sm_stage_bytes<FMT>(), lane, tig);
      if (++f_c == nch) {
        f_c = 0;
        if (++f_pass == ft.npass) {
          f_pass = 0;
          f_tau += W;
          if (f_tau < total) ft = sm_task<KIND>(p, s_act, s_off, f_tau, tpe, g);
        }
      }
    }
    cp_async_commit();  // an empty group once the stream has ended
    if (++f_slot == F::NS) f_slot = 0;
  };
#pragma unroll 1
  for (int i = 0; i < F::NS - 1; ++i) fetch_next();

  int slot = 0;
  bool range_flag = false;
#pragma unroll 1
  for (int tau = blockIdx.x * kSmWarps + warp; tau < total; tau += W) {
    const SmTask t = sm_task<KIND>(p, s_act, s_off, tau, tpe, g);
    const float ts = (FMT == kSmNv4 && p.tscale) ? __ldg(p.tscale + t.e) : 1.0f;
#pragma unroll 1
    for (int pass = 0; pass < t.npass; ++pass) {
      // this lane's token of each 8-token tile: n = pass * 16 + nt * 8 + g
      const __nv_bfloat16* brow[kSmNT];
      bool nt_on[kSmNT];
#pragma unroll
      for (int nt = 0; nt < kSmNT; ++nt) {
        const int n0 = pass * kSmTokPass + nt * 8;
        nt_on[nt] = n0 < t.m;  // warp-uniform
        const int n = n0 + g;
        brow[nt] = nullptr;
        if (n < t.m) {
          const int pos = t.row_off + n;
          const long long src = p.perm ? ld_in<COHERENT>(p.perm + pos) / p.div : pos;
          if (src >= 0 && src < p.b_rows) brow[nt] = p.b + src * p.K;
          else atomicOr(p.status, kStatusDeviceCheck);  // a bad permutation: read zeros
        }
      }
      float acc[kSmNT][4];
#pragma unroll
      for (int nt = 0; nt < kSmNT; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[nt][i] = 0.0f;

#pragma unroll 1
      for (int c = 0; c < nch; ++c) {
        // token values of this chunk: per tile, unit i's V values (V / 8 x 16 bytes)
        uint4 bv[kSmNT][4];
#pragma unroll
        for (int nt = 0; nt < kSmNT; ++nt)
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int i = q / (F::V / 8), h = q % (F::V / 8);
            bv[nt][q] = make_uint4(0u, 0u, 0u, 0u);
            if (brow[nt])
              bv[nt][q] = ld_in<kBCoherent>(reinterpret_cast<const uint4*>(
                  brow[nt] + c * kSmChunkK + F::V * (4 * i + tig) + 8 * h));
          }
        fetch_next();
        cp_async_wait<F::NS - 1>();
        const uint32_t st = ring + slot * sm_stage_bytes<FMT>();
        if (++slot == F::NS) slot = 0;
        uint4 av[2][F::U];
#pragma unroll
        for (int rr = 0; rr < 2; ++rr)
#pragma unroll
          for (int i = 0; i < F::U; ++i) av[rr][i] = lds128(st + ((rr * F::U + i) * 32 + lane) * 16);
        uint32_t sc0 = 0, sc1 = 0, sc2 = 0, sc3 = 0;
        if constexpr (F::SB > 0) {
          const uint4 s = lds128(st + 2 * F::U * 32 * 16 + lane * kSmScaleSlot);
          sc0 = s.x; sc1 = s.y; sc2 = s.z; sc3 = s.w;
        }
#pragma unroll
        for (int i = 0; i < F::U; ++i) {
#pragma unroll
          for (int j = 0; j < F::V / 4; ++j) {
            uint32_t a[2][2];  // [row g / g + 8][values 4j, 4j+1 | 4j+2, 4j+3]
            if constexpr (FMT == kSmBf16) {
#pragma unroll
              for (int rr = 0; rr < 2; ++rr) {
                a[rr][0] = word_of(av[rr][i], 2 * j);
                a[rr][1] = word_of(av[rr][i], 2 * j + 1);
              }
            } else if constexpr (FMT == kSmMx8) {
              // unit i: 16 codes in the 32-value block 2 i + tig / 2 of the chunk
              const int blk = 2 * i + (tig >> 1);
#pragma unroll
              for (int rr = 0; rr < 2; ++rr) {
                const uint32_t sbyte = ((rr ? sc1 : sc0) >> (8 * blk)) & 0xffu;
                uint32_t o[2];
                if (sbyte <= 134u) {
                  const uint32_t mbits = ((sbyte + 120u) << 7) * 0x00010001u;
                  e4m3x4_to_bf16_bits(word_of(av[rr][i], j),
                                      *reinterpret_cast<const __nv_bfloat162*>(&mbits), o);
                } else {
                  e4m3x4_to_bf16_scaled(word_of(av[rr][i], j), e8m0_to_float(sbyte), o);
                }
                a[rr][0] = o[0];
                a[rr][1] = o[1];
              }
            } else {
              // one unit of 32 codes: blocks 2 tig (j < 4) and 2 tig + 1 of the
              // chunk's 8; MMA j takes codes 4 j .. 4 j + 3 (word j / 2)
              const int blk = 2 * tig + (j >> 2);  // byte of the 8 scale bytes
#pragma unroll
              for (int rr = 0; rr < 2; ++rr) {
                const uint32_t lo = rr ? sc2 : sc0, hi = rr ? sc3 : sc1;
                const uint32_t sbyte = ((blk < 4 ? lo : hi) >> (8 * (blk & 3))) & 0xffu;
                const uint32_t w = word_of(av[rr][0], j >> 1) >> (16 * (j & 1));
                uint32_t o[2];
                e2m1x4_to_bf16(w, e4m3_scale_bf16x2(sbyte), o);
                a[rr][0] = o[0];
                a[rr][1] = o[1];
              }
            }
#pragma unroll
            for (int nt = 0; nt < kSmNT; ++nt) {
              if (!nt_on[nt]) continue;
              // tokens: values V (4 i + tig) + 4 j + {0..3} of unit i
              const int q = i * (F::V / 8) + (4 * j) / 8;
              const int wsel = ((4 * j) % 8) / 2;
              const uint32_t b0 = word_of(bv[nt][q], wsel), b1 = word_of(bv[nt][q], wsel + 1);
              mma_16816(acc[nt], a[0][0], a[1][0], a[0][1], a[1][1], b0, b1);
            }
          }
        }
      }

      // epilogue: acc[nt] = {(row g, token 2 tig), (g, 2 tig + 1), (g + 8, 2 tig), (g + 8, 2 tig + 1)}
#pragma unroll
      for (int nt = 0; nt < kSmNT; ++nt) {
        if (!nt_on[nt]) continue;
        const int n0 = pass * kSmTokPass + nt * 8 + 2 * tig;
#pragma unroll
        for (int hlf = 0; hlf < 2; ++hlf) {
          const int n = n0 + hlf;
          if (n >= t.m) continue;
          const size_t orow = static_cast<size_t>(t.row_off + n) * p.ld_out;
          if constexpr (KIND == kSmGateUp) {
            const float gt = acc[nt][hlf] * ts, up = acc[nt][2 + hlf] * ts;
            static_cast<__nv_bfloat16*>(p.out)[orow + t.col] =
                __float2bfloat16_rn(__fdividef(gt, 1.0f + __expf(-gt)) * up);
          } else {
#pragma unroll
            for (int rr = 0; rr < 2; ++rr) {
              float v = acc[nt][2 * rr + hlf] * ts;
              if (fabsf(v) > kSmHalfMax) {
                range_flag = true;
                if (fabsf(v) < INFINITY) v = copysignf(kSmHalfMax, v);
              }
              static_cast<__half*>(p.out)[orow + t.col + 8 * rr] = __float2half_rn(v);
            }
          }
        }
      }
    }
  }
  cp_async_wait<0>();  // no copy outlives the phase
  if (KIND == kSmDown && __any_sync(0xffffffffu, range_flag) && lane == 0)
    atomicOr(p.status, kStatusRange);
  __syncthreads();
}

}  // namespace moe
