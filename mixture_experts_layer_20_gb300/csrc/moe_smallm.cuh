// Warp-level small-M expert GEMM (mma.sync m16n8k16) for the decode case of
// the grouped SwiGLU FFN with quantised expert weights (moe_smallm.cu, where
// the design is described); mma_16816 and word_of also serve the router
// phase of the single-launch layer.
#pragma once

#include <cstdint>
#include <type_traits>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "moe_convert.cuh"
#include "moe_internal.h"

namespace moe {

// kSmMx8A8: MXFP8 weights and MXFP8 token rows (W8A8, fp8 warp MMAs)
enum SmFmt : int { kSmMx8 = 1, kSmNv4 = 2, kSmMx8A8 = 3 };
enum SmKind : int { kSmGateUp = 1, kSmDown = 2 };

constexpr int kSmWarps = 8;               // warps per CTA
constexpr int kSmThreads = kSmWarps * 32;
constexpr int kSmTok = 8;                 // tokens per pass (the MMA's N)
constexpr float kSmHalfMax = 65504.0f;

// Per weight format: V values per 16-byte unit; U units per lane and weight
// row per chunk, so a chunk covers KC = 4 V U values of the reduction; NS
// ring stages; SB block-scale bytes per weight row per chunk (0: none).
template <int FMT> struct SmF;
template <> struct SmF<kSmMx8> {
  static constexpr int V = 16, U = 4, NS = 3, SB = 8;
  static constexpr int kBytesX2 = 2;  // twice the bytes per value
};
template <> struct SmF<kSmNv4> {
  static constexpr int V = 32, U = 2, NS = 4, SB = 16;
  static constexpr int kBytesX2 = 1;
};
// W8A8: the same weight stages as kSmMx8 (a lane's unit i: bytes 16 tig ..
// + 15 of the chunk's 64-byte span i, of rows g and g + 8), stored at a
// swizzled unit slot so that ldmatrix reads the MMA fragments without bank
// conflicts (one fp8 MMA per 32-value run).
template <> struct SmF<kSmMx8A8> {
  static constexpr int V = 16, U = 4, NS = 3, SB = 8;
  static constexpr int kBytesX2 = 2;
};
template <int FMT>
__host__ __device__ constexpr int sm_chunk_k() {
  return 4 * SmF<FMT>::V * SmF<FMT>::U;
}
// Block-scale bytes a lane keeps per stage: both of its rows' scales.
template <int FMT>
__host__ __device__ constexpr int sm_scale_slot() {
  return 2 * SmF<FMT>::SB;
}
template <int FMT>
__host__ __device__ constexpr int sm_stage_bytes() {
  return 2 * SmF<FMT>::U * 32 * 16 + 32 * sm_scale_slot<FMT>();
}
template <int FMT>
__host__ __device__ constexpr int sm_smem_bytes() {
  return kSmWarps * SmF<FMT>::NS * sm_stage_bytes<FMT>();
}

struct SmParams {
  const uint8_t* w;          // weight rows (codes), row_bytes each
  const uint8_t* scales;     // MXFP8 [K/128][scale_rows][4], NVFP4 [K/256][scale_rows][16]
  const float* tscale;       // NVFP4: one scale per expert (null: none)
  long long scale_rows;      // weight rows of the whole tensor
  long long row_bytes;
  int K;                     // reduction length (a multiple of the chunk)
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
  int y_fp32;                // down: y in fp32 (else fp16, saturated at the fp16 range)
  unsigned* status;
  // W8A8: token rows as MXFP8 (launch_act_mxfp8's layout) instead of b
  const uint8_t* bq;         // codes [b_rows, K]
  const uint8_t* bs;         // scales [b_rows, K / 32]
};

__device__ __forceinline__ void cp_async_16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
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

// D = A B with A 16 x 32 E4M3 (row-major fragment), B 32 x 8 E4M3
// (column-major fragment), D 16 x 8 fp32 (no accumulator input).
__device__ __forceinline__ void mma_16832_e4m3(float (&d)[4], uint32_t a0, uint32_t a1,
                                               uint32_t a2, uint32_t a3, uint32_t b0,
                                               uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%10, %10, %10, %10};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.0f));
}

// Four 8 x 8 matrices of 16-bit elements (here 8 rows of 16 codes each) from
// shared memory: lanes 8 m .. 8 m + 7 give the row addresses of matrix m;
// register m of lane (g, tig) gets bytes 4 tig .. + 3 of row g of matrix m.
__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                            uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ uint32_t word_of(const uint4& v, int i) {
  return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

// One task: 16 weight rows of one expert (see the file comment of
// moe_smallm.cu) over the whole reduction, for all of the expert's tokens in
// passes of 8.  Pointers are this lane's: its two weight rows (fragment rows
// g and g + 8) at its first unit, and their block scales.
struct SmTask {
  int e, m, row_off;      // expert, its token rows, first row in the grouped layout
  int col;                // gate_up: h column c0 + g; down: y column r0 + g
  int npass;
  const uint8_t* w0;
  const uint8_t* w1;
  const uint8_t* s0;
  const uint8_t* s1;
};

template <int FMT, int KIND>
__device__ __forceinline__ SmTask sm_task(const SmParams& p, const int* s_act, const int* s_off,
                                          int tau, int tpe, int g, int tig) {
  SmTask t;
  const int a = tau / tpe;
  const int cg = tau - a * tpe;
  t.e = s_act[a];
  t.row_off = s_off[t.e];
  t.m = s_off[t.e + 1] - t.row_off;
  t.npass = (t.m + kSmTok - 1) / kSmTok;
  const long long base = static_cast<long long>(t.e) * p.w_rows_per_expert;
  long long r0, r1;
  if (KIND == kSmGateUp) {
    t.col = cg * 8 + g;
    r0 = base + t.col;
    r1 = r0 + p.up_offset;
  } else {
    t.col = cg * 16 + g;
    r0 = base + t.col;
    r1 = r0 + 8;
  }
  t.w0 = p.w + r0 * p.row_bytes + 16 * tig;
  t.w1 = p.w + r1 * p.row_bytes + 16 * tig;
  if constexpr (FMT == kSmMx8 || FMT == kSmMx8A8) {
    t.s0 = p.scales + r0 * 4;
    t.s1 = p.scales + r1 * 4;
  } else {
    t.s0 = p.scales + r0 * 16;
    t.s1 = p.scales + r1 * 16;
  }
  return t;
}

// Copies of chunk c of a task's weights (and scales) into ring slot `slot`:
// unit i of row half rr at ((rr U + i) 32 + lane) 16, the lane's scale bytes
// after the units.
template <int FMT>
__device__ __forceinline__ void sm_fetch(const SmParams& p, const SmTask& t, int c, uint32_t slot,
                                         int lane) {
  using F = SmF<FMT>;
  constexpr int kChunkBytes = sm_chunk_k<FMT>() * F::kBytesX2 / 2;  // = 64 U
  const long long off = static_cast<long long>(c) * kChunkBytes;
  // W8A8: the unit of lane (g, tig) goes to slot 4 g + (tig ^ ((g >> 1) & 3))
  const int u_slot = FMT == kSmMx8A8 ? (lane & ~3) | ((lane & 3) ^ ((lane >> 3) & 3)) : lane;
#pragma unroll
  for (int i = 0; i < F::U; ++i) {
    cp_async_16(slot + (i * 32 + u_slot) * 16, t.w0 + off + 64 * i);
    cp_async_16(slot + ((F::U + i) * 32 + u_slot) * 16, t.w1 + off + 64 * i);
  }
  const uint32_t s = slot + 2 * F::U * 32 * 16 + lane * sm_scale_slot<FMT>();
  if constexpr (FMT == kSmMx8 || FMT == kSmMx8A8) {
    // a 256-wide chunk spans two 128-wide scale stages: one word per row each
    const long long st = 2LL * c * p.scale_rows * 4;
    const long long st2 = st + p.scale_rows * 4;
    cp_async_4(s, t.s0 + st);
    cp_async_4(s + 4, t.s0 + st2);
    cp_async_4(s + 8, t.s1 + st);
    cp_async_4(s + 12, t.s1 + st2);
  } else {
    const long long st = static_cast<long long>(c) * p.scale_rows * 16;  // one stage per chunk
    cp_async_16(s, t.s0 + st);
    cp_async_16(s + 16, t.s1 + st);
  }
}

// One grouped GEMM (gate_up or down) by all warps of the grid.  sm_raw: the
// block's dynamic shared memory (sm_smem_bytes<FMT>()).  COHERENT: the
// offsets, the permutation and (down) the token rows h were written by this
// kernel before a grid-wide barrier (see ld_in).  Ends with every copy landed
// and a block-wide barrier.
template <int FMT, int KIND, bool COHERENT = false>
__device__ __forceinline__ void sm_phase(const SmParams& p, uint8_t* sm_raw) {
  using F = SmF<FMT>;
  constexpr int KC = sm_chunk_k<FMT>();
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
  const int nch = p.K / KC;
  const uint32_t ring = static_cast<uint32_t>(__cvta_generic_to_shared(sm_raw)) +
                        warp * F::NS * sm_stage_bytes<FMT>();

  // Fetch cursor: runs NS - 1 chunks ahead of the compute cursor over the
  // warp's stream of (task, pass, chunk).
  int f_tau = blockIdx.x * kSmWarps + warp;
  int f_pass = 0, f_c = 0;
  uint32_t f_slot = ring;
  SmTask ft;
  if (f_tau < total) ft = sm_task<FMT, KIND>(p, s_act, s_off, f_tau, tpe, g, tig);
  auto fetch_next = [&]() {
    if (f_tau < total) {
      sm_fetch<FMT>(p, ft, f_c, f_slot, lane);
      if (++f_c == nch) {
        f_c = 0;
        if (++f_pass == ft.npass) {
          f_pass = 0;
          f_tau += W;
          if (f_tau < total) ft = sm_task<FMT, KIND>(p, s_act, s_off, f_tau, tpe, g, tig);
        }
      }
    }
    cp_async_commit();  // an empty group once the stream has ended
    f_slot += sm_stage_bytes<FMT>();
    if (f_slot == ring + F::NS * sm_stage_bytes<FMT>()) f_slot = ring;
  };
#pragma unroll 1
  for (int i = 0; i < F::NS - 1; ++i) fetch_next();

  uint32_t st = ring;
  bool range_flag = false;
  // NVFP4: byte selectors of this lane's two block scales in a scale word
  const uint32_t ssel0 = e4m3_scale_sel(2u * (tig & 1));
  const uint32_t ssel1 = e4m3_scale_sel(2u * (tig & 1) + 1u);
  (void)ssel0;
  (void)ssel1;
#pragma unroll 1
  for (int tau = blockIdx.x * kSmWarps + warp; tau < total; tau += W) {
    const SmTask t = sm_task<FMT, KIND>(p, s_act, s_off, tau, tpe, g, tig);
    // NVFP4: the tensor scale, times 2^8 for the MMAs' weights x 2^-8 (see
    // e2m1x8_to_bf16_pairs)
    const float ts =
        FMT == kSmNv4 ? (p.tscale ? __ldg(p.tscale + t.e) : 1.0f) * 256.0f : 1.0f;
#pragma unroll 1
    for (int pass = 0; pass < t.npass; ++pass) {
      // Source row of the expert's token n (-1 past the expert's rows, or for a
      // bad permutation entry, which is recorded and read as zeros).
      auto src_row = [&](int n) -> long long {
        if (n >= t.m) return -1;
        const int pos = t.row_off + n;
        const long long src = p.perm ? ld_in<COHERENT>(p.perm + pos) / p.div : pos;
        if (src >= 0 && src < p.b_rows) return src;
        atomicOr(p.status, kStatusDeviceCheck);
        return -1;
      };
      // kAcc accumulators, taken in turn by a unit's MMAs, break the MMA
      // dependency chain; they are added in a fixed order at the end
      constexpr int kAcc = F::V / 4 < 4 ? F::V / 4 : 4;
      float acc[kAcc][4];
#pragma unroll
      for (int q = 0; q < kAcc; ++q) acc[q][0] = acc[q][1] = acc[q][2] = acc[q][3] = 0.0f;

      if constexpr (FMT == kSmMx8A8) {
        // W8A8.  B operand: token n = 8 pass + g (its MXFP8 codes); the
        // accumulator columns are tokens 8 pass + 2 tig and + 1, whose run
        // scales multiply the partial sums.  One MMA per 32-value run r of a
        // chunk, k-position = value index within the run: ldmatrix brings the
        // weight fragments (rows g / g + 8, values 4 tig + j / 16 + 4 tig + j)
        // from the units of the lanes that copied them, and the token codes
        // are stored so that a lane's 8 bytes of run r are those values.
        // This lane's row address for ldmatrix: matrix mm = lane / 8 (rows g
        // or g + 8, first or second 16 codes of the run), row jj = lane % 8.
        const int mm = lane >> 3, jj = lane & 7;
        const int ld_unit = (mm & 1) * F::U;          // units of rows g + 8 follow those of g
        const int ld_half = mm >> 1;                  // 16-code half of the run
        const long long sb = src_row(pass * kSmTok + g);
        const uint8_t* bqrow = sb >= 0 ? p.bq + sb * p.K : nullptr;
        const uint8_t* bsr[2];
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const long long sr = src_row(pass * kSmTok + 2 * tig + hh);
          bsr[hh] = sr >= 0 ? p.bs + sr * (p.K / 32) : nullptr;
        }
#pragma unroll 1
        for (int c = 0; c < nch; ++c) {
          __syncwarp();  // every lane has read the slot that fetch_next refills
          uint4 bv[F::U];
#pragma unroll
          for (int i = 0; i < F::U; ++i)
            bv[i] = bqrow ? ld_in<kBCoherent>(reinterpret_cast<const uint4*>(bqrow + c * KC + 64 * tig + 16 * i))
                          : make_uint4(0u, 0u, 0u, 0u);
          uint2 sx[2];
#pragma unroll
          for (int hh = 0; hh < 2; ++hh)
            sx[hh] = bsr[hh] ? ld_in<kBCoherent>(reinterpret_cast<const uint2*>(bsr[hh] + c * 8))
                             : make_uint2(0u, 0u);
          fetch_next();
          cp_async_wait<F::NS - 1>();
          __syncwarp();  // the other lanes' units of this slot have landed
          const uint32_t cur = st;
          st += sm_stage_bytes<FMT>();
          if (st == ring + F::NS * sm_stage_bytes<FMT>()) st = ring;
          // weight run scales: x / y row g runs 0-3 / 4-7, z / w row g + 8
          const uint4 sc = lds128(cur + 2 * F::U * 32 * 16 + lane * sm_scale_slot<FMT>());
          // the chunk's eight MMAs first (independent), then their scaling,
          // so that no MMA waits for the one before it
          float d[2 * F::U][4];
#pragma unroll
          for (int i = 0; i < F::U; ++i) {
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
              // run 2 i + hh: bytes 32 hh + 16 ld_half of span i, copied by
              // lane (jj, 2 hh + ld_half) into its swizzled slot
              const int tsrc = 2 * hh + ld_half;
              const uint32_t addr =
                  cur + ((ld_unit + i) * 32 + 4 * jj + (tsrc ^ ((jj >> 1) & 3))) * 16;
              uint32_t a0, a1, a2, a3;
              ldmatrix_x4(addr, a0, a1, a2, a3);
              mma_16832_e4m3(d[2 * i + hh], a0, a1, a2, a3, word_of(bv[i], 2 * hh),
                             word_of(bv[i], 2 * hh + 1));
            }
          }
#pragma unroll
          for (int r = 0; r < 2 * F::U; ++r) {
            const int sh = 8 * (r & 3);
            const float w0 = e8m0_to_float(((r < 4 ? sc.x : sc.y) >> sh) & 0xffu);
            const float w1 = e8m0_to_float(((r < 4 ? sc.z : sc.w) >> sh) & 0xffu);
            const float x0 = e8m0_to_float(((r < 4 ? sx[0].x : sx[0].y) >> sh) & 0xffu);
            const float x1 = e8m0_to_float(((r < 4 ? sx[1].x : sx[1].y) >> sh) & 0xffu);
            acc[0][0] = fmaf(d[r][0], w0 * x0, acc[0][0]);
            acc[0][1] = fmaf(d[r][1], w0 * x1, acc[0][1]);
            acc[0][2] = fmaf(d[r][2], w1 * x0, acc[0][2]);
            acc[0][3] = fmaf(d[r][3], w1 * x1, acc[0][3]);
          }
        }
      } else {
      // this lane's token: n = 8 pass + g (none past the expert's rows)
      const __nv_bfloat16* brow = nullptr;
      {
        const long long src = src_row(pass * kSmTok + g);
        if (src >= 0) brow = p.b + src * p.K;
      }

#pragma unroll 1
      for (int c = 0; c < nch; ++c) {
        // token values of this chunk, unit by unit: values V (4 i + tig) + [0, V)
        uint4 bv[F::U][F::V / 8];
#pragma unroll
        for (int i = 0; i < F::U; ++i)
#pragma unroll
          for (int h = 0; h < F::V / 8; ++h)
            bv[i][h] = brow ? ld_in<kBCoherent>(reinterpret_cast<const uint4*>(
                                  brow + c * KC + F::V * (4 * i + tig) + 8 * h))
                            : make_uint4(0u, 0u, 0u, 0u);
        fetch_next();
        cp_async_wait<F::NS - 1>();
        const uint32_t cur = st;
        st += sm_stage_bytes<FMT>();
        if (st == ring + F::NS * sm_stage_bytes<FMT>()) st = ring;
        const uint32_t sslot = cur + 2 * F::U * 32 * 16 + lane * sm_scale_slot<FMT>();
        const uint4 sc = lds128(sslot);
        uint4 sc2 = make_uint4(0u, 0u, 0u, 0u);
        if constexpr (FMT == kSmNv4) sc2 = lds128(sslot + 16);
        // MXFP8: a scale byte above 134 (weights beyond 2^7 in a block) needs
        // the general conversion; decided once per chunk for the whole warp, so
        // each variant of the chunk body below is one straight-line block
        bool slow = false;
        if constexpr (FMT == kSmMx8) {
          const unsigned big = __vcmpgtu4(sc.x, 0x86868686u) | __vcmpgtu4(sc.y, 0x86868686u) |
                               __vcmpgtu4(sc.z, 0x86868686u) | __vcmpgtu4(sc.w, 0x86868686u);
          slow = __any_sync(0xffffffffu, big != 0u);
        }
        auto chunk_body = [&](auto slow_tag) {
          constexpr bool kSlow = decltype(slow_tag)::value;
          (void)kSlow;
#pragma unroll
          for (int i = 0; i < F::U; ++i) {
            const uint4 a0 = lds128(cur + (i * 32 + lane) * 16);
            const uint4 a1 = lds128(cur + ((F::U + i) * 32 + lane) * 16);
            if constexpr (FMT == kSmMx8) {
              // unit i holds 16 codes of the 32-value block 2 i + tig / 2 of the
              // chunk (scale word: row half, block / 4; byte: block % 4)
              const int blk = 2 * i + (tig >> 1);
              uint32_t sb[2];
              sb[0] = ((i < 2 ? sc.x : sc.y) >> (8 * (blk & 3))) & 0xffu;
              sb[1] = ((i < 2 ? sc.z : sc.w) >> (8 * (blk & 3))) & 0xffu;
#pragma unroll
              for (int j = 0; j < F::V / 4; ++j) {
                uint32_t a[2][2];  // [row g / g + 8][values 4j, 4j+1 | 4j+2, 4j+3]
#pragma unroll
                for (int rr = 0; rr < 2; ++rr) {
                  const uint32_t codes = word_of(rr ? a1 : a0, j);
                  if constexpr (!kSlow) {
                    const uint32_t mbits = ((sb[rr] + 120u) << 7) * 0x00010001u;
                    e4m3x4_to_bf16_bits(codes, *reinterpret_cast<const __nv_bfloat162*>(&mbits),
                                        a[rr]);
                  } else {
                    e4m3x4_to_bf16_scaled(codes, e8m0_to_float(sb[rr]), a[rr]);
                  }
                }
                // tokens: values V (4 i + tig) + 4 j + {0..3}: 16-byte piece (4 j) / 8
                const uint4& bq = bv[i][(4 * j) / 8];
                const int wsel = ((4 * j) % 8) / 2;
                mma_16816(acc[j % kAcc], a[0][0], a[1][0], a[0][1], a[1][1], word_of(bq, wsel),
                          word_of(bq, wsel + 1));
              }
            } else {
              // unit i: 32 codes = blocks 8 i + 2 tig and + 1 of the chunk's 16
              // (scale word 2 i + tig / 2, bytes 2 (tig & 1) and + 1); word m of
              // the unit holds codes 8 m .. 8 m + 7, of block m / 2
              __nv_bfloat162 mul[2][2];
#pragma unroll
              for (int rr = 0; rr < 2; ++rr) {
                const uint32_t sw = word_of(rr ? sc2 : sc, 2 * i + (tig >> 1));
                mul[rr][0] = e4m3_scale_x2p118(sw, ssel0);
                mul[rr][1] = e4m3_scale_x2p118(sw, ssel1);
              }
#pragma unroll
              for (int m = 0; m < 4; ++m) {
                uint32_t q[2][4];  // [row g / g + 8][code pairs (0,4) (1,5) (2,6) (3,7)]
#pragma unroll
                for (int rr = 0; rr < 2; ++rr)
                  e2m1x8_to_bf16_pairs(word_of(rr ? a1 : a0, m), mul[rr][m >> 1], q[rr]);
                // the token values of the same positions, paired alike: the
                // 16-byte piece m holds values 8 m .. 8 m + 7 as 4 bf16 pairs
                const uint4& bq = bv[i][m];
                uint32_t b04, b15, b26, b37;
                asm("prmt.b32 %0, %1, %2, 0x5410;" : "=r"(b04) : "r"(bq.x), "r"(bq.z));
                asm("prmt.b32 %0, %1, %2, 0x7632;" : "=r"(b15) : "r"(bq.x), "r"(bq.z));
                asm("prmt.b32 %0, %1, %2, 0x5410;" : "=r"(b26) : "r"(bq.y), "r"(bq.w));
                asm("prmt.b32 %0, %1, %2, 0x7632;" : "=r"(b37) : "r"(bq.y), "r"(bq.w));
                mma_16816(acc[(2 * m) % kAcc], q[0][0], q[1][0], q[0][1], q[1][1], b04, b15);
                mma_16816(acc[(2 * m + 1) % kAcc], q[0][2], q[1][2], q[0][3], q[1][3], b26, b37);
              }
            }
          }
        };
        if (FMT == kSmMx8 && slow) chunk_body(std::true_type{});
        else chunk_body(std::false_type{});
      }
      }  // not W8A8

      // epilogue: acc = {(row g, token 2 tig), (g, 2 tig + 1), (g + 8, 2 tig), (g + 8, 2 tig + 1)}
#pragma unroll
      for (int q = 1; q < kAcc; ++q)
#pragma unroll
        for (int v = 0; v < 4; ++v) acc[0][v] += acc[q][v];
#pragma unroll
      for (int hlf = 0; hlf < 2; ++hlf) {
        const int n = pass * kSmTok + 2 * tig + hlf;
        if (n >= t.m) continue;
        const size_t orow = static_cast<size_t>(t.row_off + n) * p.ld_out;
        if constexpr (KIND == kSmGateUp) {
          const float gt = acc[0][hlf] * ts;
          const float up = acc[0][2 + hlf] * ts;
          static_cast<__nv_bfloat16*>(p.out)[orow + t.col] =
              __float2bfloat16_rn(__fdividef(gt, 1.0f + __expf(-gt)) * up);
        } else {
#pragma unroll
          for (int rr = 0; rr < 2; ++rr) {
            float v = acc[0][2 * rr + hlf] * ts;
            if (p.y_fp32) {  // the full fp32 range, no saturation
              static_cast<float*>(p.out)[orow + t.col + 8 * rr] = v;
              continue;
            }
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
  cp_async_wait<0>();  // no copy outlives the phase
  if (KIND == kSmDown && __any_sync(0xffffffffu, range_flag) && lane == 0)
    atomicOr(p.status, kStatusRange);
  __syncthreads();
}

}  // namespace moe
