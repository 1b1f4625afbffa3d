// Grouped expert GEMM kernels and their launchers: the bf16 pair kernels
// (body in moe_expert_gemm.cuh) and the quantised-weight one-CTA kernels.

#include <algorithm>
#include <mutex>

#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "moe_convert.cuh"
#include "moe_device.cuh"
#include "moe_expert_gemm.cuh"
#include "moe_internal.h"

namespace moe {
namespace {

// ---------------------------------------------------------------- MXFP8 weights
//
// The expert GEMMs with the weights stored as MXFP8 ('Hosting Qwen on
// Blackwell', "Quantization"): E4M3 codes and one E8M0 scale per 32 values
// along K (moe_mxfp8.cu).  One CTA per tile: 128 weight rows (gate_up: 64
// gate rows interleaved with the 64 matching up rows) and a chunk of up to
// 128 tokens.  Per 128-wide K stage the TMA brings the tile's codes (16 KB)
// and a bulk copy their scales (512 B) on one barrier, the tokens on another.
// Converter warps turn each code into code x 2^(scale - 127) in bf16 --
// exact, a code has four significant bits -- and store the rows into tensor
// memory; the MMAs read A from there (tcgen05.mma ... [a_tmem]) and B
// (tokens) from shared memory.  Tensor memory holds two accumulators sized
// for the launch's largest chunk and as many A buffers of 64 columns (128 K
// of bf16) as fit beside them, up to 4: the converters run that many stages
// ahead of the MMAs.  Half the weight bytes of the bf16 kernel cross HBM and
// shared memory.
//
// Measured (Qwen3 layer): CTA pairs, whose converters in both CTAs must
// arrive on the leader's barrier before each stage's MMAs, ran prefill at
// 2.92 ms against 2.47 ms for one-CTA tiles; and the converters share the
// sub-partitions' issue slots with the MMA issuer, so four converter warps
// (one per TMEM lane quarter, all four scale blocks of a row each) beat 8 and
// 16 (decode 0.654 / 0.668 / 0.709 ms).

// Weight formats: per pipeline stage a weight row brings one 128-byte row of
// codes -- 128 E4M3 values (MXFP8) or 256 E2M1 values (NVFP4) -- and its
// block scales: 4 E8M0 bytes (one per 32 values) or 16 E4M3 bytes (one per 16).
enum WFormat : int { kMx8 = 0, kNv4 = 1 };
template <int FMT> struct WFmt;
template <> struct WFmt<kMx8> {
  static constexpr int kStageK = 128;       // K values per stage
  static constexpr int kScalesPerRow = 4;   // scale bytes per row per stage
};
template <> struct WFmt<kNv4> {
  static constexpr int kStageK = 256;
  static constexpr int kScalesPerRow = 16;
};
constexpr int kBK8 = 128;                            // code bytes per row per stage
constexpr int kMaxABufs = 4;
constexpr int kA8Bytes = kWRows * kBK8;              // codes per CTA per stage
constexpr int kConvWarp0 = 6;
constexpr int kConvWarpsMx = 4;                      // MXFP8: one per TMEM lane quarter
constexpr int kConvWarpsNv = 8;                      // NVFP4: two per quarter, half the chunks each
__host__ __device__ constexpr int conv_warps(int fmt) { return fmt == 1 ? kConvWarpsNv : kConvWarpsMx; }
__host__ __device__ constexpr int threads_q(int fmt) { return (kConvWarp0 + conv_warps(fmt)) * 32; }
constexpr int kBlkPerWarp = 16 / kConvWarpsMx;       // MXFP8: 32-value scale blocks per warp per stage
constexpr int kMaxStages8 = 8;

template <int KIND, int FMT>
__device__ __forceinline__ void expert_gemm_fp8_body(const CUtensorMap& tmap_w,
                                                     const TokenMapSet& tx, const Params& p) {
  // one CTA's tile: 128 weight rows and a chunk of up to 128 tokens
  constexpr int kSlabH = 64;     // gate_up: h columns per tile (64 gate + 64 up rows)
  constexpr int kSlabRows = 128;  // down: y columns per tile
  constexpr int kStageK = WFmt<FMT>::kStageK;
  constexpr int kSubF = kStageK / kBK;              // 64-wide token boxes per stage
  constexpr int kSPR = WFmt<FMT>::kScalesPerRow;
  constexpr int kABufCols = kStageK / 2;             // TMEM columns of one A buffer (bf16 pairs)
  constexpr int kScaleBytes = kWRows * kSPR;
  constexpr int kConvWarps = conv_warps(FMT);
  extern __shared__ uint8_t smem_raw[];
  __shared__ int s_off[kMaxExperts + 1];
  __shared__ int s_pre[2][kMaxExperts + 1];
  __shared__ alignas(8) uint64_t s_bar[3 * kMaxStages8 + 2 * kMaxABufs + 5];
  __shared__ int s_half_max;
  __shared__ uint32_t s_tmem_base;
  __shared__ int s_abort;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t a_full = smem_u32(&s_bar[0]);                    // own codes + scales landed
  const uint32_t b_full = smem_u32(&s_bar[kMaxStages8]);          // tokens landed
  const uint32_t st_empty = smem_u32(&s_bar[2 * kMaxStages8]);    // stage consumed
  const uint32_t conv_full = smem_u32(&s_bar[3 * kMaxStages8]);   // A buffer converted
  const uint32_t conv_empty = conv_full + 8 * kMaxABufs;          // A buffer read by the MMAs
  const uint32_t tfull_bar = conv_empty + 8 * kMaxABufs;
  const uint32_t tempty_bar = tfull_bar + 16;
  const uint32_t drain_bar = tempty_bar + 16;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kMaxStages8; ++s) {
      mbar_init(a_full + 8 * s, 1);
      mbar_init(b_full + 8 * s, 1);
      mbar_init(st_empty + 8 * s, 1 + kConvWarps);  // the MMA commit + the converters
    }
    for (int b = 0; b < kMaxABufs; ++b) {
      mbar_init(conv_full + 8 * b, kConvWarps);
      mbar_init(conv_empty + 8 * b, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull_bar + 8 * b, 1);
      mbar_init(tempty_bar + 8 * b, 4);  // the epilogue warps
    }
    mbar_init(drain_bar, 1);
    s_abort = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmap_w);
#pragma unroll
    for (int i = 0; i < kTokenMaps; ++i) tma_prefetch_desc(&tx.m[i]);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&s_tmem_base), kTmemCols);
    tmem_relinquish();
  }

  pdl_wait_and_release();

  build_schedule(p, s_off, s_pre, &s_half_max, warp, lane, kTokMax / 2);
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();

  const uint32_t tmem_base = s_tmem_base;
  const Sched sched = make_sched(p, s_off, s_pre);
  const int total_tiles = static_cast<int>(sched.n_all);
  const int num_ks = p.K / kStageK;  // K is a multiple of the stage's K
  const WaitCtx wc{p.timeout_ns, p.status, &s_abort};
  // token rows per K box: the launch's largest chunk (twice its largest half)
  const uint32_t b_sub_bytes = static_cast<uint32_t>(2 * s_half_max) * kBK * 2;
  const uint32_t stage_bytes = (kA8Bytes + kSubF * b_sub_bytes + kScaleBytes + 1023u) & ~1023u;
  const uint32_t avail = static_cast<uint32_t>(p.smem_bytes) - (base - smem_u32(smem_raw));
  const uint32_t acc_cols = static_cast<uint32_t>(2 * s_half_max);
  const int nst = min(kMaxStages8, static_cast<int>(avail / stage_bytes));
  // tensor memory: accumulators [0, acc_cols), [acc_cols, 2 acc_cols); A buffers after them
  const uint32_t abuf0 = (2 * acc_cols + kABufCols - 1) / kABufCols * kABufCols;
  const int nbuf = min(kMaxABufs, static_cast<int>((kTmemCols - abuf0) / kABufCols));

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer (both CTAs)
      int stage = 0;
      uint32_t phase = 0;
      int issued = 0;
      bool ok = true;
      for (int tau = blockIdx.x; tau < total_tiles && ok; tau += gridDim.x) {
        const Tile t = decode_tile(tau, sched);
        const CUtensorMap* tmap_x = &tx.m[t.n / (kUnit / 2) - 1];  // t.n <= 128 rows
        // this CTA's weight rows, and how many of them exist (the last slab may be ragged)
        int row0, row1 = 0, nrow;
        if (KIND == kGateUp) {
          const int g0 = t.slab * kSlabH;
          nrow = max(0, min(64, p.n_out - g0));
          row0 = t.e * p.w_rows_per_group + g0;
          row1 = row0 + p.up_offset;
        } else {
          const int r0 = t.slab * kSlabRows;
          nrow = max(0, min(128, p.n_out - r0));
          row0 = t.e * p.w_rows_per_group + r0;
        }
        const uint32_t scale_tx = (KIND == kGateUp ? 2 : 1) * static_cast<uint32_t>(nrow) * kSPR;
        for (int ks = 0; ks < num_ks; ++ks) {
          if (!mbar_wait(st_empty + 8 * stage, phase ^ 1u, wc)) { ok = false; break; }
          const uint32_t a_dst = base + stage * stage_bytes;
          const uint32_t b_dst = a_dst + kA8Bytes;
          const uint32_t s_dst = b_dst + kSubF * b_sub_bytes;
          const uint32_t af = a_full + 8 * stage;
          mbar_arrive_expect_tx(af, kA8Bytes + scale_tx);
          const int kx = ks * kBK8;  // code bytes
          if (KIND == kGateUp)
            tma_load_5d(a_dst, &tmap_w, af, kx, 0, 0, (row0 - t.e * p.w_rows_per_group) / 16, t.e);
          else
            tma_load_2d(a_dst, &tmap_w, af, kx, row0);
          const uint8_t* sc = p.scales + (static_cast<size_t>(ks) * p.scale_rows) * kSPR;
          if (nrow > 0) {
            bulk_load(s_dst, sc + static_cast<size_t>(row0) * kSPR, nrow * kSPR, af);
            if (KIND == kGateUp)
              bulk_load(s_dst + 64 * kSPR, sc + static_cast<size_t>(row1) * kSPR, nrow * kSPR, af);
          }
          mbar_arrive_expect_tx(b_full + 8 * stage, kSubF * t.n * kBK * 2);
          for (int sub = 0; sub < kSubF; ++sub)
            tma_load_2d(b_dst + sub * b_sub_bytes, tmap_x, b_full + 8 * stage,
                        ks * kStageK + sub * kBK, t.tok0);
          ++issued;
          if (++stage == nst) { stage = 0; phase ^= 1u; }
        }
      }
      for (int i = max(0, issued - nst); i < issued; ++i) {
        mbar_wait_drain(a_full + 8 * (i % nst), (i / nst) & 1, p.status);
        mbar_wait_drain(b_full + 8 * (i % nst), (i / nst) & 1, p.status);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer
      int stage = 0, cb = 0, acc = 0;
      uint32_t phase = 0, cphase = 0, acc_phase = 0;
      bool ok = true;
      for (int tau = blockIdx.x; tau < total_tiles && ok; tau += gridDim.x) {
        const Tile t = decode_tile(tau, sched);
        const uint32_t idesc = idesc_bf16_f32(128, t.n);
        if (!mbar_wait(tempty_bar + 8 * acc, acc_phase ^ 1u, wc)) { ok = false; break; }
        tc_fence_after_sync();
        const uint32_t d_tmem = tmem_base + acc * acc_cols;
        for (int ks = 0; ks < num_ks; ++ks) {
          if (!mbar_wait(b_full + 8 * stage, phase, wc)) { ok = false; break; }
          if (!mbar_wait(conv_full + 8 * cb, cphase, wc)) { ok = false; break; }
          tc_fence_after_sync();
          const uint32_t b_addr = base + stage * stage_bytes + kA8Bytes;
          const uint32_t a_tmem = tmem_base + abuf0 + cb * kABufCols;
          if constexpr (FMT == kNv4) {
            // 16 MMAs per stage: one descriptor per stage, advanced by adds in
            // 16-byte units (measured: NVFP4 prefill -3 %; MXFP8's 8 MMAs per
            // stage were 1.6 % slower in down this way, so they keep the form below)
            const uint64_t db = smem_desc_sw128(b_addr);
            const uint64_t bstep = b_sub_bytes >> 4;
            const uint32_t acc0 = ks != 0 ? 1u : 0u;
#pragma unroll
            for (int k = 0; k < kStageK / 16; ++k)
              mma_bf16_tmem_a(d_tmem, a_tmem + k * 8, db + (k >> 2) * bstep + (k & 3) * 2, idesc,
                              k != 0 ? 1u : acc0);
          } else {
#pragma unroll
            for (int k = 0; k < kStageK / 16; ++k) {
              const uint64_t bd = smem_desc_sw128(b_addr + (k >> 2) * b_sub_bytes + (k & 3) * 32);
              mma_bf16_tmem_a(d_tmem, a_tmem + k * 8, bd, idesc, (ks | k) != 0 ? 1u : 0u);
            }
          }
          mma_commit(st_empty + 8 * stage);  // the tokens of this stage
          mma_commit(conv_empty + 8 * cb);   // the A buffer
          if (++stage == nst) { stage = 0; phase ^= 1u; }
          if (++cb == nbuf) { cb = 0; cphase ^= 1u; }
        }
        if (!ok) break;
        mma_commit(tfull_bar + 8 * acc);
        if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
      }
      mma_commit(drain_bar);
      mbar_wait_drain(drain_bar, 0, p.status);
    }
  } else if (warp < kConvWarp0) {
    // ---------------- epilogue: warps 2..5
    const int q = warp & 3;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int tau = blockIdx.x; tau < total_tiles; tau += gridDim.x) {
      const Tile t = decode_tile(tau, sched);
      const bool live = __all_sync(0xffffffffu, mbar_wait(tfull_bar + 8 * acc, acc_phase, wc));
      tc_fence_after_sync();
      const uint32_t t_row = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * acc_cols;
      epilogue_tile<KIND, KIND == kGateUp ? kSlabH : kSlabRows>(
          t, t_row, live, p, q, lane, 0u, p.tscale ? __ldg(p.tscale + t.e) : 1.0f);
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(tempty_bar + 8 * acc);
      }
      if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
    }
  } else {
    // ---------------- converters: warps 6.., TMEM lanes 32 (warp % 4) + lane.
    // Thread (q, lane) of converter kq converts scale blocks kq * kBlkPerWarp ..
    // (32 K values each) of A row r = 32 q + lane: for gate_up the row of
    // group q that is gate row 16 q + lane (lane < 16) or the matching up row.
    const int q = warp & 3;
    const int kq = (warp - kConvWarp0) >> 2;
    const int r = q * 32 + lane;
    const uint32_t t_lane = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + abuf0;
    int stage = 0, cb = 0;
    uint32_t phase = 0, cphase = 0;
    bool ok = true;
    for (int tau = blockIdx.x; tau < total_tiles && ok; tau += gridDim.x) {
      const Tile t = decode_tile(tau, sched);
      int col, srow;
      if (KIND == kGateUp) {
        col = t.slab * kSlabH + q * 16 + (lane & 15);
        srow = lane < 16 ? q * 16 + lane : 64 + q * 16 + (lane - 16);
      } else {
        col = t.slab * kSlabRows + r;
        srow = r;
      }
      const bool row_ok = col < p.n_out;
      for (int ks = 0; ks < num_ks; ++ks) {
        if (!mbar_wait(a_full + 8 * stage, phase, wc)) { ok = false; break; }
        if (!mbar_wait(conv_empty + 8 * cb, cphase ^ 1u, wc)) { ok = false; break; }
        tc_fence_after_sync();
        const uint32_t a_src = base + stage * stage_bytes;
        const uint32_t s_src = a_src + kA8Bytes + kSubF * b_sub_bytes;
        const uint32_t t_buf = t_lane + cb * kABufCols;
        if constexpr (FMT == kNv4) {
          // NVFP4: the row's 16 block scales, then its 8 chunks of 32 codes (two
          // blocks each), all loaded before converting; 16 TMEM columns per chunk
          constexpr int kCh = 8 / (kConvWarps / 4);  // chunks of this warp
          static_assert(kCh == 4, "the scale words below cover four chunks");
          uint32_t scw[2] = {0u, 0u};                // the 8 block scales of this warp's chunks
          if (row_ok)
            asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];"
                         : "=r"(scw[0]), "=r"(scw[1])
                         : "r"(s_src + srow * 16 + kq * 8));
          uint32_t wv[kCh][4];
#pragma unroll
          for (int c = 0; c < kCh; ++c) {
            const int ch = kq * kCh + c;
            asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(wv[c][0]), "=r"(wv[c][1]), "=r"(wv[c][2]), "=r"(wv[c][3])
                         : "r"(a_src + r * 128 + ((ch ^ (r & 7)) << 4)));
          }
#pragma unroll
          for (int c = 0; c < kCh; ++c) {
            const int ch = kq * kCh + c;
            uint32_t out[16];
#pragma unroll
            for (int hb = 0; hb < 2; ++hb) {  // block 2 ch + hb: words 2 hb, 2 hb + 1
              const int lb = 2 * c + hb;  // block within this warp's 8
              const __nv_bfloat162 mul = e4m3_scale_bf16x2((scw[lb >> 2] >> (8 * (lb & 3))) & 0xffu);
#pragma unroll
              for (int wi = 0; wi < 2; ++wi) {
                const uint32_t w = wv[c][2 * hb + wi];
                e2m1x4_to_bf16(w, mul, out + 8 * hb + 4 * wi);
                e2m1x4_to_bf16(w >> 16, mul, out + 8 * hb + 4 * wi + 2);
              }
            }
            if (!row_ok) {
#pragma unroll
              for (int i = 0; i < 16; ++i) out[i] = 0u;
            }
            tmem_st_32x32b_x16(t_buf + ch * 16, out);
          }
        } else {
        uint32_t sc = 0;
        if (row_ok) asm volatile("ld.shared.b32 %0, [%1];" : "=r"(sc) : "r"(s_src + srow * 4));
        // every code load of this warp's blocks first (two 16-byte chunks of
        // the 128-byte row per block), then the conversions and TMEM stores:
        // one shared-memory round trip per stage
        uint32_t wv[kBlkPerWarp][8];
#pragma unroll
        for (int bi = 0; bi < kBlkPerWarp; ++bi)
#pragma unroll
          for (int hch = 0; hch < 2; ++hch) {
            const int chunk = (kq * kBlkPerWarp + bi) * 2 + hch;
            asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(wv[bi][4 * hch]), "=r"(wv[bi][4 * hch + 1]),
                           "=r"(wv[bi][4 * hch + 2]), "=r"(wv[bi][4 * hch + 3])
                         : "r"(a_src + r * 128 + ((chunk ^ (r & 7)) << 4)));
          }
#pragma unroll
        for (int bi = 0; bi < kBlkPerWarp; ++bi) {
          const int blk = kq * kBlkPerWarp + bi;  // 32 K values: one scale, 16 TMEM columns
          const uint32_t sbyte = (sc >> (8 * blk)) & 0xffu;
          const bool fast = sbyte <= 134u;
          // 2^(S - 7) as a bf16 pair (exponent field S + 120)
          const uint32_t mbits = ((sbyte + 120u) << 7) * 0x00010001u;
          const __nv_bfloat162 mul = *reinterpret_cast<const __nv_bfloat162*>(&mbits);
          const float scale = e8m0_to_float(sbyte);
          uint32_t out[16];
          if (fast) {
#pragma unroll
            for (int i = 0; i < 8; ++i) e4m3x4_to_bf16_bits(wv[bi][i], mul, out + 2 * i);
          } else {
#pragma unroll
            for (int i = 0; i < 4; ++i)
              e4m3x8_to_bf16(wv[bi][2 * i], wv[bi][2 * i + 1], scale, out + 4 * i);
          }
          if (!row_ok) {
#pragma unroll
            for (int i = 0; i < 16; ++i) out[i] = 0u;
          }
          tmem_st_32x32b_x16(t_buf + blk * 16, out);
        }
        }
        tmem_st_wait();
        __syncwarp();
        if (lane == 0) mbar_arrive(st_empty + 8 * stage);  // codes and scales of this stage read
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(conv_full + 8 * cb);
        }
        if (++stage == nst) { stage = 0; phase ^= 1u; }
        if (++cb == nbuf) { cb = 0; cphase ^= 1u; }
      }
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

__global__ void __launch_bounds__(threads_q(kMx8), 1)
    moe_gate_up_swiglu_mxfp8_kernel(const __grid_constant__ CUtensorMap tmap_w,
                                    const __grid_constant__ TokenMapSet tx, const Params p) {
  expert_gemm_fp8_body<kGateUp, kMx8>(tmap_w, tx, p);
}

__global__ void __launch_bounds__(threads_q(kMx8), 1)
    moe_down_mxfp8_kernel(const __grid_constant__ CUtensorMap tmap_w,
                          const __grid_constant__ TokenMapSet tx, const Params p) {
  expert_gemm_fp8_body<kDown, kMx8>(tmap_w, tx, p);
}

__global__ void __launch_bounds__(threads_q(kNv4), 1)
    moe_gate_up_swiglu_nvfp4_kernel(const __grid_constant__ CUtensorMap tmap_w,
                                    const __grid_constant__ TokenMapSet tx, const Params p) {
  expert_gemm_fp8_body<kGateUp, kNv4>(tmap_w, tx, p);
}

__global__ void __launch_bounds__(threads_q(kNv4), 1)
    moe_down_nvfp4_kernel(const __grid_constant__ CUtensorMap tmap_w,
                          const __grid_constant__ TokenMapSet tx, const Params p) {
  expert_gemm_fp8_body<kDown, kNv4>(tmap_w, tx, p);
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreadsSched, 1)
    moe_gate_up_swiglu_kernel(const __grid_constant__ CUtensorMap tmap_w,
                              const __grid_constant__ TokenMapSet tx, const Params p) {
  expert_gemm_body<kGateUp>(tmap_w, tx, p);
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreadsSched, 1)
    moe_down_kernel(const __grid_constant__ CUtensorMap tmap_w,
                    const __grid_constant__ TokenMapSet tx, const Params p) {
  expert_gemm_body<kDown>(tmap_w, tx, p);
}

typedef void (*ExpertKernel)(const CUtensorMap, const TokenMapSet, const Params);

// The bf16 GEMMs hand their tiles out through the workspace's tile counter up
// to this many token rows per expert on average (decode batches).
constexpr long long kDynRowsPerExpert = 8;
// ... and warm L2 with this many 64-wide K boxes of their first tile's
// weights before waiting for the kernel before them.  down's CTAs take the
// SMs that gate_up's leave during its last tiles, so its prefetch overlaps
// gate_up's tail; gate_up's CTAs wait for the one-CTA grouping kernel only.
// Same-box A/B (decode layer, alternating twice): both 0.7068 / 0.7069 ms,
// gate_up's alone 0.7085 / 0.7086, none 0.7085 / 0.7086.
constexpr int kPrefetchBoxesGateUp = 0;
constexpr int kPrefetchBoxesDown = 16;

// Dynamic shared memory of a launch: all that a block may use beyond the
// kernel's static shared memory (the pipeline takes as many stages as fit).
// Set as the kernel's limit on first use per device; 0 on failure.
int ensure_smem_attr(ExpertKernel k, int which) {
  static std::mutex mu;
  static int bytes[6][64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  std::lock_guard<std::mutex> lock(mu);
  if (bytes[which][dev]) return bytes[which][dev];
  int optin = 0;
  cudaFuncAttributes fa{};
  if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess ||
      cudaFuncGetAttributes(&fa, k) != cudaSuccess)
    return 0;
  const int dyn = optin - static_cast<int>(fa.sharedSizeBytes);
  if (dyn < kMinStages * kSub * (kABytes + (kTokMax / 2) * kBK * 2) + 1024) return 0;
  if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, dyn) != cudaSuccess)
    return 0;
  bytes[which][dev] = dyn;
  return dyn;
}

// Pairs that can be resident at once.  A pair needs two SMs of one GPC, so
// this can be fewer than half the SMs; a persistent grid larger than it would
// run its surplus pairs' whole tile lists as a second wave.
int resident_pairs(ExpertKernel k, int which, int smem_bytes, int threads) {
  static std::mutex mu;
  static int cached[4][64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
  std::lock_guard<std::mutex> lock(mu);
  if (!cached[which][dev]) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * (device_sm_count() / 2), 1, 1);
    cfg.blockDim = dim3(threads, 1, 1);
    cfg.dynamicSmemBytes = smem_bytes;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, k, &cfg) != cudaSuccess || n <= 0) {
      cudaGetLastError();
      n = device_sm_count() / 2;
    }
    cached[which][dev] = std::min(n, device_sm_count() / 2);
  }
  return cached[which][dev];
}

cudaError_t launch_expert(cudaStream_t s, const char* name, ExpertKernel k, int which,
                          const CUtensorMap& mw, const TokenMapSet& mx, Params p,
                          long long tiles_bound, int threads = kThreads) {
  const int smem = ensure_smem_attr(k, which);
  if (smem <= 0) {
    cudaGetLastError();
    return cudaErrorInvalidConfiguration;
  }
  p.smem_bytes = smem;
  const long long pairs =
      std::max(1LL, std::min<long long>(resident_pairs(k, which, smem, threads), tiles_bound));
  KernelScope scope(s, name);
  return launch_kernel(k, dim3(static_cast<unsigned>(2 * pairs)), dim3(threads),
                       static_cast<size_t>(smem), s, mw, mx, p);
}

// One CTA per SM (the kernels take all the shared memory), static stride over tiles.
cudaError_t launch_expert_1cta(cudaStream_t s, const char* name, ExpertKernel k, int which,
                               const CUtensorMap& mw, const TokenMapSet& mx, Params p,
                               long long tiles_bound, int threads) {
  const int smem = ensure_smem_attr(k, which);
  if (smem <= 0) {
    cudaGetLastError();
    return cudaErrorInvalidConfiguration;
  }
  p.smem_bytes = smem;
  const long long grid = std::max(1LL, std::min<long long>(device_sm_count(), tiles_bound));
  KernelScope scope(s, name);
  return launch_kernel(k, dim3(static_cast<unsigned>(grid)), dim3(threads),
                       static_cast<size_t>(smem), s, mw, mx, p);
}

}  // namespace

cudaError_t launch_grouped_ffn(cudaStream_t s, const void* a, const int32_t* offsets, int rows,
                               int d, int E, int I, const void* w_gate_up, const void* w_down,
                               void* h, void* y, unsigned* status,
                               unsigned long long timeout_ns, const TokenGather* gather,
                               bool y_fp32, unsigned* sched_words) {
  const int groups = offsets ? E : 1;
  const long long chunks_bound =
      offsets ? rows / kTokMax + std::min(E, rows) : (rows + kTokMax - 1) / kTokMax;

  CUtensorMap mw;
  TokenMapSet mx;
  Params p{};
  cudaError_t e = make_gate_up_weight_map(&mw, w_gate_up, d, I, groups);
  if (e == cudaSuccess) e = make_gate_up_token_maps(mx, p, a, rows, d, gather);
  if (e != cudaSuccess) return e;
  p.K = d;
  p.n_out = I;
  p.slabs = (I + 127) / 128;
  p.groups = groups;
  p.offsets = offsets;
  p.total_rows = rows;
  p.w_rows_per_group = 2 * I;
  p.up_offset = I;
  p.out = h;
  p.ld_out = I;
  p.status = status;
  p.timeout_ns = timeout_ns;
  // Dynamic schedule for decode-sized layers only.  Same-box A/B against the
  // static stride (alternating twice): decode -0.6 % (gate_up 459.6 against
  // 463.2 us), prefill no change, the skewed layer +1.5 %, the DeepSeek-like
  // layer +1 %.
  const bool dyn = sched_words != nullptr && rows <= kDynRowsPerExpert * groups;
  if (dyn) {
    p.tile_ctr = sched_words + kTileCounterWord;
    p.exit_ctr = sched_words + kTileExitWord;
    p.prefetch_boxes = kPrefetchBoxesGateUp;
  }
  e = launch_expert(s, offsets ? "moe_gate_up_swiglu" : "moe_shared_gate_up_swiglu",
                    moe_gate_up_swiglu_kernel, 0, mw, mx, p, chunks_bound * p.slabs,
                    dyn ? kThreadsSched : kThreads);
  if (e != cudaSuccess) return e;

  CUtensorMap mw2;
  TokenMapSet mx2;
  e = make_bf16_map(&mw2, w_down, static_cast<uint64_t>(groups) * d, I, 128);
  if (e == cudaSuccess) e = make_token_maps(mx2, h, rows, I);
  if (e != cudaSuccess) return e;
  Params q{};
  q.K = I;
  q.n_out = d;
  q.slabs = (d + 255) / 256;
  q.groups = groups;
  q.offsets = offsets;
  q.total_rows = rows;
  q.w_rows_per_group = d;
  q.up_offset = 0;
  q.out = y;
  q.ld_out = d;
  q.y_fp32 = y_fp32 ? 1 : 0;
  q.status = status;
  q.timeout_ns = timeout_ns;
  q.tile_ctr = p.tile_ctr;  // gate_up has reset them by the time down takes a tile
  q.exit_ctr = p.exit_ctr;
  q.prefetch_boxes = dyn ? kPrefetchBoxesDown : 0;
  return launch_expert(s, offsets ? "moe_down" : "moe_shared_down", moe_down_kernel, 1, mw2, mx2,
                       q, chunks_bound * q.slabs, dyn ? kThreadsSched : kThreads);
}

cudaError_t launch_grouped_ffn_quant(cudaStream_t s, int fmt, const void* a,
                                     const int32_t* offsets, int rows, int d, int E, int I,
                                     const uint8_t* codes_gate_up, const uint8_t* scales_gate_up,
                                     const float* tscale_gate_up, const uint8_t* codes_down,
                                     const uint8_t* scales_down, const float* tscale_down,
                                     void* h, void* y, unsigned* status,
                                     unsigned long long timeout_ns, bool y_fp32) {
  const bool nv = fmt == kNv4;
  const uint64_t d_bytes = nv ? d / 2 : d;  // code bytes of a W_gate_up row
  const uint64_t i_bytes = nv ? I / 2 : I;  // code bytes of a W_down row
  // one CTA per tile, chunks of at most 128 tokens
  const long long chunks_bound = rows / (kTokMax / 2) + std::min(E, rows);

  // codes of W_gate_up [E][2][I][d] viewed as (d, 16 rows, gate|up, I/16 row groups, E): one
  // box = 128 code bytes of 4 row groups, each 16 gate rows followed by the 16 matching up rows
  CUtensorMap mw;
  TokenMapSet mx;
  const uint64_t dims[5] = {d_bytes, 16, 2, static_cast<uint64_t>(I / 16),
                            static_cast<uint64_t>(E)};
  const uint64_t strides[4] = {d_bytes, static_cast<uint64_t>(I) * d_bytes, 16ull * d_bytes,
                               2ull * I * d_bytes};
  const uint32_t box[5] = {kBK8, 16, 2, 4, 1};
  Params p{};
  cudaError_t e = make_u8_map_nd(&mw, codes_gate_up, 5, dims, strides, box);
  if (e == cudaSuccess) e = make_token_maps(mx, a, rows, d);
  if (e != cudaSuccess) return e;
  p.K = d;
  p.n_out = I;
  p.slabs = I / 64;
  p.groups = E;
  p.offsets = offsets;
  p.total_rows = rows;
  p.w_rows_per_group = 2 * I;
  p.up_offset = I;
  p.out = h;
  p.ld_out = I;
  p.scales = scales_gate_up;
  p.scale_rows = 2LL * I * E;
  p.tscale = nv ? tscale_gate_up : nullptr;
  p.status = status;
  p.timeout_ns = timeout_ns;
  e = nv ? launch_expert_1cta(s, "moe_gate_up_swiglu_nvfp4", moe_gate_up_swiglu_nvfp4_kernel, 4,
                              mw, mx, p, chunks_bound * p.slabs, threads_q(kNv4))
         : launch_expert_1cta(s, "moe_gate_up_swiglu_mxfp8", moe_gate_up_swiglu_mxfp8_kernel, 2,
                              mw, mx, p, chunks_bound * p.slabs, threads_q(kMx8));
  if (e != cudaSuccess) return e;

  CUtensorMap mw2;
  TokenMapSet mx2;
  const uint64_t dims2[2] = {i_bytes, static_cast<uint64_t>(E) * d};
  const uint64_t strides2[1] = {i_bytes};
  const uint32_t box2[2] = {kBK8, 128};
  e = make_u8_map_nd(&mw2, codes_down, 2, dims2, strides2, box2);
  if (e == cudaSuccess) e = make_token_maps(mx2, h, rows, I);
  if (e != cudaSuccess) return e;
  Params q{};
  q.K = I;
  q.n_out = d;
  q.slabs = (d + 127) / 128;
  q.groups = E;
  q.offsets = offsets;
  q.total_rows = rows;
  q.w_rows_per_group = d;
  q.out = y;
  q.ld_out = d;
  q.y_fp32 = y_fp32 ? 1 : 0;
  q.scales = scales_down;
  q.scale_rows = static_cast<long long>(E) * d;
  q.tscale = nv ? tscale_down : nullptr;
  q.status = status;
  q.timeout_ns = timeout_ns;
  return nv ? launch_expert_1cta(s, "moe_down_nvfp4", moe_down_nvfp4_kernel, 5, mw2, mx2, q,
                                 chunks_bound * q.slabs, threads_q(kNv4))
            : launch_expert_1cta(s, "moe_down_mxfp8", moe_down_mxfp8_kernel, 3, mw2, mx2, q,
                                 chunks_bound * q.slabs, threads_q(kMx8));
}

}  // namespace moe
