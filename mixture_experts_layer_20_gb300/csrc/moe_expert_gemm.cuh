// The bf16 expert GEMM body (2-SM tcgen05 pairs, weights on M) and its tile
// schedule: device code shared by the grouped-GEMM kernels (moe_expert_gemm.cu)
// and the single-launch decode layer (moe_fused.cu).
//
// Grouped expert GEMMs of the MoE layer on sm_103a: 2-SM tcgen05 MMAs with the
// expert weights on the M side.
//
//   gate_up : h[t, c] = silu(x[t] . W_gate[c]) * (x[t] . W_up[c]), bf16
//   down    : y[t, c] = h[t] . W_down[c], accumulated in fp32, stored in fp16
//
// for every token row t of an expert's contiguous range of the grouped
// activations ('Chapter 9. Distributed inference', section 9.3.2: three
// d x I matrices per expert; section 9.4.3: one grouped GEMM for all experts).
//
// Work unit (a "tile") = one expert, one slab of 256 weight rows, one chunk
// of that expert's tokens.  Weights are the MMA's M side, so M is always
// full; tokens are the N side, chunked so that no expert is padded by more
// than 15 rows (an expert with m rows gets ceil(m/256) chunks that share its
// ceil(m/16) 16-row units as evenly as possible, so a CTA's half of a chunk
// is a multiple of 8 rows up to 128 and one TMA instruction fetches it; each TMA or
// MMA instruction costs its single issuing thread tens of cycles, so few
// large ones keep the tensor pipe fed).  A cluster of two CTAs (a pair) computes a
// tile with tcgen05.mma.cta_group::2 (M = 256): each CTA holds 128 weight
// rows and half of the token rows of every K block, so each SM moves at most
// 32 KB per 64-wide K block.  A pipeline stage holds two such K blocks: the
// thread that issues the MMAs pays tens of cycles per instruction and per
// barrier round, so 8 MMAs per wait / commit keep it ahead of a 256 x 256
// tile's tensor work.  The stages are sized for the launch's largest chunk:
// 3 fit in shared memory for 256-token chunks, 4 when no chunk exceeds 192.
// Tiles are ordered (expert, slab, chunk): pairs running at the same time
// read the same weight slab, which is then read from HBM once.  Pair p takes
// tiles p, p + pairs, ...; or, for decode-sized layers, the pairs take them
// in order from a counter in global memory (a scheduler warp of the leader
// fetches the next indices and publishes them to both CTAs of its pair), so
// a pair that streams its weights faster takes more tiles.
//
// gate_up: rank r of the pair holds the gate rows [128 s + 64 r, +64) of slab
// s and the matching up rows, interleaved in groups of 16 (A rows 32 j .. 32 j
// + 15: gate rows 16 j .. 16 j + 15 of the CTA's 64, A rows 32 j + 16 .. 32 j
// + 31: the matching up rows), so the gate and up accumulators of one h column
// sit in TMEM lanes l and l + 16 of the same 32-lane quarter, which one
// epilogue warp reads: a register shuffle pairs them.  With the weights on M,
// a warp's lanes are consecutive output columns, so every store of one token
// row is contiguous.
//
// Roles, per CTA (192 threads, 224 with the scheduler warp 6 of the dynamic
// schedule): warp 0 loads both operands with TMA into its
// own shared memory, counting the bytes of both CTAs on the leader's full
// barrier; warp 1 owns the tensor memory (512 columns: two accumulators of up
// to 256 fp32 columns) and, in the leader, one of its threads issues the MMAs
// and commits to both CTAs' barriers; warps 2-5 read the accumulator with
// tcgen05.ld and store the tile while the next one accumulates.  Every wait
// is bounded; on timeout a CTA records it, drains its copies in flight (and,
// in the leader, its MMAs), and both CTAs still meet at the final cluster
// barrier before freeing tensor memory.

#pragma once

#include <cuda_fp16.h>

#include "moe_device.cuh"
#include "moe_internal.h"

namespace moe {


constexpr int kBK = 64;     // one 128-byte swizzle row of bf16: the K of one TMA box
constexpr int kSub = 2;     // K boxes per pipeline stage: 8 MMAs per barrier round
constexpr int kMaxStages = 4;                      // down: pipeline stages (3 for 256-token chunks)
constexpr int kMaxStagesGateUp = 6;                // gate_up: more stages when chunks are small
constexpr int kMaxStagesAny = kMaxStagesGateUp;    // size of the barrier arrays
static_assert(kMaxStages <= kMaxStagesAny, "the barrier arrays hold kMaxStagesAny stages");
constexpr int kTileRing = 16;  // tile token counts passed from the producer to the MMA issuer
static_assert(kMaxStagesAny + 1 < kTileRing, "the producer runs at most kMaxStagesAny tiles ahead");
constexpr int kWRows = 128;                        // weight rows per CTA
constexpr int kTokMax = 256;                       // tokens per tile (MMA N)
constexpr int kUnit = 16;                          // token rows: chunks are multiples of this
constexpr int kABytes = kWRows * kBK * 2;          // 16 KB per K box
constexpr int kMinStages = 3;                      // 3 stages of the largest (256-token) chunks
constexpr int kThreads = 192;
// With the dynamic schedule a seventh warp fetches the tiles (kSchedAhead at
// most ahead of the producer).
constexpr int kThreadsSched = kThreads + 32;
constexpr int kSchedAhead = 4;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAccCols = 256;
constexpr uint32_t kEpiArrivals = 8;               // 4 epilogue warps x 2 CTAs
constexpr float kHalfMax = 65504.0f;               // largest finite fp16

enum Kind : int { kGateUp = 1, kDown = 2 };

struct Params {
  int K;                  // reduction length (d or I), a multiple of 64
  int n_out;              // output columns: I (h) or d (y)
  int slabs;              // 256-row weight slabs per expert
  int groups;             // experts, or 1 when offsets == nullptr
  const int32_t* offsets;  // [groups + 1] token row offsets, or nullptr
  int total_rows;         // token rows of the B operand
  int w_rows_per_group;   // weight rows per expert in the A tensor map
  int up_offset;          // gate_up: I
  void* out;              // gate_up: h bf16 [rows, I]; down: y fp16 [rows, d]
  long long ld_out;
  // Token rows gathered on the fly (null: B is [total_rows, K] in row order):
  // B row of slot pos is row gather_perm[pos] / gather_div of the map over
  // the unpermuted tokens; slots past total_rows read row gather_oob (zeros).
  const int32_t* gather_perm;
  int gather_div;
  int gather_oob;
  const uint8_t* scales;  // MXFP8 / NVFP4 weights: block scales [K / stage K][scale_rows][per row]
  long long scale_rows;   // MXFP8 / NVFP4 weights: weight rows of the whole tensor
  const float* tscale;    // NVFP4 weights: tensor scale per expert (null: none)
  int smem_bytes;         // dynamic shared memory of the launch
  int y_fp32;             // down: y in fp32 (else fp16, saturated at the fp16 range)
  // Dynamic schedule (null: tile pair + i * pairs for the i-th tile of a
  // pair): the leader of each pair takes its next tile from *tile_ctr, in
  // order; the last CTA to leave (*exit_ctr) resets both to zero.
  unsigned* tile_ctr;
  unsigned* exit_ctr;
  int prefetch_boxes;     // dynamic schedule: K boxes of weights to warm L2 with before the wait
  unsigned* status;
  unsigned long long timeout_ns;
};

struct Tile {
  int e, slab, tok0, tok_end, n;
};

// Gathered B operand: lane l of the producer warp brings token rows
// 4 l .. 4 l + 3 of the `cnt` rows from slot row0 on; their source rows.
struct GatherRows {
  int r[4];
  bool on;  // this lane has rows to bring
};

// COHERENT: perm was written by this kernel before a grid-wide barrier.
template <bool COHERENT = false>
__device__ __forceinline__ GatherRows gather_rows(const Params& p, int row0, int cnt, int lane) {
  GatherRows g;
  g.on = p.gather_perm != nullptr && 4 * lane < cnt;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int pos = row0 + 4 * lane + i;
    g.r[i] = g.on && pos < p.total_rows ? ld_in<COHERENT>(p.gather_perm + pos) / p.gather_div
                                        : p.gather_oob;
  }
  return g;
}

// The launch's tiles, as built by build_schedule in shared memory.  Experts
// with several token chunks ("multi") reuse each weight slab from L2 for
// their second and later chunks, so their tiles lean on the tensor cores;
// single-chunk experts stream every slab from HBM.  Tile position tau of the
// launch interleaves the two classes in proportion (multi-chunk tile number
// floor(tau * n_multi / n_all) comes next whenever that count grows at tau),
// so the pairs working at the same time mix both kinds and the two roofs
// overlap instead of adding up one after the other (a skewed routing gives a
// few experts many chunks and most one).  Within a class tiles stay in
// (expert, slab, chunk) order: the chunks of one slab sit in neighbouring
// positions and run at the same time, so the slab is read from HBM once.
// With one class only (prefill: all experts multi-chunk; decode: all single)
// the order is plain (expert, slab, chunk).
struct Sched {
  const int* off;      // [G + 1] token row offsets
  const int* pre_multi;   // [G + 1] exclusive chunk prefix of multi-chunk experts
  const int* pre_single;  // [G + 1] the same for single-chunk experts
  int slabs, groups;
  long long n_multi;   // tiles of multi-chunk experts
  long long n_all;     // all tiles
};

__device__ __forceinline__ Tile decode_tile(int tau, const Sched& sc) {
  const long long before = static_cast<long long>(tau) * sc.n_multi / sc.n_all;
  const bool multi = (static_cast<long long>(tau) + 1) * sc.n_multi / sc.n_all > before;
  const int idx = multi ? static_cast<int>(before) : tau - static_cast<int>(before);
  const int* pre = multi ? sc.pre_multi : sc.pre_single;
  const int slabs = sc.slabs;
  // the expert whose tiles of this class hold idx: the last with pre * slabs <= idx
  // (experts without tiles in the class repeat the prefix and are passed over)
  int lo = 0, hi = sc.groups - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (pre[mid] * slabs <= idx) lo = mid; else hi = mid - 1;
  }
  Tile t;
  t.e = lo;
  const int ch = pre[lo + 1] - pre[lo];
  const int local = idx - pre[lo] * slabs;
  t.slab = local / ch;
  const int c = local - t.slab * ch;
  // the expert's ceil(m / 16) row units, spread over its ch chunks as evenly as
  // possible (the first `rem` chunks take one unit more)
  const int* s_off = sc.off;
  const int m = s_off[lo + 1] - s_off[lo];
  const int u = (m + kUnit - 1) / kUnit;
  const int base_u = u / ch, rem = u - base_u * ch;
  t.tok0 = s_off[lo] + kUnit * (c * base_u + min(c, rem));
  t.n = kUnit * (base_u + (c < rem ? 1 : 0));
  t.tok_end = min(t.tok0 + t.n, s_off[lo + 1]);
  return t;
}

// The token operand comes through one of sixteen tensor maps whose boxes are
// 8, 16, ..., 128 rows: one TMA instruction loads a CTA's n/2 token rows.
constexpr int kTokenMaps = kTokMax / kUnit;
struct TokenMapSet {
  CUtensorMap m[kTokenMaps];
};

// Schedule (all threads of the CTA): token chunks per expert (at most TOKCAP
// tokens each), their exclusive prefix per class (s_pre[0]: experts with two
// or more chunks, s_pre[1]: experts with one; entry G holds the class total),
// and the largest chunk half of the launch in *s_half_max.  Inconsistent
// offsets give an empty schedule and MOE_ERR_DEVICE_CHECK.
// COHERENT: the offsets were written by this kernel before a grid-wide barrier.
template <bool COHERENT = false>
__device__ __forceinline__ void build_schedule(const Params& p, int* s_off,
                                               int (*s_pre)[kMaxExperts + 1], int* s_half_max,
                                               int warp, int lane, int TOKCAP) {
  const int G = p.groups;
  for (int i = threadIdx.x; i <= G; i += blockDim.x)
    s_off[i] = p.offsets ? ld_in<COHERENT>(p.offsets + i) : (i == 0 ? 0 : p.total_rows);
  __syncthreads();
  if (warp == 0) {
    const int per = (G + 31) / 32;
    int local_m = 0, local_s = 0;
    int half_max = kUnit / 2;
    bool bad = false;
    for (int j = 0; j < per; ++j) {
      const int g = lane * per + j;
      if (g < G) {
        const int m = s_off[g + 1] - s_off[g];
        bad |= m < 0;
        if (m > 0) {
          const int ch = (m + TOKCAP - 1) / TOKCAP;
          if (ch > 1) local_m += ch; else local_s += 1;
          half_max = max(half_max, (((m + kUnit - 1) / kUnit + ch - 1) / ch) * (kUnit / 2));
        }
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) half_max = max(half_max, __shfl_xor_sync(0xffffffffu, half_max, o));
    int incl_m = local_m, incl_s = local_s;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int vm = __shfl_up_sync(0xffffffffu, incl_m, o);
      const int vs = __shfl_up_sync(0xffffffffu, incl_s, o);
      if (lane >= o) { incl_m += vm; incl_s += vs; }
    }
    int run_m = incl_m - local_m, run_s = incl_s - local_s;
    for (int j = 0; j < per; ++j) {
      const int g = lane * per + j;
      if (g < G) {
        s_pre[0][g] = run_m;
        s_pre[1][g] = run_s;
        const int m = s_off[g + 1] - s_off[g];
        const int ch = m > 0 ? (m + TOKCAP - 1) / TOKCAP : 0;
        if (ch > 1) run_m += ch; else run_s += ch;
      }
    }
    bad |= (s_off[0] != 0) || (s_off[G] != p.total_rows);
    bad = __any_sync(0xffffffffu, bad);
    __syncwarp();
    if (lane == 31) {
      s_pre[0][G] = bad ? 0 : incl_m;
      s_pre[1][G] = bad ? 0 : incl_s;
    }
    if (lane == 0) *s_half_max = bad ? TOKCAP / 2 : min(half_max, TOKCAP / 2);
    if (bad && lane == 0 && blockIdx.x == 0) atomicOr(p.status, kStatusDeviceCheck);
  }
}

// The launch's tile list over the schedule in shared memory (after the
// barrier that follows build_schedule).
__device__ __forceinline__ Sched make_sched(const Params& p, const int* s_off,
                                            const int (*s_pre)[kMaxExperts + 1]) {
  Sched sc;
  sc.off = s_off;
  sc.pre_multi = s_pre[0];
  sc.pre_single = s_pre[1];
  sc.slabs = p.slabs;
  sc.groups = p.groups;
  sc.n_multi = static_cast<long long>(s_pre[0][p.groups]) * p.slabs;
  sc.n_all = sc.n_multi + static_cast<long long>(s_pre[1][p.groups]) * p.slabs;
  return sc;
}

// Epilogue of one tile (one of warps 2-5, q = warp % 4, reading TMEM lanes
// 32 q .. 32 q + 31 from t_row): gate_up stores h = silu(gate) * up in bf16,
// down stores y in fp16; `live` false (a wait gave up) stores nothing.
// y in fp16: finite values beyond +-65504 are stored as +-65504 and
// infinities as they are, and either sets kStatusRange (NaN passes unflagged).
template <int KIND, int SLAB = (KIND == kGateUp ? 128 : 256)>
__device__ __forceinline__ void epilogue_tile(const Tile& t, uint32_t t_row, bool live,
                                              const Params& p, int q, int lane, uint32_t rank,
                                              float tscale = 1.0f) {
  // SLAB: output columns of one tile (h columns for gate_up, y columns for down).
  // tscale: the weights' tensor scale (NVFP4), applied to the accumulators.
  if constexpr (KIND == kDown) {
    const int col = t.slab * SLAB + rank * 128 + q * 32 + lane;
    const bool col_ok = live && col < p.n_out;
    bool out_of_range = false;
#pragma unroll 1
    for (int c = 0; c < t.n; c += 16) {
      uint32_t v[16];
      tmem_ld_32x32b_x16(t_row + c, v);
      tmem_ld_wait();
      const int nvalid = min(16, t.tok_end - t.tok0 - c);  // uniform across the warp
      float f[16];
      float m = 0.0f;  // largest |y| of the valid rows (NaN does not count)
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        f[j] = __uint_as_float(v[j]) * tscale;
        if (j < nvalid) m = fmaxf(m, fabsf(f[j]));
      }
      if (p.y_fp32) {  // the full fp32 range, no saturation
        float* yq = static_cast<float*>(p.out) + (size_t)(t.tok0 + c) * p.ld_out + col;
        if (col_ok) {
#pragma unroll
          for (int j = 0; j < 16; ++j)
            if (j < nvalid) yq[(size_t)j * p.ld_out] = f[j];
        }
        continue;
      }
      if (m > kHalfMax) {  // rare: saturate the finite values beyond the fp16 range
        out_of_range = true;
#pragma unroll
        for (int j = 0; j < 16; ++j)
          if (fabsf(f[j]) > kHalfMax && fabsf(f[j]) < INFINITY) f[j] = copysignf(kHalfMax, f[j]);
      }
      __half2 hv[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) hv[i] = __floats2half2_rn(f[2 * i], f[2 * i + 1]);
      __half* yp = static_cast<__half*>(p.out) + (size_t)(t.tok0 + c) * p.ld_out + col;
      if (col_ok) {
        if (nvalid == 16) {
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            yp[(size_t)(2 * i) * p.ld_out] = __low2half(hv[i]);
            yp[(size_t)(2 * i + 1) * p.ld_out] = __high2half(hv[i]);
          }
        } else {
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            if (2 * i < nvalid) yp[(size_t)(2 * i) * p.ld_out] = __low2half(hv[i]);
            if (2 * i + 1 < nvalid) yp[(size_t)(2 * i + 1) * p.ld_out] = __high2half(hv[i]);
          }
        }
      }
    }
    if (__any_sync(0xffffffffu, col_ok && out_of_range) && lane == 0) atomicOr(p.status, kStatusRange);
  } else {
    // In each warp's quarter of the TMEM lanes, lanes 0-15 hold 16 gate
    // rows and lanes 16-31 the matching up rows (the weight map
    // interleaves them in groups of 16), so one shuffle pairs them: lane
    // l < 16 computes tokens c..c+7 and lane l + 16 tokens c+8..c+15 of
    // h column l, and all four warps share the SwiGLU and the stores.
    const bool lo = lane < 16;
    const int col = t.slab * SLAB + rank * 64 + q * 16 + (lane & 15);
    const bool col_ok = live && col < p.n_out;
    __nv_bfloat16* h = static_cast<__nv_bfloat16*>(p.out) + col;
#pragma unroll 1
    for (int c = 0; c < t.n; c += 16) {
      uint32_t v[16];
      tmem_ld_32x32b_x16(t_row + c, v);
      tmem_ld_wait();
      if (tscale != 1.0f) {
#pragma unroll
        for (int j = 0; j < 16; ++j) v[j] = __float_as_uint(__uint_as_float(v[j]) * tscale);
      }
      const int row0 = t.tok0 + c + (lo ? 0 : 8);
      const int nvalid = min(8, t.tok_end - row0);  // <= 0: rows past the expert's end
      __nv_bfloat16* hp = h + (size_t)row0 * p.ld_out;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float mine = __uint_as_float(lo ? v[i] : v[8 + i]);
        const float other =
            __shfl_xor_sync(0xffffffffu, __uint_as_float(lo ? v[8 + i] : v[i]), 16);
        const float g = lo ? mine : other;
        const float u = lo ? other : mine;
        if (col_ok && i < nvalid)
          hp[(size_t)i * p.ld_out] =
              __float2bfloat16_rn(__fdividef(g, 1.0f + __expf(-g)) * u);
      }
    }
  }
}

// FUSED: a phase of the single-launch layer.  The kernel allocated the
// pair's 512 tensor-memory columns once (fused_tmem) and frees them itself;
// the offsets and the permutation come from earlier phases of the same kernel
// (read through L2); the token rows the TMA loads may have been written by
// generic stores of an earlier phase, so the producer orders its TMA (async
// proxy) after them with a proxy fence, and the phase ends with one for its own
// stores.
template <int KIND, bool FUSED = false>
__device__ __forceinline__ void expert_gemm_body(const CUtensorMap& tmap_w, const TokenMapSet& tx,
                                                 const Params& p, uint32_t fused_tmem = 0) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ int s_off[kMaxExperts + 1];
  __shared__ int s_pre[2][kMaxExperts + 1];
  __shared__ alignas(8) uint64_t s_bar[(kSub + 1) * kMaxStagesAny + 5];
  __shared__ int s_half_max;
  __shared__ uint32_t s_tmem_base;
  __shared__ int s_abort;
  // Token count of the tile whose first stage the producer armed, by tile
  // sequence number mod kTileRing: the MMA issuer reads it after that stage's
  // full barrier instead of decoding the tile itself (it is at most
  // kMaxStagesAny stages, so as many tiles, behind the producer).
  __shared__ int s_tile_n[kTileRing];
  // Dynamic schedule: tile index by tile sequence number mod kTileRing (-1:
  // no more tiles), written in both CTAs by the leader's scheduler warp
  // before it arrives on s_tbar of that slot (locally and remotely); every
  // other role of both CTAs waits there.  The scheduler stays at most
  // kSchedAhead tiles ahead of the leader's producer (s_prod_next: tiles the
  // producer has taken) and at most kMaxStagesAny + 3 tiles separate the
  // producer from the slowest reader, so a slot is read before it is reused.
  __shared__ int s_tau[kTileRing];
  __shared__ alignas(8) uint64_t s_tbar[kTileRing];
  __shared__ int s_prod_next;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int pair = blockIdx.x >> 1;
  const int num_pairs = gridDim.x >> 1;

  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  // full: one per stage.  empty: gate_up releases each K box of a stage on
  // its own barrier (box 0 of stage s at empty_bar + 8 s, box b > 0 at
  // empty_hi + 8 ((b - 1) kMaxStagesAny + s)), so a box is refilled as soon as the MMAs that read it are done while the
  // stage's other box is still in use; down releases a stage at once (box 0's
  // barrier).  Measured on one box: gate_up -2 % at prefill, -9 % on the
  // DeepSeek-like layer; down at decode +3 % with per-box release (its short
  // 16-token tiles pay for the extra commit and wait per stage).
  constexpr bool kBoxRelease = KIND == kGateUp;
  const uint32_t full_bar = smem_u32(&s_bar[0]);
  const uint32_t empty_bar = smem_u32(&s_bar[kMaxStagesAny]);
  const uint32_t tfull_bar = smem_u32(&s_bar[2 * kMaxStagesAny]);
  const uint32_t tempty_bar = smem_u32(&s_bar[2 * kMaxStagesAny + 2]);
  const uint32_t drain_bar = smem_u32(&s_bar[2 * kMaxStagesAny + 4]);
  const uint32_t empty_hi = smem_u32(&s_bar[2 * kMaxStagesAny + 5]);
  const uint32_t tbar = smem_u32(&s_tbar[0]);
  auto empty_box = [&](int b, int st) {
    return b == 0 ? empty_bar + 8 * st : empty_hi + 8 * ((b - 1) * kMaxStagesAny + st);
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < kMaxStagesAny; ++s) {
      mbar_init(full_bar + 8 * s, 1);  // leader: counts both CTAs' bytes; unused in the follower
      for (int b = 0; b < kSub; ++b) mbar_init(empty_box(b, s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull_bar + 8 * a, 1);
      mbar_init(tempty_bar + 8 * a, kEpiArrivals);
    }
    mbar_init(drain_bar, 1);
    for (int i = 0; i < kTileRing; ++i) mbar_init(tbar + 8 * i, 1);
    s_prod_next = 0;
    s_abort = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmap_w);
#pragma unroll
    for (int i = 0; i < kTokenMaps; ++i) tma_prefetch_desc(&tx.m[i]);
  }
  if (!FUSED && warp == 1) {
    tmem_alloc_pair(smem_u32(&s_tmem_base), kTmemCols);
    tmem_relinquish_pair();
  }

  // Decode-sized launches: the weights do not depend on the kernels before
  // this one (routing, grouping), so while they finish, each CTA warms L2
  // with the first kPrefetchBoxes K boxes of its half of the tile its pair
  // would take first if every expert had tokens (at decode nearly all do);
  // a wrong guess costs only the bandwidth.
  if (!FUSED && p.tile_ctr != nullptr && p.prefetch_boxes > 0 && threadIdx.x == 0) {
    const int e = pair / p.slabs, slab = pair - (pair / p.slabs) * p.slabs;
    // whole boxes inside the weight tensor only (a partial last slab is skipped)
    const bool inside = KIND == kGateUp ? (slab * 128 + static_cast<int>(rank) * 64 + 64) * 2 <= p.w_rows_per_group
                                        : slab * 256 + static_cast<int>(rank) * 128 + 128 <= p.w_rows_per_group;
    if (e < p.groups && inside) {
      const int nb = min(p.prefetch_boxes, p.K / kBK);
      for (int kb = 0; kb < nb; ++kb) {
        if (KIND == kGateUp)
          tma_prefetch_l2_5d(&tmap_w, kb * kBK, 0, 0, (slab * 128 + static_cast<int>(rank) * 64) / 16, e);
        else
          tma_prefetch_l2_2d(&tmap_w, kb * kBK,
                             e * p.w_rows_per_group + slab * 256 + static_cast<int>(rank) * 128);
      }
    }
  }
  pdl_wait_and_release();

  build_schedule<FUSED>(p, s_off, s_pre, &s_half_max, warp, lane, kTokMax);
  tc_fence_before_sync();
  __syncthreads();
  cluster_sync();  // the peer's barriers are initialised before any remote arrive
  tc_fence_after_sync();

  const uint32_t tmem_base = FUSED ? fused_tmem : s_tmem_base;
  const Sched sched = make_sched(p, s_off, s_pre);
  const int total_tiles = static_cast<int>(sched.n_all);
  const int num_kb = p.K / kBK;                   // 64-wide K boxes
  const WaitCtx wc{p.timeout_ns, p.status, &s_abort};
  // (the scheduler warp must exist: launched with kThreadsSched threads)
  const bool dyn = !FUSED && p.tile_ctr != nullptr && blockDim.x >= kThreadsSched;
  // Tile of sequence number `seq` of this pair (one thread): the static
  // stride, or the index the leader's producer published; -1 past the last
  // tile, or once a wait has given up.
  auto tile_at = [&](int seq) -> int {
    if (!dyn) {
      const long long t = pair + static_cast<long long>(seq) * num_pairs;
      return t < total_tiles ? static_cast<int>(t) : -1;
    }
    const int slot = seq % kTileRing;
    if (!mbar_wait_cluster(tbar + 8 * slot, (seq / kTileRing) & 1, wc)) return -1;
    return s_tau[slot];
  };
  // The same for a whole warp (lane 0 waits).
  auto tile_at_warp = [&](int seq) -> int {
    int t = 0;
    if (lane == 0) t = tile_at(seq);
    return __shfl_sync(0xffffffffu, t, 0);
  };
  const int num_ks = (num_kb + kSub - 1) / kSub;  // pipeline stages per tile
  // Stage geometry: a stage holds kSub K boxes of the weights and of the
  // largest token-chunk half of this launch, so smaller chunks leave room for
  // more stages.  Both CTAs of a pair derive the same layout.
  const uint32_t b_sub_bytes = static_cast<uint32_t>(s_half_max) * kBK * 2;
  const uint32_t stage_bytes = kSub * (kABytes + b_sub_bytes);
  const uint32_t avail = static_cast<uint32_t>(p.smem_bytes) - (base - smem_u32(smem_raw));
  // Measured at decode (16-token chunks): gate_up streams its weights at 6.95
  // TB/s with six stages in flight against 6.85 with four; down, whose tiles
  // are 12 stages long, is slower with more (248 against 239 us).
  const int max_st = KIND == kGateUp ? kMaxStagesGateUp : kMaxStages;
  const int nst = min(max_st, static_cast<int>(avail / stage_bytes));

  if (warp == 0) {
    // ---------------- TMA producer (warp 0 of both CTAs, own shared memory;
    // the bytes of both are counted on the leader's full barrier, which the
    // leader arms with the pair's total).  Lane 0 waits, arms and loads the
    // weights; the token rows come in one box per K box, or, gathered, four
    // rows per lane.
    int stage = 0;
    uint32_t phase = 0;
    int issued = 0;
    bool ok = true;
    int seq = 0;
    const uint32_t full_leader = mapa_shared(full_bar, 0);
    if (FUSED) fence_proxy_async_global();  // earlier phases' generic stores before this TMA
    for (;; ++seq) {
      const int tau = ok ? tile_at_warp(seq) : -1;
      if (tau < 0) break;
      if (dyn && leader && lane == 0) *static_cast<volatile int*>(&s_prod_next) = seq + 1;
      const Tile t = decode_tile(tau, sched);
      const int half = t.n / 2;  // token rows per CTA: 8, 16, ..., 128
      const CUtensorMap* tmap_x = &tx.m[t.n / kUnit - 1];
      const uint32_t tx_bytes = kABytes + half * 128;  // per CTA
      const int trow = t.tok0 + rank * half;  // this CTA's first token row
      const int wrow = KIND == kGateUp ? t.slab * 128 + rank * 64
                                       : t.e * p.w_rows_per_group + t.slab * 256 + rank * 128;
      const GatherRows gr = gather_rows<FUSED>(p, trow, half, lane);
      if constexpr (!kBoxRelease) {
        for (int ks = 0; ks < num_ks; ++ks) {
          const int nsub = min(kSub, num_kb - ks * kSub);
          const bool got = lane == 0 ? mbar_wait(empty_bar + 8 * stage, phase ^ 1u, wc) : true;
          if (!__shfl_sync(0xffffffffu, got, 0)) { ok = false; break; }
          const uint32_t fb = full_leader + 8 * stage;
          const uint32_t a_dst = base + stage * stage_bytes;
          const uint32_t b_dst = a_dst + kSub * kABytes;
          if (lane == 0) {
            if (ks == 0) s_tile_n[seq % kTileRing] = t.n;  // before the arrive that releases it
            if (leader) mbar_arrive_expect_tx(full_bar + 8 * stage, 2 * nsub * tx_bytes);
            for (int sub = 0; sub < nsub; ++sub) {
              const int kx = (ks * kSub + sub) * kBK;
              if (KIND == kGateUp)
                tma_load_5d_pair(a_dst + sub * kABytes, &tmap_w, fb, kx, 0, 0, wrow / 16, t.e);
              else
                tma_load_2d_pair(a_dst + sub * kABytes, &tmap_w, fb, kx, wrow);
              if (p.gather_perm == nullptr)
                tma_load_2d_pair(b_dst + sub * b_sub_bytes, tmap_x, fb, kx, trow);
            }
          }
          if (gr.on) {
            for (int sub = 0; sub < nsub; ++sub)
              tma_gather4_pair(b_dst + sub * b_sub_bytes + lane * 512, &tx.m[0], fb,
                               (ks * kSub + sub) * kBK, gr.r[0], gr.r[1], gr.r[2], gr.r[3]);
          }
          ++issued;
          if (++stage == nst) { stage = 0; phase ^= 1u; }
        }
      } else {
        for (int ks = 0; ks < num_ks && ok; ++ks) {
          const int nsub = min(kSub, num_kb - ks * kSub);
          const uint32_t fb = full_leader + 8 * stage;
          const uint32_t a_dst = base + stage * stage_bytes;
          const uint32_t b_dst = a_dst + kSub * kABytes;
          bool armed = false;  // the stage's barrier is armed and its first box on the way
#pragma unroll
          for (int sub = 0; sub < kSub; ++sub) {
            // box `sub` of this stage is free once the MMAs that read it are done
            const bool got = lane == 0 ? mbar_wait(empty_box(sub, stage), phase ^ 1u, wc) : true;
            if (!__shfl_sync(0xffffffffu, got, 0)) { ok = false; break; }
            armed = true;
            if (lane == 0) {
              if (sub == 0) {
                if (ks == 0) s_tile_n[seq % kTileRing] = t.n;  // before the arrive that releases it
                if (leader) mbar_arrive_expect_tx(full_bar + 8 * stage, 2 * nsub * tx_bytes);
              }
              if (sub < nsub) {
                const int kx = (ks * kSub + sub) * kBK;
                // gate_up: one box holds 4 groups of {16 gate rows, the 16 matching up rows}
                if (KIND == kGateUp)
                  tma_load_5d_pair(a_dst + sub * kABytes, &tmap_w, fb, kx, 0, 0, wrow / 16, t.e);
                else
                  tma_load_2d_pair(a_dst + sub * kABytes, &tmap_w, fb, kx, wrow);
                if (p.gather_perm == nullptr)
                  tma_load_2d_pair(b_dst + sub * b_sub_bytes, tmap_x, fb, kx, trow);
              }
            }
            if (gr.on && sub < nsub)
              tma_gather4_pair(b_dst + sub * b_sub_bytes + lane * 512, &tx.m[0], fb,
                               (ks * kSub + sub) * kBK, gr.r[0], gr.r[1], gr.r[2], gr.r[3]);
          }
          if (armed) ++issued;  // drained at the end even if a later box never came
          if (!ok) break;
          if (++stage == nst) { stage = 0; phase ^= 1u; }
        }
      }
    }
    if (lane == 0) {
      if (leader) {
        for (int i = max(0, issued - nst); i < issued; ++i)
          mbar_wait_drain(full_bar + 8 * (i % nst), (i / nst) & 1, p.status);
      } else if (!ok) {
        // The follower cannot see its copies complete (they count on the
        // leader's barrier); after a give-up it leaves them time to land.
        const unsigned long long t0 = globaltimer_ns();
        while (globaltimer_ns() - t0 < 50000ull) {
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      // ---------------- MMA issuer (leader)
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int seq = 0; ok; ++seq) {
        if (tile_at(seq) < 0) break;
        if (!mbar_wait(tempty_bar + 8 * acc, acc_phase ^ 1u, wc)) { ok = false; break; }
        tc_fence_after_sync();
        const uint32_t d_tmem = tmem_base + acc * kAccCols;  // TMEM column c: chunk token c
        uint32_t idesc = 0;
        for (int ks = 0; ks < num_ks; ++ks) {
          if (!mbar_wait(full_bar + 8 * stage, phase, wc)) { ok = false; break; }
          if (ks == 0) idesc = idesc_bf16_f32(256, s_tile_n[seq % kTileRing]);
          // Descriptors built once per stage; a K step of 16 moves 32 bytes,
          // i.e. 2 in the descriptor's 16-byte address field (no carry out of
          // it: shared addresses stay below 256 KB).
          const uint32_t a_addr = base + stage * stage_bytes;
          const uint64_t da = smem_desc_sw128(a_addr);
          const uint64_t db = smem_desc_sw128(a_addr + kSub * kABytes);
          const uint32_t acc0 = ks != 0 ? 1u : 0u;
#pragma unroll
          for (int sub = 0; sub < kSub; ++sub) {
            if (sub == 0 || ks * kSub + sub < num_kb) {  // the last stage may hold fewer boxes
              const uint64_t das = da + sub * (kABytes >> 4), dbs = db + sub * (b_sub_bytes >> 4);
#pragma unroll
              for (int k = 0; k < kBK / 16; ++k)
                mma_bf16_pair(d_tmem, das + 2 * k, dbs + 2 * k, idesc, (sub | k) != 0 ? 1u : acc0);
            }
            // frees box `sub` of this stage in both CTAs (also when the box is
            // absent, so every box barrier completes one phase per stage), or
            // the whole stage after its last box
            if (kBoxRelease) mma_commit_pair(empty_box(sub, stage));
            else if (sub == kSub - 1) mma_commit_pair(empty_bar + 8 * stage);
          }
          if (++stage == nst) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        mma_commit_pair(tfull_bar + 8 * acc);     // accumulator ready in both CTAs
        if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
      }
      mma_commit_pair(drain_bar);
      mbar_wait_drain(drain_bar, 0, p.status);
    } else if (lane == 0) {
      // follower: the leader's last commit also arrives here once its MMAs are done
      mbar_wait_drain(drain_bar, 0, p.status);
    }
  } else if (warp >= kThreads / 32) {
    // ---------------- scheduler (dynamic schedule, leader, lane 0): takes
    // the next tile from the global counter and publishes it to both CTAs.
    // Its own thread waits out the atomic's round trip, so the producer's
    // barrier arrives (release operations) never wait for it.
    if (dyn && leader && lane == 0) {
      for (int seq = 0;; ++seq) {
        bool go = !*wc.abort_flag;
        if (go && seq >= *static_cast<volatile int*>(&s_prod_next) + kSchedAhead) {
          const unsigned long long t0 = globaltimer_ns();
          while (seq >= *static_cast<volatile int*>(&s_prod_next) + kSchedAhead) {
            if (*wc.abort_flag) { go = false; break; }
            if (globaltimer_ns() - t0 > wc.timeout_ns) { go = give_up(wc); break; }
            __nanosleep(64);
          }
        }
        int v = -1;
        if (go) {
          const unsigned got = atomicAdd(p.tile_ctr, 1u);
          if (got < static_cast<unsigned>(total_tiles)) v = static_cast<int>(got);
        }
        const int slot = seq % kTileRing;
        s_tau[slot] = v;
        st_shared_cluster_u32(mapa_shared(smem_u32(&s_tau[slot]), 1), static_cast<uint32_t>(v));
        mbar_arrive(tbar + 8 * slot);
        mbar_arrive_cluster(mapa_shared(tbar + 8 * slot, 1));
        if (v < 0) break;
      }
    }
  } else {
    // ---------------- epilogue: warps 2..5, TMEM lanes 32 (warp % 4) + lane
    const int q = warp & 3;
    const uint32_t tempty_leader = mapa_shared(tempty_bar, 0);
    int acc = 0;
    uint32_t acc_phase = 0;
    // After a wait gives up, the loop still runs to the end (later waits fail
    // at once; with the dynamic schedule, to the last tile published) with its
    // stores switched off.
    for (int seq = 0;; ++seq) {
      const int tau = tile_at_warp(seq);
      if (tau < 0) break;
      const Tile t = decode_tile(tau, sched);
      const bool live = __all_sync(0xffffffffu, mbar_wait(tfull_bar + 8 * acc, acc_phase, wc));
      tc_fence_after_sync();
      const uint32_t t_row = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * kAccCols;
      epilogue_tile<KIND>(t, t_row, live, p, q, lane, rank);
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) {
        if (leader) mbar_arrive(tempty_bar + 8 * acc);
        else mbar_arrive_cluster(tempty_leader + 8 * acc);
      }
      if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
    }
  }

  if (FUSED) fence_proxy_async_global();  // this phase's stores before later TMA reads
  tc_fence_before_sync();
  __syncthreads();
  cluster_sync();
  if (!FUSED && warp == 1) {
    __syncwarp();
    tc_fence_after_sync();
    tmem_dealloc_pair(tmem_base, kTmemCols);
  }
  // Dynamic schedule: the last CTA to leave (every CTA has taken its last
  // tile by now) resets the counters for the next launch.
  if (dyn && threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(p.exit_ctr, 1u) == gridDim.x - 1) {
      atomicExch(p.tile_ctr, 0u);
      atomicExch(p.exit_ctr, 0u);
      __threadfence();
    }
  }
}

// ---------------------------------------------------------------- host side

// W_gate_up [groups][2][I][d] viewed as (d, 16 rows, gate|up, I/16 row groups,
// groups): one box = 4 row groups, each 16 gate rows followed by the 16
// matching up rows (the interleaving the epilogue's shuffle relies on).
inline cudaError_t make_gate_up_weight_map(CUtensorMap* mw, const void* w_gate_up, int d, int I,
                                           int groups) {
  const uint64_t dims[5] = {static_cast<uint64_t>(d), 16, 2, static_cast<uint64_t>(I / 16),
                            static_cast<uint64_t>(groups)};
  const uint64_t strides[4] = {static_cast<uint64_t>(d) * 2, static_cast<uint64_t>(I) * d * 2,
                               16ull * d * 2, 2ull * I * d * 2};
  const uint32_t box[5] = {64, 16, 2, 4, 1};
  return make_bf16_map_nd(mw, w_gate_up, 5, dims, strides, box);
}

// Token-operand maps over a [rows, K] bf16 matrix, boxes of 8, 16, ..., 128 rows.
inline cudaError_t make_token_maps(TokenMapSet& mx, const void* a, int rows, int K) {
  for (int i = 0; i < kTokenMaps; ++i) {
    cudaError_t e = make_bf16_map(&mx.m[i], a, rows, K, (kUnit / 2) * (i + 1));
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

// Gate_up's token operand: boxes over a [rows, K] matrix, or, gathering, a
// one-row box over the unpermuted tokens in every slot; sets p's gather fields.
inline cudaError_t make_gate_up_token_maps(TokenMapSet& mx, Params& p, const void* a, int rows, int K,
                                    const TokenGather* g) {
  p.gather_perm = nullptr;
  if (!g) return make_token_maps(mx, a, rows, K);
  const cudaError_t e = make_bf16_map(&mx.m[0], g->src, g->src_rows, K, 1);
  if (e != cudaSuccess) return e;
  for (int i = 1; i < kTokenMaps; ++i) mx.m[i] = mx.m[0];
  p.gather_perm = g->perm;
  p.gather_div = g->div;
  p.gather_oob = g->src_rows;
  return cudaSuccess;
}

}  // namespace moe
