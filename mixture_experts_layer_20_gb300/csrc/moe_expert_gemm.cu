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
// read the same weight slab, which is then read from HBM once.
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
// Roles, per CTA (192 threads): warp 0 loads both operands with TMA into its
// own shared memory, counting the bytes of both CTAs on the leader's full
// barrier; warp 1 owns the tensor memory (512 columns: two accumulators of up
// to 256 fp32 columns) and, in the leader, one of its threads issues the MMAs
// and commits to both CTAs' barriers; warps 2-5 read the accumulator with
// tcgen05.ld and store the tile while the next one accumulates.  Every wait
// is bounded; on timeout a CTA records it, drains its copies in flight (and,
// in the leader, its MMAs), and both CTAs still meet at the final cluster
// barrier before freeing tensor memory.

#include <algorithm>
#include <mutex>

#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "moe_convert.cuh"
#include "moe_device.cuh"
#include "moe_internal.h"

namespace moe {
namespace {

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

__device__ __forceinline__ GatherRows gather_rows(const Params& p, int row0, int cnt, int lane) {
  GatherRows g;
  g.on = p.gather_perm != nullptr && 4 * lane < cnt;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int pos = row0 + 4 * lane + i;
    g.r[i] = g.on && pos < p.total_rows ? __ldg(p.gather_perm + pos) / p.gather_div : p.gather_oob;
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
__device__ __forceinline__ void build_schedule(const Params& p, int* s_off,
                                               int (*s_pre)[kMaxExperts + 1], int* s_half_max,
                                               int warp, int lane, int TOKCAP) {
  const int G = p.groups;
  for (int i = threadIdx.x; i <= G; i += blockDim.x)
    s_off[i] = p.offsets ? __ldg(p.offsets + i) : (i == 0 ? 0 : p.total_rows);
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

template <int KIND>
__device__ __forceinline__ void expert_gemm_body(const CUtensorMap& tmap_w, const TokenMapSet& tx,
                                                 const Params& p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ int s_off[kMaxExperts + 1];
  __shared__ int s_pre[2][kMaxExperts + 1];
  __shared__ alignas(8) uint64_t s_bar[2 * kMaxStagesAny + 5];
  __shared__ int s_half_max;
  __shared__ uint32_t s_tmem_base;
  __shared__ int s_abort;
  // Token count of the tile whose first stage the producer armed, by tile
  // sequence number mod kTileRing: the MMA issuer reads it after that stage's
  // full barrier instead of decoding the tile itself (it is at most
  // kMaxStagesAny stages, so as many tiles, behind the producer).
  __shared__ int s_tile_n[kTileRing];

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int pair = blockIdx.x >> 1;
  const int num_pairs = gridDim.x >> 1;

  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t full_bar = smem_u32(&s_bar[0]);
  const uint32_t empty_bar = smem_u32(&s_bar[kMaxStagesAny]);
  const uint32_t tfull_bar = smem_u32(&s_bar[2 * kMaxStagesAny]);
  const uint32_t tempty_bar = smem_u32(&s_bar[2 * kMaxStagesAny + 2]);
  const uint32_t drain_bar = smem_u32(&s_bar[2 * kMaxStagesAny + 4]);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kMaxStagesAny; ++s) {
      mbar_init(full_bar + 8 * s, 1);  // leader: counts both CTAs' bytes; unused in the follower
      mbar_init(empty_bar + 8 * s, 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull_bar + 8 * a, 1);
      mbar_init(tempty_bar + 8 * a, kEpiArrivals);
    }
    mbar_init(drain_bar, 1);
    s_abort = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmap_w);
#pragma unroll
    for (int i = 0; i < kTokenMaps; ++i) tma_prefetch_desc(&tx.m[i]);
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(&s_tmem_base), kTmemCols);
    tmem_relinquish_pair();
  }

  pdl_wait_and_release();

  build_schedule(p, s_off, s_pre, &s_half_max, warp, lane, kTokMax);
  tc_fence_before_sync();
  __syncthreads();
  cluster_sync();  // the peer's barriers are initialised before any remote arrive
  tc_fence_after_sync();

  const uint32_t tmem_base = s_tmem_base;
  const Sched sched = make_sched(p, s_off, s_pre);
  const int total_tiles = static_cast<int>(sched.n_all);
  const int num_kb = p.K / kBK;                   // 64-wide K boxes
  const WaitCtx wc{p.timeout_ns, p.status, &s_abort};
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
    for (int tau = pair; tau < total_tiles && ok; tau += num_pairs, ++seq) {
      const Tile t = decode_tile(tau, sched);
      const int half = t.n / 2;  // token rows per CTA: 8, 16, ..., 128
      const CUtensorMap* tmap_x = &tx.m[t.n / kUnit - 1];
      const uint32_t tx_bytes = kABytes + half * 128;  // per CTA
      const int trow = t.tok0 + rank * half;  // this CTA's first token row
      const int wrow = KIND == kGateUp ? t.slab * 128 + rank * 64
                                       : t.e * p.w_rows_per_group + t.slab * 256 + rank * 128;
      const GatherRows gr = gather_rows(p, trow, half, lane);
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
            // gate_up: one box holds 4 groups of {16 gate rows, the 16 matching up rows}
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
      int seq = 0;
      for (int tau = pair; tau < total_tiles && ok; tau += num_pairs, ++seq) {
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
          }
          mma_commit_pair(empty_bar + 8 * stage);  // frees this stage in both CTAs
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
  } else {
    // ---------------- epilogue: warps 2..5, TMEM lanes 32 (warp % 4) + lane
    const int q = warp & 3;
    const uint32_t tempty_leader = mapa_shared(tempty_bar, 0);
    int acc = 0;
    uint32_t acc_phase = 0;
    // After a wait gives up, the loop still runs to the end (later waits fail
    // at once) with its stores switched off.
    for (int tau = pair; tau < total_tiles; tau += num_pairs) {
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

  tc_fence_before_sync();
  __syncthreads();
  cluster_sync();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after_sync();
    tmem_dealloc_pair(tmem_base, kTmemCols);
  }
}

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

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    moe_gate_up_swiglu_kernel(const __grid_constant__ CUtensorMap tmap_w,
                              const __grid_constant__ TokenMapSet tx, const Params p) {
  expert_gemm_body<kGateUp>(tmap_w, tx, p);
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    moe_down_kernel(const __grid_constant__ CUtensorMap tmap_w,
                    const __grid_constant__ TokenMapSet tx, const Params p) {
  expert_gemm_body<kDown>(tmap_w, tx, p);
}

typedef void (*ExpertKernel)(const CUtensorMap, const TokenMapSet, const Params);

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

// Token-operand maps over a [rows, K] bf16 matrix, boxes of 8, 16, ..., 128 rows.
cudaError_t make_token_maps(TokenMapSet& mx, const void* a, int rows, int K) {
  for (int i = 0; i < kTokenMaps; ++i) {
    cudaError_t e = make_bf16_map(&mx.m[i], a, rows, K, (kUnit / 2) * (i + 1));
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

// Gate_up's token operand: boxes over a [rows, K] matrix, or, gathering, a
// one-row box over the unpermuted tokens in every slot; sets p's gather fields.
cudaError_t make_gate_up_token_maps(TokenMapSet& mx, Params& p, const void* a, int rows, int K,
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
                               unsigned long long timeout_ns, const TokenGather* gather) {
  const int groups = offsets ? E : 1;
  const long long chunks_bound =
      offsets ? rows / kTokMax + std::min(E, rows) : (rows + kTokMax - 1) / kTokMax;

  // W_gate_up [groups][2][I][d] viewed as (d, 16 rows, gate|up, I/16 row groups, groups): one
  // box = 4 row groups, each 16 gate rows followed by the 16 matching up rows
  CUtensorMap mw;
  TokenMapSet mx;
  const uint64_t dims[5] = {static_cast<uint64_t>(d), 16, 2, static_cast<uint64_t>(I / 16),
                            static_cast<uint64_t>(groups)};
  const uint64_t strides[4] = {static_cast<uint64_t>(d) * 2, static_cast<uint64_t>(I) * d * 2,
                               16ull * d * 2, 2ull * I * d * 2};
  const uint32_t box[5] = {64, 16, 2, 4, 1};
  Params p{};
  cudaError_t e = make_bf16_map_nd(&mw, w_gate_up, 5, dims, strides, box);
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
  e = launch_expert(s, offsets ? "moe_gate_up_swiglu" : "moe_shared_gate_up_swiglu",
                    moe_gate_up_swiglu_kernel, 0, mw, mx, p, chunks_bound * p.slabs);
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
  q.status = status;
  q.timeout_ns = timeout_ns;
  return launch_expert(s, offsets ? "moe_down" : "moe_shared_down", moe_down_kernel, 1, mw2, mx2,
                       q, chunks_bound * q.slabs);
}

cudaError_t launch_grouped_ffn_quant(cudaStream_t s, int fmt, const void* a,
                                     const int32_t* offsets, int rows, int d, int E, int I,
                                     const uint8_t* codes_gate_up, const uint8_t* scales_gate_up,
                                     const float* tscale_gate_up, const uint8_t* codes_down,
                                     const uint8_t* scales_down, const float* tscale_down,
                                     void* h, void* y, unsigned* status,
                                     unsigned long long timeout_ns) {
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
