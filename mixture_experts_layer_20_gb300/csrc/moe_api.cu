// C ABI of the MoE layer: argument checks, workspace layout, the launch
// sequence of moe_forward, device status, launch counting and tracing.

#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "../../include/moe.h"
#include "moe_internal.h"

namespace moe {
namespace {

constexpr size_t kAlign = 256;
// Quantised expert weights: the warp-level small-M kernels serve layers with
// at most this many token rows per expert on average (decode batches).  They
// take 8 tokens per pass over an expert's weights, so an expert with more rows
// reads its weights again; measured at 16 rows per expert, the second pass
// came from DRAM (the other warps' streams evict it from L2).
constexpr long long kSmallMRowsPerExpert = 8;
// single_launch: decode-sized layers, at most this many rows per expert on average.
constexpr long long kSingleLaunchRowsPerExpert = 16;
constexpr unsigned long long kDefaultTimeoutNs = 2000000000ull;

std::atomic<unsigned long long> g_launches{0};
// Launches made by this thread, and whether it is capturing a graph (then no
// tracing events are recorded: they would become graph nodes).
thread_local unsigned long long t_launches = 0;
thread_local bool t_capturing = false;
std::atomic<unsigned long long> g_timeout_ns{kDefaultTimeoutNs};
thread_local std::string g_last_error;

size_t align_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

moe_status_t fail(moe_status_t st, const std::string& msg) {
  g_last_error = msg;
  return st;
}

moe_status_t cuda_fail(cudaError_t e, const char* where) {
  return fail(MOE_ERR_CUDA, std::string(where) + ": " + cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// --- tracing ---------------------------------------------------------------

struct Record {
  const char* name;
  cudaEvent_t start, stop;
};

std::mutex g_prof_mu;
bool g_prof_on = false;
std::string g_prof_only;  // trace only launches of this kernel name (empty: all)
std::vector<Record> g_records;
std::vector<cudaEvent_t> g_event_pool;
constexpr size_t kMaxRecords = 1 << 16;

cudaEvent_t take_event() {
  if (!g_event_pool.empty()) {
    cudaEvent_t e = g_event_pool.back();
    g_event_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}

// --- shape checks -------------------------------------------------------------

moe_status_t check_shapes(int T, int d, int E, int I, int top_k) {
  if (T < 0 || d <= 0 || E <= 0 || I <= 0 || top_k <= 0)
    return fail(MOE_ERR_INVALID_ARG, "T must be >= 0 and d, E, I, top_k > 0");
  if (d % 64 || I % 64) return fail(MOE_ERR_UNSUPPORTED, "d and I must be multiples of 64");
  if (E > kMaxExperts) return fail(MOE_ERR_UNSUPPORTED, "at most 256 experts");
  if (top_k > E || top_k > kMaxTopK) return fail(MOE_ERR_INVALID_ARG, "top_k must be <= min(E, 8)");
  if (static_cast<long long>(T) * top_k > (1LL << 30))
    return fail(MOE_ERR_UNSUPPORTED, "T * top_k must be <= 2^30");
  return MOE_OK;
}

struct Layout {
  size_t status, logits, ids, gates, counts, offsets, perm, slot_pos, chunk, x_perm, h, h_shared,
      y, y_shared, x_stage, out_stage, act_x, act_x_scales, act_h, act_h_scales, total;
};

// y_fp32: the expert outputs y and y_shared kept in fp32 (else fp16).
// act8: room for the MXFP8 tokens of the W8A8 expert GEMMs (x and h).
Layout forward_layout(int T, int d, int E, int I, int top_k, int I_shared, bool y_fp32 = false,
                      bool act8 = false) {
  const size_t n = static_cast<size_t>(T) * top_k;
  const size_t nchunks = (n + kPermuteChunk - 1) / kPermuteChunk;
  Layout L{};
  size_t off = 0;
  auto take = [&](size_t bytes) { const size_t at = off; off += align_up(bytes); return at; };
  L.status = take(kAlign);
  // decode-sized layers may run as one launch, whose router keeps partial
  // sums over 128-wide ranges of d (four times the 512-wide ones)
  const bool decode_sized = d % 128 == 0 && n <= static_cast<size_t>(kPermuteSmallMax) &&
                            n <= static_cast<size_t>(kSingleLaunchRowsPerExpert) * E;
  L.logits = take(decode_sized ? std::max(router_partial_bytes(T, d, E), fused_partial_bytes(T, d, E))
                               : router_partial_bytes(T, d, E));
  L.ids = take(n * 4);
  L.gates = take(n * 4);
  L.counts = take(static_cast<size_t>(E) * 4);
  L.offsets = take(static_cast<size_t>(E + 1) * 4);
  L.perm = take(n * 4);
  L.slot_pos = take(n * 4);
  L.chunk = take(nchunks * E * 4);
  L.x_perm = take(n * d * 2);
  L.h = take(n * I * 2);
  L.h_shared = take(static_cast<size_t>(T) * I_shared * 2);
  const size_t ybytes = y_fp32 ? 4 : 2;
  L.y = take(n * d * ybytes);
  L.y_shared = take(I_shared ? static_cast<size_t>(T) * d * ybytes : 0);
  L.x_stage = take(static_cast<size_t>(T) * d * 2);
  L.out_stage = take(static_cast<size_t>(T) * d * 2);
  L.act_x = take(act8 ? static_cast<size_t>(T) * d : 0);
  L.act_x_scales = take(act8 ? static_cast<size_t>(T) * d / 32 : 0);
  L.act_h = take(act8 ? n * I : 0);
  L.act_h_scales = take(act8 ? n * I / 32 : 0);
  L.total = off;
  return L;
}

// Single-step calls use the workspace from offset 0: status word, then scratch.
size_t permute_ws_need(int n, int E) {
  const size_t nchunks = (static_cast<size_t>(n) + kPermuteChunk - 1) / kPermuteChunk;
  return kAlign + align_up(nchunks * E * 4);
}
size_t ffn_ws_need(int rows, int I) { return kAlign + align_up(static_cast<size_t>(rows) * I * 2); }

unsigned* status_word(void* ws) { return static_cast<unsigned*>(ws); }

}  // namespace

KernelScope::KernelScope(cudaStream_t stream, const char* name) : stream_(stream), slot_(-1) {
  g_launches.fetch_add(1, std::memory_order_relaxed);
  ++t_launches;
  if (t_capturing) return;
  std::lock_guard<std::mutex> lock(g_prof_mu);
  if (!g_prof_on || g_records.size() >= kMaxRecords) return;
  if (!g_prof_only.empty() && g_prof_only != name) return;
  Record r{name, take_event(), take_event()};
  if (!r.start || !r.stop) return;
  cudaEventRecord(r.start, stream_);
  g_records.push_back(r);
  slot_ = static_cast<int>(g_records.size()) - 1;
}

KernelScope::~KernelScope() {
  if (slot_ < 0) return;
  std::lock_guard<std::mutex> lock(g_prof_mu);
  cudaEventRecord(g_records[slot_].stop, stream_);
}

void set_last_error(const std::string& msg) { g_last_error = msg; }

int device_sm_count() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
  if (!cached[dev]) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    cached[dev] = n > 0 ? n : 1;
  }
  return cached[dev];
}

namespace {

// The kernels are built for sm_103a only.
moe_status_t check_device() {
  static int ok_cache[64] = {0};  // 0 unknown, 1 ok, 2 unsupported
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev >= 0 && dev < 64 && ok_cache[dev] == 1) return MOE_OK;
  int major = 0, minor = 0;
  cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  const bool ok = major == 10 && minor == 3;
  if (dev >= 0 && dev < 64) ok_cache[dev] = ok ? 1 : 2;
  if (!ok) {
    char buf[96];
    std::snprintf(buf, sizeof buf, "device is sm_%d%d; this library is built for sm_103a", major,
                  minor);
    return fail(MOE_ERR_UNSUPPORTED, buf);
  }
  return MOE_OK;
}

moe_status_t route_impl(const moe_bf16* x, const moe_bf16* w_router, const float* bias,
                        int bias_selection_only, int T, int d, int E, int top_k, int32_t* ids,
                        float* gates, float* partial, unsigned* status, cudaStream_t s) {
  cudaError_t e = launch_router(s, x, w_router, bias, bias_selection_only, T, d, E, top_k, ids,
                                gates, partial, status, g_timeout_ns.load());
  return e == cudaSuccess ? MOE_OK : cuda_fail(e, "router launch");
}

}  // namespace
}  // namespace moe

using namespace moe;

struct moe_graph_s {
  cudaGraphExec_t exec;
  unsigned long long kernels;  // kernels per replay
};

extern "C" {

size_t moe_workspace_size(int T, int d, int E, int I, int top_k, int I_shared) {
  if (T < 0 || d <= 0 || E <= 0 || I <= 0 || top_k <= 0 || I_shared < 0) return 0;
  return forward_layout(T, d, E, I, top_k, I_shared).total;
}

size_t moe_workspace_size_ex(int T, int d, int E, int I, int top_k,
                             const moe_forward_ext_t* ext) {
  const int I_shared = ext ? ext->I_shared : 0;
  if (T < 0 || d <= 0 || E <= 0 || I <= 0 || top_k <= 0 || I_shared < 0) return 0;
  return forward_layout(T, d, E, I, top_k, I_shared, ext && ext->y_fp32, ext && ext->act_mxfp8)
      .total;
}

static moe_status_t workspace_layout(int T, int d, int E, int I, int top_k, int I_shared,
                                     bool y_fp32, bool act8, moe_workspace_layout_t* out) {
  if (!out || T < 0 || d <= 0 || E <= 0 || I <= 0 || top_k <= 0 || I_shared < 0)
    return fail(MOE_ERR_INVALID_ARG, "bad arguments to moe_workspace_layout");
  const Layout L = forward_layout(T, d, E, I, top_k, I_shared, y_fp32, act8);
  out->status = L.status;
  out->router_logits = L.logits;
  out->topk_ids = L.ids;
  out->topk_gates = L.gates;
  out->expert_counts = L.counts;
  out->expert_offsets = L.offsets;
  out->perm = L.perm;
  out->slot_pos = L.slot_pos;
  out->chunk_table = L.chunk;
  out->x_perm = L.x_perm;
  out->h = L.h;
  out->h_shared = L.h_shared;
  out->y = L.y;
  out->y_shared = L.y_shared;
  out->x_stage = L.x_stage;
  out->out_stage = L.out_stage;
  out->act_x = L.act_x;
  out->act_x_scales = L.act_x_scales;
  out->act_h = L.act_h;
  out->act_h_scales = L.act_h_scales;
  out->total = L.total;
  return MOE_OK;
}

moe_status_t moe_workspace_layout(int T, int d, int E, int I, int top_k, int I_shared,
                                  moe_workspace_layout_t* out) {
  return workspace_layout(T, d, E, I, top_k, I_shared, false, false, out);
}

moe_status_t moe_workspace_layout_ex(int T, int d, int E, int I, int top_k,
                                     const moe_forward_ext_t* ext, moe_workspace_layout_t* out) {
  return workspace_layout(T, d, E, I, top_k, ext ? ext->I_shared : 0, ext && ext->y_fp32,
                          ext && ext->act_mxfp8, out);
}

moe_status_t moe_workspace_init(void* ws, size_t ws_bytes, moe_stream_t stream) {
  if (!ws || ws_bytes < kAlign || !aligned16(ws))
    return fail(MOE_ERR_WORKSPACE, "workspace must be >= 256 bytes and 16-byte aligned");
  cudaError_t e = cudaMemsetAsync(ws, 0, kAlign, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MOE_OK : cuda_fail(e, "cudaMemsetAsync");
}

moe_status_t moe_route(const moe_bf16* x, const moe_bf16* w_router, const float* router_bias,
                       int T, int d, int E, int top_k, int32_t* topk_ids, float* topk_gates,
                       void* ws, size_t ws_bytes, moe_stream_t stream) {
  return moe_route_ex(x, w_router, router_bias, 0, T, d, E, top_k, topk_ids, topk_gates, ws,
                      ws_bytes, stream);
}

moe_status_t moe_route_ex(const moe_bf16* x, const moe_bf16* w_router, const float* router_bias,
                          int bias_selection_only, int T, int d, int E, int top_k,
                          int32_t* topk_ids, float* topk_gates, void* ws, size_t ws_bytes,
                          moe_stream_t stream) {
  moe_status_t st = check_shapes(T, d, E, 64, top_k);
  if (st != MOE_OK) return st;
  if (T == 0) return MOE_OK;
  if (!x || !w_router || !topk_ids || !topk_gates || !ws)
    return fail(MOE_ERR_INVALID_ARG, "moe_route: null pointer");
  if (!aligned16(x) || !aligned16(w_router) || !aligned16(ws))
    return fail(MOE_ERR_INVALID_ARG, "moe_route: pointers must be 16-byte aligned");
  if (ws_bytes < kAlign + router_partial_bytes(T, d, E))
    return fail(MOE_ERR_WORKSPACE, "moe_route: workspace too small");
  if ((st = check_device()) != MOE_OK) return st;
  float* partial = reinterpret_cast<float*>(static_cast<char*>(ws) + kAlign);
  return route_impl(x, w_router, router_bias, bias_selection_only, T, d, E, top_k, topk_ids,
                    topk_gates, partial, status_word(ws), reinterpret_cast<cudaStream_t>(stream));
}

moe_status_t moe_permute(const int32_t* topk_ids, const moe_bf16* x, int T, int d, int E,
                         int top_k, int32_t* expert_counts, int32_t* expert_offsets,
                         int32_t* perm, int32_t* slot_pos, moe_bf16* x_perm, void* ws,
                         size_t ws_bytes, moe_stream_t stream) {
  moe_status_t st = check_shapes(T, d, E, 64, top_k);
  if (st != MOE_OK) return st;
  if (T == 0) return MOE_OK;
  if (!topk_ids || !expert_counts || !expert_offsets || !perm || !slot_pos || !ws)
    return fail(MOE_ERR_INVALID_ARG, "moe_permute: null pointer");
  if (x && (!x_perm || !aligned16(x) || !aligned16(x_perm)))
    return fail(MOE_ERR_INVALID_ARG, "moe_permute: x and x_perm must be 16-byte aligned");
  if (!aligned16(ws) || ws_bytes < permute_ws_need(T * top_k, E))
    return fail(MOE_ERR_WORKSPACE, "moe_permute: workspace too small");
  if ((st = check_device()) != MOE_OK) return st;
  int32_t* table = reinterpret_cast<int32_t*>(static_cast<char*>(ws) + kAlign);
  cudaError_t e = launch_permute(reinterpret_cast<cudaStream_t>(stream), topk_ids, x, T, d, E,
                                 top_k, expert_counts, expert_offsets, perm, slot_pos, x_perm,
                                 table, status_word(ws));
  return e == cudaSuccess ? MOE_OK : cuda_fail(e, "permute launch");
}

moe_status_t moe_expert_ffn(const moe_bf16* x_perm, const int32_t* expert_offsets,
                            const moe_bf16* w_gate_up, const moe_bf16* w_down, int rows, int d,
                            int E, int I, moe_f16* y, void* ws, size_t ws_bytes,
                            moe_stream_t stream) {
  moe_status_t st = check_shapes(rows, d, E, I, 1);
  if (st != MOE_OK) return st;
  if (rows == 0) return MOE_OK;
  if (!x_perm || !expert_offsets || !w_gate_up || !w_down || !y || !ws)
    return fail(MOE_ERR_INVALID_ARG, "moe_expert_ffn: null pointer");
  if (!aligned16(x_perm) || !aligned16(w_gate_up) || !aligned16(w_down) || !aligned16(y))
    return fail(MOE_ERR_INVALID_ARG, "moe_expert_ffn: pointers must be 16-byte aligned");
  if (!aligned16(ws) || ws_bytes < ffn_ws_need(rows, I))
    return fail(MOE_ERR_WORKSPACE, "moe_expert_ffn: workspace too small");
  if ((st = check_device()) != MOE_OK) return st;
  void* h = static_cast<char*>(ws) + kAlign;
  cudaError_t e = launch_grouped_ffn(reinterpret_cast<cudaStream_t>(stream), x_perm,
                                     expert_offsets, rows, d, E, I, w_gate_up, w_down, h, y,
                                     status_word(ws), g_timeout_ns.load(), nullptr, false,
                                     status_word(ws));
  return e == cudaSuccess ? MOE_OK : cuda_fail(e, "expert FFN launch");
}

moe_status_t moe_combine(const moe_f16* y, const int32_t* slot_pos, const float* topk_gates,
                         const moe_f16* y_shared, int T, int d, int top_k, moe_bf16* out, void* ws,
                         size_t ws_bytes, moe_stream_t stream) {
  moe_status_t st = check_shapes(T, d, top_k, 64, top_k);
  if (st != MOE_OK) return st;
  if (T == 0) return MOE_OK;
  if (!y || !slot_pos || !topk_gates || !out || !ws)
    return fail(MOE_ERR_INVALID_ARG, "moe_combine: null pointer");
  if (!aligned16(y) || !aligned16(out) || (y_shared && !aligned16(y_shared)))
    return fail(MOE_ERR_INVALID_ARG, "moe_combine: pointers must be 16-byte aligned");
  if (!aligned16(ws) || ws_bytes < kAlign)
    return fail(MOE_ERR_WORKSPACE, "moe_combine: workspace too small");
  if ((st = check_device()) != MOE_OK) return st;
  cudaError_t e = launch_combine(reinterpret_cast<cudaStream_t>(stream), y, slot_pos, topk_gates,
                                 y_shared, T, d, top_k, out, status_word(ws));
  return e == cudaSuccess ? MOE_OK : cuda_fail(e, "combine launch");
}

namespace {

// MXFP8 expert weights (codes and scales); null for bf16 weights.
// Quantised expert weights: fmt 0 MXFP8, 1 NVFP4 (tensor scales used).
struct MxWeights {
  int fmt;
  const uint8_t *codes_gate_up, *scales_gate_up, *codes_down, *scales_down;
  const float *tscale_gate_up, *tscale_down;
};

moe_status_t forward_impl(const moe_bf16* x, const moe_bf16* w_router,
                          const moe_bf16* w_gate_up, const moe_bf16* w_down, const MxWeights* mx,
                          int T, int d, int E, int I, int top_k, moe_bf16* out, void* ws,
                          size_t ws_bytes, moe_stream_t stream, const moe_forward_ext_t* ext) {
  moe_status_t st = check_shapes(T, d, E, I, top_k);
  if (st != MOE_OK) return st;
  if (mx && mx->fmt == 0 && (d % 128 || I % 128))
    return fail(MOE_ERR_UNSUPPORTED, "MXFP8 weights need d and I multiples of 128");
  if (mx && mx->fmt == 1 && (d % 256 || I % 256))
    return fail(MOE_ERR_UNSUPPORTED, "NVFP4 weights need d and I multiples of 256");
  const float* bias = ext ? ext->router_bias : nullptr;
  const int bias_sel = ext ? ext->bias_selection_only : 0;
  const bool single = ext && ext->single_launch;
  const bool y32 = ext && ext->y_fp32;
  const bool act8 = ext && ext->act_mxfp8;
  const int I_shared = ext ? ext->I_shared : 0;
  const moe_bf16* wgu_s = ext ? ext->w_gate_up_shared : nullptr;
  const moe_bf16* wd_s = ext ? ext->w_down_shared : nullptr;
  if (I_shared < 0 || I_shared % 64) return fail(MOE_ERR_UNSUPPORTED, "I_shared must be a multiple of 64");
  if (I_shared && (!wgu_s || !wd_s)) return fail(MOE_ERR_INVALID_ARG, "shared expert weights missing");
  if (T == 0) return MOE_OK;
  if (!x || !w_router || !w_gate_up || !w_down || !out || !ws)
    return fail(MOE_ERR_INVALID_ARG, "moe_forward: null pointer");
  if (!aligned16(x) || !aligned16(w_router) || !aligned16(w_gate_up) || !aligned16(w_down) ||
      !aligned16(out) || !aligned16(ws) || (I_shared && (!aligned16(wgu_s) || !aligned16(wd_s))))
    return fail(MOE_ERR_INVALID_ARG, "moe_forward: pointers must be 16-byte aligned");
  const Layout L = forward_layout(T, d, E, I, top_k, I_shared, y32, act8);
  if (ws_bytes < L.total) return fail(MOE_ERR_WORKSPACE, "moe_forward: workspace too small");
  if (single && y32)
    return fail(MOE_ERR_UNSUPPORTED, "single_launch keeps y in fp16 (y_fp32 unsupported)");
  if (single && (mx || I_shared || d % 128 || I % 128 ||
                 static_cast<long long>(T) * top_k > kPermuteSmallMax ||
                 static_cast<long long>(T) * top_k > kSingleLaunchRowsPerExpert * E))
    return fail(MOE_ERR_UNSUPPORTED,
                "single_launch needs bf16 expert weights, no shared expert, d and I multiples of "
                "128, T*top_k <= 4096 and at most 16 rows per expert on average");
  if (act8 && !(mx && mx->fmt == 0 && !I_shared && !single && d % 256 == 0 && I % 256 == 0 &&
                static_cast<long long>(T) * top_k <= kSmallMRowsPerExpert * static_cast<long long>(E)))
    return fail(MOE_ERR_UNSUPPORTED,
                "act_mxfp8 needs MXFP8 expert weights, decode sizes (at most 8 rows per expert "
                "on average, d and I multiples of 256) and no shared expert");
  if ((st = check_device()) != MOE_OK) return st;

  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  char* w = static_cast<char*>(ws);
  unsigned* status = status_word(ws);
  int32_t* ids = reinterpret_cast<int32_t*>(w + L.ids);
  float* gates = reinterpret_cast<float*>(w + L.gates);
  int32_t* counts = reinterpret_cast<int32_t*>(w + L.counts);
  int32_t* offsets = reinterpret_cast<int32_t*>(w + L.offsets);
  int32_t* perm = reinterpret_cast<int32_t*>(w + L.perm);
  int32_t* slot_pos = reinterpret_cast<int32_t*>(w + L.slot_pos);
  int32_t* table = reinterpret_cast<int32_t*>(w + L.chunk);
  void* h = w + L.h;
  void* y = w + L.y;
  const unsigned long long tmo = g_timeout_ns.load();
  const int rows = T * top_k;

  float* partial = reinterpret_cast<float*>(w + L.logits);
  if (single) {
    FusedLayer F{};
    F.x = x;
    F.w_router = w_router;
    F.bias = bias;
    F.bias_selection_only = bias_sel;
    F.w_gate_up = w_gate_up;
    F.w_down = w_down;
    F.T = T;
    F.d = d;
    F.E = E;
    F.I = I;
    F.k = top_k;
    F.partial = partial;
    F.ids = ids;
    F.gates = gates;
    F.counts = counts;
    F.offsets = offsets;
    F.perm = perm;
    F.slot_pos = slot_pos;
    F.h = h;
    F.y = y;
    F.out = out;
    F.status = status;
    F.timeout_ns = tmo;
    const cudaError_t fe = launch_decode_fused(s, F);
    return fe == cudaSuccess ? MOE_OK : cuda_fail(fe, "single-launch layer");
  }
  if ((st = route_impl(x, w_router, bias, bias_sel, T, d, E, top_k, ids, gates, partial, status,
                       s)) != MOE_OK)
    return st;
  // Few rows per expert (decode): the bf16 gate_up GEMM gathers its token
  // rows from x through perm (four rows per TMA gather), so no permuted copy
  // of x is written.  Many rows: one TMA box per K box of x_perm loads faster
  // than that many gathers.
  // Quantised weights with few rows per expert (decode) take the warp-level
  // small-M kernels, which read the token rows from x through perm.
  void* x_perm = w + L.x_perm;
  const bool small_m = mx && rows <= kSmallMRowsPerExpert * static_cast<long long>(E) &&
                       d % 256 == 0 && I % 256 == 0;
  const bool gather_rows = small_m || (!mx && rows <= 128LL * E);
  cudaError_t e = launch_permute(s, ids, gather_rows ? nullptr : x, T, d, E, top_k, counts,
                                 offsets, perm, slot_pos, x_perm, table, status);
  if (e != cudaSuccess) return cuda_fail(e, "permute launch");
  const TokenGather gather{x, perm, top_k, T};
  if (act8)
    e = launch_grouped_ffn_smallm_a8(
        s, x, T, perm, top_k, offsets, rows, d, E, I, mx->codes_gate_up, mx->scales_gate_up,
        mx->codes_down, mx->scales_down, reinterpret_cast<uint8_t*>(w + L.act_x),
        reinterpret_cast<uint8_t*>(w + L.act_x_scales), h, reinterpret_cast<uint8_t*>(w + L.act_h),
        reinterpret_cast<uint8_t*>(w + L.act_h_scales), y, status, y32);
  else if (small_m)
    e = launch_grouped_ffn_smallm(s, mx->fmt == 0 ? 1 : 2, x, perm, top_k, offsets, rows, d, E, I,
                                  mx->codes_gate_up, mx->scales_gate_up, mx->tscale_gate_up,
                                  mx->codes_down, mx->scales_down, mx->tscale_down, h, y, status,
                                  y32);
  else if (mx)
    e = launch_grouped_ffn_quant(s, mx->fmt, x_perm, offsets, rows, d, E, I, mx->codes_gate_up,
                                 mx->scales_gate_up, mx->tscale_gate_up, mx->codes_down,
                                 mx->scales_down, mx->tscale_down, h, y, status, tmo, y32);
  else
    e = launch_grouped_ffn(s, x_perm, offsets, rows, d, E, I, w_gate_up, w_down, h, y, status,
                           tmo, gather_rows ? &gather : nullptr, y32, status);
  if (e != cudaSuccess) return cuda_fail(e, "expert FFN launch");
  void* y_shared = nullptr;
  if (I_shared) {
    y_shared = w + L.y_shared;
    e = launch_grouped_ffn(s, x, nullptr, T, d, 1, I_shared, wgu_s, wd_s, w + L.h_shared,
                           y_shared, status, tmo, nullptr, y32, status);
    if (e != cudaSuccess) return cuda_fail(e, "shared expert launch");
  }
  e = launch_combine(s, y, slot_pos, gates, y_shared, T, d, top_k, out, status, y32);
  return e == cudaSuccess ? MOE_OK : cuda_fail(e, "combine launch");
}

}  // namespace

moe_status_t moe_forward_ex(const moe_bf16* x, const moe_bf16* w_router,
                            const moe_bf16* w_gate_up, const moe_bf16* w_down, int T, int d,
                            int E, int I, int top_k, moe_bf16* out, void* ws, size_t ws_bytes,
                            moe_stream_t stream, const moe_forward_ext_t* ext) {
  return forward_impl(x, w_router, w_gate_up, w_down, nullptr, T, d, E, I, top_k, out, ws,
                      ws_bytes, stream, ext);
}

moe_status_t moe_forward_mxfp8(const moe_bf16* x, const moe_bf16* w_router,
                               const uint8_t* codes_gate_up, const uint8_t* scales_gate_up,
                               const uint8_t* codes_down, const uint8_t* scales_down, int T,
                               int d, int E, int I, int top_k, moe_bf16* out, void* ws,
                               size_t ws_bytes, moe_stream_t stream,
                               const moe_forward_ext_t* ext) {
  if (T > 0 && (!codes_gate_up || !scales_gate_up || !codes_down || !scales_down ||
                !aligned16(codes_gate_up) || !aligned16(scales_gate_up) ||
                !aligned16(codes_down) || !aligned16(scales_down)))
    return fail(MOE_ERR_INVALID_ARG, "moe_forward_mxfp8: null or unaligned weight pointer");
  const MxWeights mx{0, codes_gate_up, scales_gate_up, codes_down, scales_down, nullptr, nullptr};
  // the bf16 weight pointers are not read on this path; pass the codes to pass the null checks
  return forward_impl(x, w_router, reinterpret_cast<const moe_bf16*>(codes_gate_up),
                      reinterpret_cast<const moe_bf16*>(codes_down), &mx, T, d, E, I, top_k, out,
                      ws, ws_bytes, stream, ext);
}

moe_status_t moe_forward_nvfp4(const moe_bf16* x, const moe_bf16* w_router,
                               const uint8_t* codes_gate_up, const uint8_t* scales_gate_up,
                               const float* tscale_gate_up, const uint8_t* codes_down,
                               const uint8_t* scales_down, const float* tscale_down, int T,
                               int d, int E, int I, int top_k, moe_bf16* out, void* ws,
                               size_t ws_bytes, moe_stream_t stream,
                               const moe_forward_ext_t* ext) {
  if (T > 0 && (!codes_gate_up || !scales_gate_up || !codes_down || !scales_down ||
                !tscale_gate_up || !tscale_down || !aligned16(codes_gate_up) ||
                !aligned16(scales_gate_up) || !aligned16(codes_down) || !aligned16(scales_down)))
    return fail(MOE_ERR_INVALID_ARG, "moe_forward_nvfp4: null or unaligned weight pointer");
  const MxWeights mx{1, codes_gate_up, scales_gate_up, codes_down, scales_down, tscale_gate_up,
                     tscale_down};
  // the bf16 weight pointers are not read on this path; pass the codes to pass the null checks
  return forward_impl(x, w_router, reinterpret_cast<const moe_bf16*>(codes_gate_up),
                      reinterpret_cast<const moe_bf16*>(codes_down), &mx, T, d, E, I, top_k, out,
                      ws, ws_bytes, stream, ext);
}

moe_status_t moe_forward(const moe_bf16* x, const moe_bf16* w_router, const moe_bf16* w_gate_up,
                         const moe_bf16* w_down, int T, int d, int E, int I, int top_k,
                         moe_bf16* out, void* ws, size_t ws_bytes, moe_stream_t stream) {
  return moe_forward_ex(x, w_router, w_gate_up, w_down, T, d, E, I, top_k, out, ws, ws_bytes,
                        stream, nullptr);
}

moe_status_t moe_forward_host(const moe_bf16* x_host, const moe_bf16* w_router,
                              const moe_bf16* w_gate_up, const moe_bf16* w_down, int T, int d,
                              int E, int I, int top_k, moe_bf16* out_host, void* ws,
                              size_t ws_bytes, moe_stream_t stream, const moe_forward_ext_t* ext) {
  moe_status_t st = check_shapes(T, d, E, I, top_k);
  if (st != MOE_OK) return st;
  if (T == 0) return MOE_OK;
  if (!x_host || !out_host || !ws) return fail(MOE_ERR_INVALID_ARG, "moe_forward_host: null pointer");
  const int I_shared = ext ? ext->I_shared : 0;
  const Layout L =
      forward_layout(T, d, E, I, top_k, I_shared, ext && ext->y_fp32, ext && ext->act_mxfp8);
  if (ws_bytes < L.total || !aligned16(ws))
    return fail(MOE_ERR_WORKSPACE, "moe_forward_host: workspace too small");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  char* w = static_cast<char*>(ws);
  moe_bf16* x_dev = reinterpret_cast<moe_bf16*>(w + L.x_stage);
  moe_bf16* out_dev = reinterpret_cast<moe_bf16*>(w + L.out_stage);
  const size_t bytes = static_cast<size_t>(T) * d * 2;
  cudaError_t e = cudaMemcpyAsync(x_dev, x_host, bytes, cudaMemcpyHostToDevice, s);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpyAsync x");
  st = moe_forward_ex(x_dev, w_router, w_gate_up, w_down, T, d, E, I, top_k, out_dev, ws,
                      ws_bytes, stream, ext);
  if (st != MOE_OK) return st;
  e = cudaMemcpyAsync(out_host, out_dev, bytes, cudaMemcpyDeviceToHost, s);
  return e == cudaSuccess ? MOE_OK : cuda_fail(e, "cudaMemcpyAsync out");
}

moe_status_t moe_mxfp8_quantize(const moe_bf16* w, long long rows, int K, uint8_t* codes,
                                uint8_t* scales, moe_stream_t stream) {
  if (rows < 0 || K <= 0 || K % 128) return fail(MOE_ERR_INVALID_ARG, "moe_mxfp8_quantize: K must be a positive multiple of 128");
  if (rows == 0) return MOE_OK;
  if (!w || !codes || !scales || !aligned16(w) || !aligned16(codes) || !aligned16(scales))
    return fail(MOE_ERR_INVALID_ARG, "moe_mxfp8_quantize: null or unaligned pointer");
  moe_status_t st = check_device();
  if (st != MOE_OK) return st;
  const cudaError_t e =
      launch_mxfp8_quantize(reinterpret_cast<cudaStream_t>(stream), w, rows, K, codes, scales);
  return e == cudaSuccess ? MOE_OK : cuda_fail(e, "mxfp8 quantize launch");
}

moe_status_t moe_nvfp4_quantize(const moe_bf16* w, int groups, long long rows_per_group, int K,
                                uint8_t* codes, uint8_t* scales, float* tensor_scales,
                                moe_stream_t stream) {
  if (groups < 0 || rows_per_group < 0 || K <= 0 || K % 256)
    return fail(MOE_ERR_INVALID_ARG, "moe_nvfp4_quantize: K must be a positive multiple of 256");
  if (groups == 0 || rows_per_group == 0) return MOE_OK;
  if (!w || !codes || !scales || !tensor_scales || !aligned16(w) || !aligned16(codes) ||
      !aligned16(scales) || reinterpret_cast<uintptr_t>(tensor_scales) % 4)
    return fail(MOE_ERR_INVALID_ARG, "moe_nvfp4_quantize: null or unaligned pointer");
  moe_status_t st = check_device();
  if (st != MOE_OK) return st;
  const cudaError_t e = launch_nvfp4_quantize(reinterpret_cast<cudaStream_t>(stream), w, groups,
                                              rows_per_group, K, codes, scales, tensor_scales);
  return e == cudaSuccess ? MOE_OK : cuda_fail(e, "nvfp4 quantize launch");
}

moe_status_t moe_forward_graph(const moe_bf16* x, const moe_bf16* w_router,
                               const moe_bf16* w_gate_up, const moe_bf16* w_down, int T, int d,
                               int E, int I, int top_k, moe_bf16* out, void* ws, size_t ws_bytes,
                               const moe_forward_ext_t* ext, int host_buffers,
                               moe_graph_t* graph) {
  if (!graph) return fail(MOE_ERR_INVALID_ARG, "moe_forward_graph: null graph pointer");
  *graph = nullptr;
  moe_status_t st = check_shapes(T, d, E, I, top_k);
  if (st != MOE_OK) return st;
  if (T == 0) return fail(MOE_ERR_INVALID_ARG, "moe_forward_graph: T must be positive");
  if ((st = check_device()) != MOE_OK) return st;
  cudaStream_t cs = nullptr;
  cudaError_t e = cudaStreamCreateWithFlags(&cs, cudaStreamNonBlocking);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamCreateWithFlags");
  const unsigned long long k0 = t_launches;
  e = cudaStreamBeginCapture(cs, cudaStreamCaptureModeRelaxed);
  if (e != cudaSuccess) {
    cudaStreamDestroy(cs);
    return cuda_fail(e, "cudaStreamBeginCapture");
  }
  t_capturing = true;
  const moe_stream_t ms = reinterpret_cast<moe_stream_t>(cs);
  st = host_buffers ? moe_forward_host(x, w_router, w_gate_up, w_down, T, d, E, I, top_k, out, ws,
                                       ws_bytes, ms, ext)
                    : moe_forward_ex(x, w_router, w_gate_up, w_down, T, d, E, I, top_k, out, ws,
                                     ws_bytes, ms, ext);
  t_capturing = false;
  const unsigned long long kernels = t_launches - k0;
  g_launches.fetch_sub(kernels, std::memory_order_relaxed);  // captured, not run
  cudaGraph_t g = nullptr;
  const cudaError_t ee = cudaStreamEndCapture(cs, &g);
  cudaStreamDestroy(cs);
  if (st != MOE_OK) {
    if (g) cudaGraphDestroy(g);
    return st;
  }
  if (ee != cudaSuccess) return cuda_fail(ee, "cudaStreamEndCapture");
  cudaGraphExec_t exec = nullptr;
  e = cudaGraphInstantiate(&exec, g, 0);
  cudaGraphDestroy(g);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGraphInstantiate");
  *graph = new moe_graph_s{exec, kernels};
  return MOE_OK;
}

moe_status_t moe_graph_launch(moe_graph_t graph, moe_stream_t stream) {
  if (!graph) return fail(MOE_ERR_INVALID_ARG, "moe_graph_launch: null graph");
  const cudaError_t e = cudaGraphLaunch(graph->exec, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "cudaGraphLaunch");
  g_launches.fetch_add(graph->kernels, std::memory_order_relaxed);
  return MOE_OK;
}

moe_status_t moe_graph_destroy(moe_graph_t graph) {
  if (!graph) return MOE_OK;
  const cudaError_t e = cudaGraphExecDestroy(graph->exec);
  delete graph;
  return e == cudaSuccess ? MOE_OK : cuda_fail(e, "cudaGraphExecDestroy");
}

moe_status_t moe_get_device_status(void* ws, size_t ws_bytes, moe_stream_t stream) {
  if (!ws || ws_bytes < kAlign) return fail(MOE_ERR_WORKSPACE, "workspace too small");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  unsigned word = 0;
  e = cudaMemcpy(&word, ws, sizeof word, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpy status");
  if (word) {
    e = cudaMemsetAsync(ws, 0, sizeof word, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "clear status");
  }
  if (word & kStatusTimeout) return fail(MOE_ERR_TIMEOUT, "a device-side wait gave up");
  if (word & kStatusDeviceCheck) return fail(MOE_ERR_DEVICE_CHECK, "device-side check failed");
  if (word & kStatusRange)
    return fail(MOE_ERR_RANGE, "an expert output was outside the fp16 range of y");
  return MOE_OK;
}

const char* moe_status_string(moe_status_t s) {
  switch (s) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG";
    case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED";
    case MOE_ERR_WORKSPACE: return "MOE_ERR_WORKSPACE";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
    case MOE_ERR_TIMEOUT: return "MOE_ERR_TIMEOUT";
    case MOE_ERR_RANGE: return "MOE_ERR_RANGE";
    case MOE_ERR_DEVICE_CHECK: return "MOE_ERR_DEVICE_CHECK";
  }
  return "MOE_ERR_UNKNOWN";
}

const char* moe_last_error(void) { return g_last_error.c_str(); }

moe_status_t moe_set_wait_timeout_ns(unsigned long long ns) {
  g_timeout_ns.store(ns ? ns : kDefaultTimeoutNs);
  return MOE_OK;
}

unsigned long long moe_launch_count(void) { return g_launches.load(); }

moe_status_t moe_profiler_enable(int enable) {
  std::lock_guard<std::mutex> lock(g_prof_mu);
  g_prof_on = enable != 0;
  return MOE_OK;
}

moe_status_t moe_profiler_only(const char* kernel_name) {
  std::lock_guard<std::mutex> lock(g_prof_mu);
  g_prof_only = kernel_name ? std::string(kernel_name, strnlen(kernel_name, 63)) : std::string();
  return MOE_OK;
}

moe_status_t moe_profiler_collect(char* names, int* launches, double* total_ms, int n_max,
                                  int* n_out) {
  if (!names || !launches || !total_ms || !n_out || n_max <= 0)
    return fail(MOE_ERR_INVALID_ARG, "moe_profiler_collect: bad arguments");
  std::lock_guard<std::mutex> lock(g_prof_mu);
  int n = 0;
  moe_status_t st = MOE_OK;
  for (const Record& r : g_records) {
    float ms = 0.f;
    cudaError_t e = cudaEventSynchronize(r.stop);
    if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, r.start, r.stop);
    if (e != cudaSuccess) { st = cuda_fail(e, "profiler events"); break; }
    int i = 0;
    while (i < n && std::strncmp(names + 64 * i, r.name, 63) != 0) ++i;
    if (i == n) {
      if (n == n_max) continue;
      std::strncpy(names + 64 * i, r.name, 63);
      names[64 * i + 63] = 0;
      launches[i] = 0;
      total_ms[i] = 0.0;
      ++n;
    }
    launches[i] += 1;
    total_ms[i] += ms;
  }
  for (const Record& r : g_records) {
    g_event_pool.push_back(r.start);
    g_event_pool.push_back(r.stop);
  }
  g_records.clear();
  *n_out = n;
  return st;
}

}  // extern "C"
