/*
 * moe.h -- C ABI of the Mixture-of-Experts FFN layer on NVIDIA GB300 (sm_103a).
 *
 * The layer (sources: 'Chapter 9. Distributed inference', section 9.3.4, the
 * four steps around Fig. 9-16; 'Hosting Qwen on Blackwell', "MoE Dispatch -
 * Combine" and "Expert parallelism"; 'PagedAttention, speculative decoding,
 * MoE and Blackwell', section 2):
 *
 *   1. route    : logits L = x W_r^T (+ b); per token the k largest logits
 *                 (an equal logit loses to a lower expert index); gates =
 *                 softmax of the chosen logits (= full softmax renormalised
 *                 over the chosen k).  Slots are stored in ascending expert id.
 *   2. permute  : per-expert row counts (they sum to T*k), exclusive offsets,
 *                 and a stable grouping of the T*k assignments by expert.
 *   3. expert   : each expert e is a SwiGLU FFN of three d x I matrices:
 *                 h = silu(x W_gate^T) * (x W_up^T), rounded to bf16;
 *                 y = h W_down^T, accumulated in fp32, stored in fp16.
 *   4. combine  : out[t] = sum_j gates[t,j] * y[slot_pos[t,j]] (+ shared
 *                 expert output), summed in fp32 in slot order, rounded once
 *                 to bf16.
 *
 * Conventions for every call
 *   - All tensors are dense, row-major, on the current CUDA device, and owned
 *     by the caller.  The library never allocates, frees or synchronises on
 *     these calls; all work is queued on `stream` and is asynchronous.
 *   - moe_bf16 is the raw bit pattern of an IEEE bfloat16 value.
 *   - Every device pointer must be 16-byte aligned.  Shapes: d % 64 == 0,
 *     I % 64 == 0, 1 <= E <= 256, 1 <= top_k <= min(E, 8), T >= 0.
 *     T == 0 is a no-op that returns MOE_OK.
 *   - Argument errors are found on the host before anything is queued and
 *     return MOE_ERR_INVALID_ARG / MOE_ERR_UNSUPPORTED / MOE_ERR_WORKSPACE.
 *     A failed launch returns MOE_ERR_CUDA (details: moe_last_error()).
 *   - `ws` is a device workspace of at least moe_workspace_size() bytes for
 *     the shapes in use; its first 256 bytes hold a sticky device status word
 *     and the expert GEMMs' tile counters (which every launch leaves at zero
 *     again), and must start at zero (moe_workspace_init); calls that share
 *     one workspace must run one after another.  Kernels record there what
 *     they find on the device: an expert id out of range, inconsistent
 *     offsets or slot positions (MOE_ERR_DEVICE_CHECK), a wait that gave up
 *     (MOE_ERR_TIMEOUT), an expert output outside fp16 range (MOE_ERR_RANGE).
 *     Such a kernel skips the bad work instead of faulting;
 *     read the word with moe_get_device_status().
 *   - Calls that share a workspace must be ordered on one stream.
 */
#ifndef MOE_H_
#define MOE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,   /* a null/unaligned pointer or a bad shape */
  MOE_ERR_UNSUPPORTED = 2,   /* valid but unsupported shape or device */
  MOE_ERR_WORKSPACE = 3,     /* workspace too small */
  MOE_ERR_CUDA = 4,          /* a CUDA runtime/driver call failed */
  MOE_ERR_TIMEOUT = 5,       /* a device-side wait gave up (bounded) */
  MOE_ERR_DEVICE_CHECK = 6,  /* device-side validation found bad indices */
  MOE_ERR_RANGE = 7          /* an expert output left the fp16 range of y */
} moe_status_t;

typedef uint16_t moe_bf16;
typedef uint16_t moe_f16;   /* raw bits of an IEEE binary16 value */
typedef struct CUstream_st* moe_stream_t;  /* same type as cudaStream_t */

/* Workspace bytes that moe_forward / moe_forward_ex need for these shapes;
 * it also covers every single-step call below on the same shapes
 * (rows = T * top_k).  I_shared = 0 when there is no shared expert. */
size_t moe_workspace_size(int T, int d, int E, int I, int top_k, int I_shared);

/* Zero the workspace's status word (queued on `stream`). */
moe_status_t moe_workspace_init(void* ws, size_t ws_bytes, moe_stream_t stream);

/* Step 1, route.  x [T,d] bf16, w_router [E,d] bf16, router_bias [E] fp32 or
 * NULL (added to the logits before selection and gating).  Writes
 * topk_ids [T,top_k] int32 (ascending within a token) and topk_gates
 * [T,top_k] fp32 (sum to 1 per token).  Logits are fp32 sums of bf16
 * products on the tensor cores, accumulated over 512-wide ranges of d and
 * then added in range order, so a token's result does not depend on the
 * other tokens of the batch.  ws: at least moe_workspace_size(T, d, E, 64,
 * top_k, 0) bytes (it holds the partial sums).
 * Cite: 'PagedAttention, speculative decoding, MoE and Blackwell', section 2
 * (gating network, top-K); 'Chapter 9. Distributed inference', section 9.3.4. */
moe_status_t moe_route(const moe_bf16* x, const moe_bf16* w_router,
                       const float* router_bias, int T, int d, int E, int top_k,
                       int32_t* topk_ids, float* topk_gates,
                       void* ws, size_t ws_bytes, moe_stream_t stream);

/* moe_route with a choice of what the bias does.  bias_selection_only = 0:
 * as moe_route.  1: the experts are chosen on logits + router_bias, the gates
 * are the softmax of the chosen experts' unbiased logits (the bias only
 * steers the load; 'PagedAttention, speculative decoding, MoE and
 * Blackwell', section 2, bias adjustment for balancing).  Same buffers,
 * workspace and errors as moe_route. */
moe_status_t moe_route_ex(const moe_bf16* x, const moe_bf16* w_router,
                          const float* router_bias, int bias_selection_only, int T, int d,
                          int E, int top_k, int32_t* topk_ids, float* topk_gates, void* ws,
                          size_t ws_bytes, moe_stream_t stream);

/* Step 2, group by expert.  topk_ids [T,top_k] int32 in [0,E).  Writes
 * expert_counts [E], expert_offsets [E+1] (offsets[E] = T*top_k),
 * perm [T*top_k] (row p of the grouped layout holds assignment perm[p] =
 * t*top_k+j; within an expert, ascending t*top_k+j) and slot_pos
 * [T*top_k] (its inverse).  If x is not NULL, also gathers
 * x_perm [T*top_k, d] bf16 with x_perm[p] = x[perm[p] / top_k].
 * Ids out of range are skipped and flagged MOE_ERR_DEVICE_CHECK.
 * Cite: 'Chapter 9. Distributed inference', section 9.3.4 (permute the input
 * rows by expert) and section 9.4.1 (m_j sum to n k); 'Hosting Qwen on
 * Blackwell', "Expert parallelism" (GEMM input buffers). */
moe_status_t moe_permute(const int32_t* topk_ids, const moe_bf16* x,
                         int T, int d, int E, int top_k,
                         int32_t* expert_counts, int32_t* expert_offsets,
                         int32_t* perm, int32_t* slot_pos, moe_bf16* x_perm,
                         void* ws, size_t ws_bytes, moe_stream_t stream);

/* Step 2 for callers that cannot allocate device memory.  The pages have no
 * counterpart to this call: it is a convenience of this library.
 *
 * Same arguments and results as moe_permute, without the workspace.  Some
 * callers have no device memory to give: a serving process that reserved
 * the GPU's memory for its own pool at start-up (a cudaMalloc here would fail
 * or fragment that pool), or a host framework whose plugin interface hands a
 * kernel only its inputs and outputs.  For them the grouping's one scratch
 * buffer (the per-chunk, per-expert count table) lives in a fixed device
 * array inside this library: 256 KB plus a 256-byte status word, held on
 * every GPU that loads the library until the process exits.  This call
 * allocates and frees nothing.
 *
 * Limit: the table has one entry per (chunk of 1024 assignments, expert):
 * ceil(T*top_k / 1024) * E <= 65536, e.g. T*top_k <= 262,144 with E = 256
 * (1,048,576 with E = 64); larger sizes return MOE_ERR_UNSUPPORTED with a
 * message naming the limit (use moe_permute for them).
 * device_status: a device uint32 into which the kernels OR their status bits
 * (1 = a wait gave up, 2 = an expert id out of range was skipped); the caller
 * zeroes it.  If NULL, the bits go to the library's own status word, which
 * each call clears first and which cannot be read back.
 * The first call on each device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current and keeps it for that
 * device's current CUDA context; a call made in a new context (after
 * cudaDeviceReset, say) looks it up again.  Make the first call on a device,
 * and the first after a reset, before any stream capture.  All calls share
 * the array: calls whose work
 * can overlap on the GPU (unordered streams) race and may give wrong
 * results, so order them on one stream. */
moe_status_t moe_permute_static_scratch(const int32_t* topk_ids, const moe_bf16* x,
                                        int T, int d, int E, int top_k,
                                        int32_t* expert_counts, int32_t* expert_offsets,
                                        int32_t* perm, int32_t* slot_pos, moe_bf16* x_perm,
                                        uint32_t* device_status, moe_stream_t stream);

/* Step 3, grouped expert FFN.  Rows [expert_offsets[e], expert_offsets[e+1])
 * of x_perm [rows,d] go through expert e: w_gate_up [E,2I,d] (per expert,
 * rows [0,I) gate, [I,2I) up), w_down [E,d,I].  Writes y [rows,d] fp16: the
 * fp32 accumulators rounded to nearest; finite values beyond +-65504 are
 * stored as +-65504 and infinities as they are, and either flags
 * MOE_ERR_RANGE (NaN passes through unflagged).
 * h is kept in the workspace as bf16.  Offsets that do not start at 0, go
 * down, or do not end at `rows` make the kernels skip all work and flag
 * MOE_ERR_DEVICE_CHECK.
 * Cite: 'Chapter 9. Distributed inference', section 9.3.2 (three matrices per
 * expert, F_e(m) = 2 m P_e) and section 9.4.3 (grouped GEMM). */
moe_status_t moe_expert_ffn(const moe_bf16* x_perm, const int32_t* expert_offsets,
                            const moe_bf16* w_gate_up, const moe_bf16* w_down,
                            int rows, int d, int E, int I, moe_f16* y,
                            void* ws, size_t ws_bytes, moe_stream_t stream);

/* Step 4, combine.  out[t] = bf16( sum_{j<top_k} topk_gates[t,j] *
 * y[slot_pos[t,j]] (+ y_shared[t]) ), fp32 sums in j order (deterministic).
 * y [rows,d] fp16 with rows = T*top_k, y_shared [T,d] fp16 or NULL.
 * A slot position outside [0,rows) is skipped and flagged.
 * Cite: 'Chapter 9. Distributed inference', section 9.3.4, step four;
 * 'Hosting Qwen on Blackwell', "MoE Dispatch - Combine". */
moe_status_t moe_combine(const moe_f16* y, const int32_t* slot_pos,
                         const float* topk_gates, const moe_f16* y_shared,
                         int T, int d, int top_k, moe_bf16* out,
                         void* ws, size_t ws_bytes, moe_stream_t stream);

/* The whole layer: steps 1-4 on one stream, intermediates in `ws`.
 * x [T,d], w_router [E,d], w_gate_up [E,2I,d], w_down [E,d,I] -> out [T,d].
 * Cite: 'Chapter 9. Distributed inference', section 9.3.4 (the four steps of
 * one MoE layer around Fig. 9-16: route, permute by expert, expert matrix
 * multiplications, weighted combine). */
moe_status_t moe_forward(const moe_bf16* x, const moe_bf16* w_router,
                         const moe_bf16* w_gate_up, const moe_bf16* w_down,
                         int T, int d, int E, int I, int top_k, moe_bf16* out,
                         void* ws, size_t ws_bytes, moe_stream_t stream);

/* Optional parts of the layer.  router_bias: [E] fp32 added to the logits;
 * bias_selection_only: 0 = the bias enters selection and gates, 1 = selection
 * only (see moe_route_ex).  Shared expert ('PagedAttention, speculative
 * decoding, MoE and Blackwell', section 2: experts that process every token):
 * w_gate_up_shared [2*I_shared,d], w_down_shared [d,I_shared]; its output is
 * added with weight 1.
 * single_launch = 1: the whole layer runs as one kernel launch ('Hosting Qwen
 * on Blackwell', "Expert parallelism": decode fuses dispatch, GEMMs and
 * combine into one kernel): a cooperative launch whose phases (router,
 * top-k, grouping, gate_up, down, combine) are separated by grid-wide
 * barriers bounded by the wait timeout.  For decode-sized batches with bf16
 * expert weights: d and I multiples of 128, no shared expert, T*top_k <= 4096
 * and at most 16 rows per expert on average (else MOE_ERR_UNSUPPORTED).  The
 * barrier counters live in the workspace's first 256 bytes, which must start
 * at zero (moe_workspace_init) like the status word.  The router sums its
 * logits over 128-wide ranges of d here (512 otherwise), so a near-tie may
 * route differently from the multi-launch layer; both are checked against
 * the same reference.
 * y_fp32 = 1: the expert outputs y (and the shared expert's) are kept in fp32
 * instead of fp16 between the down GEMM and the combine, so an output beyond
 * the fp16 range (|y| > 65504) is neither saturated nor flagged
 * (MOE_ERR_RANGE cannot occur); the down GEMM's stores and the combine's
 * reads of y double, and the workspace must hold moe_workspace_size_ex(...,
 * ext) bytes (MOE_ERR_WORKSPACE otherwise).  Not with single_launch
 * (MOE_ERR_UNSUPPORTED).
 * act_mxfp8 = 1 (moe_forward_mxfp8 only): the expert GEMMs' token operands
 * are micro-scaled too, W8A8 ('Hosting Qwen on Blackwell', "Quantization":
 * micro-scaling for the best decode throughput): x before gate_up and h
 * (after its bf16 rounding) before down are quantised to MXFP8 along the
 * reduction, in runs of 32 with one E8M0 scale each (the weights' rule), and
 * the GEMMs multiply the codes with fp8 tensor-core MMAs, each run's fp32
 * sum scaled by its two scales.  Decode sizes only: at most 8 rows per expert
 * on average, d and I multiples of 256, no shared expert, not single_launch
 * (MOE_ERR_UNSUPPORTED otherwise).  The workspace must hold
 * moe_workspace_size_ex(..., ext) bytes; the codes and scales are left in
 * its act_x / act_h regions (moe_workspace_layout_ex).
 * Zero-initialise the struct: later fields default to 0. */
typedef struct {
  const float* router_bias;
  const moe_bf16* w_gate_up_shared;
  const moe_bf16* w_down_shared;
  int I_shared;
  int bias_selection_only;
  int single_launch;
  int y_fp32;
  int act_mxfp8;
} moe_forward_ext_t;

/* Workspace bytes for moe_forward_ex (and the other calls taking ext) with
 * these options: the shared expert (ext->I_shared), fp32 y (ext->y_fp32) and
 * MXFP8 tokens (ext->act_mxfp8); ext may be NULL (then equal to
 * moe_workspace_size(..., 0)). */
size_t moe_workspace_size_ex(int T, int d, int E, int I, int top_k,
                             const moe_forward_ext_t* ext);

moe_status_t moe_forward_ex(const moe_bf16* x, const moe_bf16* w_router,
                            const moe_bf16* w_gate_up, const moe_bf16* w_down,
                            int T, int d, int E, int I, int top_k, moe_bf16* out,
                            void* ws, size_t ws_bytes, moe_stream_t stream,
                            const moe_forward_ext_t* ext);

/* The whole layer on host buffers: x_host [T,d] and out_host [T,d] are in host
 * memory (pinned for asynchronous copies); weights stay on the device.  The
 * copies go through the workspace (regions x_stage / out_stage) and are
 * queued on `stream` with the layer between them; the call returns without
 * synchronising, so out_host is ready once the stream reaches this point.
 * ext may be NULL. */
moe_status_t moe_forward_host(const moe_bf16* x_host, const moe_bf16* w_router,
                              const moe_bf16* w_gate_up, const moe_bf16* w_down,
                              int T, int d, int E, int I, int top_k, moe_bf16* out_host,
                              void* ws, size_t ws_bytes, moe_stream_t stream,
                              const moe_forward_ext_t* ext);

/* MXFP8 expert weights ('Hosting Qwen on Blackwell', "Quantization": the
 * weights are converted statically after training).  Quantises w [rows, K]
 * bf16 (K a multiple of 128) to E4M3 codes [rows, K] uint8 and E8M0 scales
 * [K/128][rows][4] uint8 following the OCP microscaling definition: one scale
 * per 32 values along K, X = floor(log2(max |v|)) - 8 stored as X + 127
 * (clamped to 0..254; an all-zero run stores 0), elements v / 2^X rounded to
 * nearest even and clamped to +-448.  The scale layout keeps the four scales
 * of a 128-wide K block of a row in one 32-bit word, which is what
 * moe_forward_mxfp8 reads.  Device pointers, 16-byte aligned; asynchronous on
 * `stream`.  MOE_ERR_INVALID_ARG for bad pointers or shapes. */
moe_status_t moe_mxfp8_quantize(const moe_bf16* w, long long rows, int K, uint8_t* codes,
                                uint8_t* scales, moe_stream_t stream);

/* The whole layer with MXFP8 expert weights (quantised by moe_mxfp8_quantize):
 * codes_gate_up [E, 2I, d] and scales_gate_up [d/128][E*2I][4], codes_down
 * [E, d, I] and scales_down [I/128][E*d][4].  Activations, router, shared
 * expert (ext) and outputs are as in moe_forward_ex; the experts compute
 * with the dequantised weights (codes x 2^(scale - 127), exact in bf16) on
 * the bf16 tensor cores, half the weight bytes read from HBM.  d and I must
 * be multiples of 128 (else MOE_ERR_UNSUPPORTED).  Layers with at most 8
 * token rows per expert on average (decode) and d, I multiples of 256 run
 * warp-level kernels that decode the codes in registers next to their MMAs;
 * the others one CTA per tile of 128 weight rows and at most 128 tokens.
 * Same workspace as moe_forward. */
moe_status_t moe_forward_mxfp8(const moe_bf16* x, const moe_bf16* w_router,
                               const uint8_t* codes_gate_up, const uint8_t* scales_gate_up,
                               const uint8_t* codes_down, const uint8_t* scales_down, int T,
                               int d, int E, int I, int top_k, moe_bf16* out, void* ws,
                               size_t ws_bytes, moe_stream_t stream,
                               const moe_forward_ext_t* ext);

/* NVFP4 expert weights ('PagedAttention, speculative decoding, MoE and
 * Blackwell', section 3: two-level micro-scaling, 16-value blocks with an FP8
 * scale each and one FP32 scale per tensor).  Quantises `groups` matrices
 * w [groups][rows_per_group][K] bf16 (K a multiple of 256; one matrix = one
 * expert's W_gate_up or W_down) to E2M1 codes [groups*rows_per_group][K/2]
 * (value 2i in the low nibble of byte i), E4M3 block scales
 * [K/256][groups*rows_per_group][16] and one fp32 tensor scale per matrix.
 * Rule (the pages give none; fp32, round to nearest, in this order):
 * g = amax / (448 * 6) (1 for an all-zero matrix); block scale =
 * E4M3((amax_block / 6) / g); element = E2M1(w / (scale * g)), nearest even,
 * saturating at 6, -0 stored as +0.  Device pointers (codes, scales 16-byte
 * aligned); asynchronous on `stream`. */
moe_status_t moe_nvfp4_quantize(const moe_bf16* w, int groups, long long rows_per_group, int K,
                                uint8_t* codes, uint8_t* scales, float* tensor_scales,
                                moe_stream_t stream);

/* The whole layer with NVFP4 expert weights (moe_nvfp4_quantize of W_gate_up
 * as E matrices [2I, d] and of W_down as E matrices [d, I]).  The experts
 * compute with E2M1 value x block scale (exact in bf16) on the bf16 tensor
 * cores and apply each expert's tensor scale to the fp32 accumulators; the
 * rest is moe_forward_ex.  d and I must be multiples of 256 (else
 * MOE_ERR_UNSUPPORTED).  Layers with at most 8 token rows per expert on
 * average (decode) run warp-level kernels that decode the codes in registers
 * next to their MMAs.  Same workspace as moe_forward. */
moe_status_t moe_forward_nvfp4(const moe_bf16* x, const moe_bf16* w_router,
                               const uint8_t* codes_gate_up, const uint8_t* scales_gate_up,
                               const float* tscale_gate_up, const uint8_t* codes_down,
                               const uint8_t* scales_down, const float* tscale_down, int T,
                               int d, int E, int I, int top_k, moe_bf16* out, void* ws,
                               size_t ws_bytes, moe_stream_t stream,
                               const moe_forward_ext_t* ext);

/* The whole layer as a CUDA graph, for calls repeated with the same shapes and
 * buffers (decode steps).  moe_forward_graph captures one moe_forward_ex
 * (host_buffers = 0: x, out in device memory) or one moe_forward_host
 * (host_buffers = 1: x, out pinned host buffers, the copies captured too) into
 * an executable graph; nothing runs at capture.  moe_graph_launch replays it
 * on `stream`, reading x and writing out (and the workspace) as the captured
 * call would: change the contents of x between replays, not the pointers.
 * All buffers must outlive the graph.  Errors as the captured call, plus
 * MOE_ERR_CUDA when capture or instantiation fails.  The pages fuse the whole
 * decode step into one launch ('Hosting Qwen on Blackwell', "Expert
 * parallelism"); a graph replays the layer's kernels with one host call. */
typedef struct moe_graph_s* moe_graph_t;

moe_status_t moe_forward_graph(const moe_bf16* x, const moe_bf16* w_router,
                               const moe_bf16* w_gate_up, const moe_bf16* w_down, int T, int d,
                               int E, int I, int top_k, moe_bf16* out, void* ws, size_t ws_bytes,
                               const moe_forward_ext_t* ext, int host_buffers,
                               moe_graph_t* graph);
moe_status_t moe_graph_launch(moe_graph_t graph, moe_stream_t stream);
moe_status_t moe_graph_destroy(moe_graph_t graph);

/* Where moe_forward(_ex) keeps its intermediates: byte offsets into `ws`
 * (each 256-byte aligned) for the same shapes.  act_x / act_x_scales hold
 * the MXFP8 tokens x of act_mxfp8 ([T, d] codes, [T, d / 32] E8M0 scales),
 * act_h / act_h_scales those of h ([T*top_k, I], [T*top_k, I / 32]); their
 * codes are stored per 256-wide chunk in the order the GEMMs read them (byte
 * 64 t + 8 r + j of a chunk holds value 32 r + 4 t + (j & 3) + 16 (j >> 2)).
 * Without act_mxfp8 these regions are empty. */
typedef struct {
  size_t status, router_logits, topk_ids, topk_gates, expert_counts, expert_offsets, perm,
         slot_pos, chunk_table, x_perm, h, h_shared, y, y_shared, x_stage, out_stage,
         act_x, act_x_scales, act_h, act_h_scales, total;
} moe_workspace_layout_t;

moe_status_t moe_workspace_layout(int T, int d, int E, int I, int top_k, int I_shared,
                                  moe_workspace_layout_t* layout);
/* The same for the options in ext (fp32 y: y and y_shared take 4 bytes a
 * value); ext may be NULL. */
moe_status_t moe_workspace_layout_ex(int T, int d, int E, int I, int top_k,
                                     const moe_forward_ext_t* ext,
                                     moe_workspace_layout_t* layout);

/* Synchronise `stream`, read and clear the workspace's device status word. */
moe_status_t moe_get_device_status(void* ws, size_t ws_bytes, moe_stream_t stream);

const char* moe_status_string(moe_status_t status);
/* Message of the last failing call on this thread ("" if none). */
const char* moe_last_error(void);

/* Bound on every device-side wait, in nanoseconds (default 2e9; 0 restores
 * the default).  After it a kernel records MOE_ERR_TIMEOUT, drains its own
 * copies and tensor-core work in flight, frees its tensor memory and
 * returns; the context stays usable.  A bound of 1 makes every wait that is
 * not already satisfied give up at once (used to test this path). */
moe_status_t moe_set_wait_timeout_ns(unsigned long long ns);

/* Kernel launches made by this library since it was loaded. */
unsigned long long moe_launch_count(void);

/* Tracing.  While enabled, every kernel launch is bracketed by CUDA events on
 * its stream.  moe_profiler_collect() synchronises those events and returns,
 * per kernel name (in first-launch order), the launch count and total
 * milliseconds; it then clears the records.  names: n_max entries of 64 bytes.
 * Returns the number of kernel names written in *n_out. */
moe_status_t moe_profiler_enable(int enable);
/* Restrict tracing to launches of one kernel name (as reported by
 * moe_profiler_collect, at most 63 bytes); NULL or "" traces every launch.
 * Each traced launch costs two event records on its stream, which also
 * delay the next launch, so a timed region traces only the kernel whose
 * duration it needs. */
moe_status_t moe_profiler_only(const char* kernel_name);
moe_status_t moe_profiler_collect(char* names, int* launches, double* total_ms,
                                  int n_max, int* n_out);

#ifdef __cplusplus
}
#endif

#endif /* MOE_H_ */
