"""Plain fp64 CPU oracle of the Mixture-of-Experts FFN layer.

TEST INFRASTRUCTURE ONLY. Nothing on the product path imports this module: the
CUDA library and its Python binding share no code, table or helper with it.
Only the tests, the smoke check and the benchmark's CPU-baseline / reference
arm call it.

What the layer computes, and where each step comes from:

* Router.  A light learned gating network scores every expert for each token
  and sends the token to its top-K experts ('PagedAttention, speculative
  decoding, MoE and Blackwell', section 2, "How MoE layers work"; 'Chapter 9.
  Distributed inference', section 9.3.4, the four steps around Fig. 9-16: "the
  router picks eight experts for each token").  Gates are the softmax of the
  logits, restricted to the chosen k and renormalised to sum to one; ties go to
  the lower expert index.  The pages do not spell out the gate function; this
  is the layer's specification and the plainest reading of "weighted by the
  routing weights" in section 9.3.4.
* Grouping.  Each token's row is laid out once per chosen expert, the rows of
  one expert contiguous (section 9.3.4, step three: "permute the input rows by
  expert and run the expert matrix multiplications"; 'Hosting Qwen on
  Blackwell', "Expert parallelism": the dispatch kernel gathers the routing
  information and prepares the MoE GEMM input buffers).  The per-expert row
  counts m_j sum to n*k (section 9.4.1, the definition of m_j).
* Expert FFN.  An expert is three matrices of d x I (section 9.3.2: Qwen3-235B-
  A22B's expert has 3 x 4096 x 1536 parameters) used as a SwiGLU block:
  h = silu(x W_gate^T) * (x W_up^T), y = h W_down^T.  Matrix work is 2 m P_e
  FLOPs for m rows (section 9.3.2, F_e(m)).
* Combine.  A token's output is the routing-weighted sum of its k expert
  outputs (section 9.3.4, step four; 'Hosting Qwen on Blackwell', "MoE
  Dispatch - Combine": weighted accumulation in combine).  An always-on shared
  expert adds its output with weight one ('PagedAttention, speculative
  decoding, MoE and Blackwell', section 2, shared experts).
* MXFP8 expert weights ('Hosting Qwen on Blackwell', "Quantization": the
  weights are converted to MXFP8 statically after training).  MXFP8 is the
  OCP microscaling format with FP8 E4M3 elements: each run of 32 consecutive
  values along the reduction dimension shares one power-of-two scale (an E8M0
  exponent) chosen from the run's largest magnitude so that it maps into
  E4M3's top binade; the elements are rounded to nearest, ties to even, and
  clamped to E4M3's largest finite value.  A layer with MXFP8 weights is the
  layer computed with the dequantised weights (codes times scales), which the
  oracle obtains with mxfp8_quantize / mxfp8_dequantize.
* MXFP8 activations (``act_mxfp8``).  The same section says micro-scaling is
  what the tensor cores need for the best throughput; the deployed format
  then also carries the activations as MXFP8.  The pages do not say which
  activations or where; the plainest reading, taken here: each expert GEMM's
  token operand is quantised like its weights, along the reduction axis in
  runs of 32 -- x before gate_up, and h (after its rounding to bf16) before
  down -- and the GEMM is then the exact product of the dequantised values.
* NVFP4 expert weights ('PagedAttention, speculative decoding, MoE and
  Blackwell', section 3: two-level micro-scaling, blocks of 16 values each
  with its own FP8 scale, plus one FP32 scale for the whole tensor; 'Hosting
  Qwen on Blackwell', "Quantization", names the format as considered).  The
  elements are FP4 E2M1 (values 0, 0.5, 1, 1.5, 2, 3, 4, 6 and their
  negatives).  The pages give no rule for choosing the scales; the oracle
  takes the plainest one that uses both ranges fully: the tensor scale maps
  the tensor's largest magnitude to 448 x 6 (the largest E4M3 scale times
  the largest element), each block's scale is its largest magnitude / 6 in
  units of the tensor scale, rounded to E4M3, and each element is the value
  divided by (block scale x tensor scale) rounded to nearest-even E2M1,
  saturating at 6.  These steps are taken in fp32 (IEEE, round to nearest) in
  the order written, so that a GPU kernel doing the same operations produces
  the same codes; the tensor is one expert's matrix.
* Router bias.  A per-expert bias is added to the logits; by default it takes
  part in both the selection and the gates.  The variant the same section
  names for balancing (DeepSeek's bias adjustment) uses the bias only to pick
  the experts: selection on logits + bias, gates from the unbiased logits of
  the chosen experts (``bias_for_selection_only``).

Precision: every product and sum is fp64 over the exact values of the bf16
inputs.  The one deliberate rounding is h -> bf16 (round to nearest, ties to
even): the down projection's input is a bf16 activation in the layer being
modelled, so the oracle rounds h exactly once, like any bf16 implementation
must.  The final output is left unrounded.

Inputs are raw bf16 bit patterns (numpy uint16) so that the oracle decodes them
itself.  Weight arguments only need ``w[e]`` indexing, so a caller may pass a
lazy per-expert accessor instead of a whole [E, ...] array.
"""

from __future__ import annotations

import numpy as np

__all__ = [
    "bf16_bits_to_f64",
    "round_to_bf16",
    "f64_to_bf16_bits",
    "router_logits",
    "select_top_k",
    "route",
    "permute",
    "swiglu_ffn",
    "expert_ffn",
    "combine",
    "forward",
    "forward_tokens",
    "e4m3_values",
    "round_to_e4m3",
    "mxfp8_quantize",
    "mxfp8_dequantize",
    "mxfp8_round_rows",
    "e2m1_values",
    "round_to_e2m1",
    "nvfp4_quantize",
    "nvfp4_dequantize",
]


# --------------------------------------------------------------------------
# bf16 encoding (IEEE binary32 with the low 16 mantissa bits dropped)
# --------------------------------------------------------------------------

def bf16_bits_to_f64(bits) -> np.ndarray:
    """Exact value of each bf16 bit pattern, as fp64."""
    b = np.asarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def round_to_bf16(x) -> np.ndarray:
    """Round fp64 values to the nearest bf16 value, ties to even (one rounding).

    bf16 keeps 8 significant bits.  For |x| in [2^(e-1), 2^e) the spacing of
    bf16 values is 2^(e-8); below the smallest normal (2^-126) it stays 2^-133.
    Dividing by a power of two is exact, and numpy's round() breaks ties to
    even, so this is round-to-nearest-even straight from fp64.
    """
    x = np.asarray(x, dtype=np.float64)
    _, e = np.frexp(x)
    e = np.maximum(e, -125)
    spacing = np.ldexp(1.0, e - 8)
    r = np.round(x / spacing) * spacing
    if np.any(np.abs(r) > 3.3895313892515355e38):  # largest finite bf16
        raise OverflowError("value outside the bf16 range")
    return r


def f64_to_bf16_bits(x) -> np.ndarray:
    """Bit patterns of round_to_bf16(x)."""
    r = round_to_bf16(x).astype(np.float32)  # exact: bf16 values are fp32 values
    return (r.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


# --------------------------------------------------------------------------
# Router: logits, top-k selection, renormalised gates
# --------------------------------------------------------------------------

def router_logits(x_bits, w_router_bits, router_bias=None) -> np.ndarray:
    """L[t, e] = x[t] . W_r[e] (+ b[e]) in fp64."""
    x = bf16_bits_to_f64(x_bits)
    w = bf16_bits_to_f64(w_router_bits)
    logits = x @ w.T
    if router_bias is not None:
        logits = logits + np.asarray(router_bias, dtype=np.float64)[None, :]
    return logits


def select_top_k(logits_row, top_k: int) -> list:
    """Indices of the k largest logits; an equal logit loses to a lower index.

    Returned in ascending expert-id order: the chosen set is what the method
    defines, and a canonical slot order makes the combine order well defined.
    """
    E = len(logits_row)
    ranked = sorted(range(E), key=lambda e: (-logits_row[e], e))
    return sorted(ranked[:top_k])


def route(x_bits, w_router_bits, top_k: int, router_bias=None,
          bias_for_selection_only: bool = False):
    """Top-k routing with softmax gates renormalised over the chosen experts.

    With bias_for_selection_only the bias decides which experts are chosen but
    the gates are computed from the unbiased logits ('PagedAttention,
    speculative decoding, MoE and Blackwell', section 2: bias adjustment steers
    the load without changing the mixing weights).

    Returns (ids [T,k] int32, gates [T,k] fp64, logits [T,E] fp64); logits are
    the ones the selection used.
    """
    logits = router_logits(x_bits, w_router_bits, router_bias)
    gate_logits = logits
    if bias_for_selection_only and router_bias is not None:
        gate_logits = router_logits(x_bits, w_router_bits, None)
    T, E = logits.shape
    if not 1 <= top_k <= E:
        raise ValueError("top_k must be in [1, E]")
    ids = np.empty((T, top_k), dtype=np.int32)
    gates = np.empty((T, top_k), dtype=np.float64)
    for t in range(T):
        chosen = select_top_k(logits[t], top_k)
        # softmax over all E experts ...
        row = gate_logits[t]
        p = np.exp(row - row.max())
        p = p / p.sum()
        # ... keep the chosen k and renormalise them to sum to one
        kept = p[chosen]
        ids[t] = chosen
        gates[t] = kept / kept.sum()
    return ids, gates, logits


# --------------------------------------------------------------------------
# MXFP8: FP8 E4M3 elements with one E8M0 (power-of-two) scale per 32 values
# --------------------------------------------------------------------------

E4M3_MAX = 448.0        # 1.75 * 2^8, the largest finite E4M3 value
E4M3_EMAX = 8           # exponent of E4M3's top binade
MX_BLOCK = 32           # values that share one scale


def e4m3_values() -> np.ndarray:
    """fp64 value of each of the 256 E4M3 codes (bit 7 sign, bits 6-3 the
    exponent with bias 7, bits 2-0 the mantissa; exponent 0 is subnormal,
    codes 0x7f / 0xff are NaN, there are no infinities)."""
    vals = np.empty(256, dtype=np.float64)
    for c in range(256):
        sign = -1.0 if c & 0x80 else 1.0
        e = (c >> 3) & 0xF
        m = c & 0x7
        if e == 0xF and m == 0x7:
            vals[c] = np.nan
        elif e == 0:
            vals[c] = sign * m * 2.0 ** -9           # (m / 8) * 2^(1 - 7)
        else:
            vals[c] = sign * (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return vals


def round_to_e4m3(v) -> np.ndarray:
    """Round fp64 values to the E4M3 grid: nearest, ties to even, magnitudes
    above 448 clamped to 448.  Returns the rounded fp64 values."""
    v = np.clip(np.asarray(v, dtype=np.float64), -E4M3_MAX, E4M3_MAX)
    a = np.abs(v)
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    quantum = np.where(a >= 2.0 ** -6, 2.0 ** (np.maximum(e, -6) - 3), 2.0 ** -9)
    return np.minimum(np.rint(a / quantum) * quantum, E4M3_MAX) * np.sign(v)


def mxfp8_quantize(w):
    """Quantise along the last axis (a multiple of 32) to MXFP8.

    Per block of 32: X = floor(log2(max |v|)) - 8, stored as the E8M0 byte
    X + 127 (clamped to 0..254; an all-zero block stores 0); elements are
    round_to_e4m3(v / 2^X) encoded as E4M3 codes.  Returns (codes uint8 with
    w's shape, scales uint8 with the last axis divided by 32)."""
    w = np.asarray(w, dtype=np.float64)
    K = w.shape[-1]
    if K % MX_BLOCK:
        raise ValueError("the quantised axis must be a multiple of 32")
    blocks = w.reshape(*w.shape[:-1], K // MX_BLOCK, MX_BLOCK)
    amax = np.abs(blocks).max(axis=-1)
    with np.errstate(divide="ignore"):
        xexp = np.floor(np.log2(np.where(amax > 0, amax, 1.0))) - E4M3_EMAX
    scale_byte = np.where(amax > 0, np.clip(xexp + 127, 0, 254), 0).astype(np.uint8)
    xexp = scale_byte.astype(np.float64) - 127
    q = round_to_e4m3(blocks / 2.0 ** xexp[..., None])
    # encode: codes 0x00..0x7e hold the non-negative values in increasing order
    positive = e4m3_values()[:0x7F]
    mag = np.searchsorted(positive, np.abs(q))
    codes = np.where(q < 0, mag | 0x80, mag).astype(np.uint8)
    return codes.reshape(w.shape), scale_byte


def mxfp8_dequantize(codes, scales) -> np.ndarray:
    """codes times 2^(scale byte - 127), in fp64."""
    codes = np.asarray(codes, dtype=np.uint8)
    K = codes.shape[-1]
    vals = e4m3_values()[codes].reshape(*codes.shape[:-1], K // MX_BLOCK, MX_BLOCK)
    x = 2.0 ** (np.asarray(scales, dtype=np.float64) - 127)
    return (vals * x[..., None]).reshape(codes.shape)


E2M1_MAX = 6.0          # the largest E2M1 value
NV_BLOCK = 16           # values that share one E4M3 scale
NV_TENSOR_DIV = np.float32(E4M3_MAX * E2M1_MAX)   # 2688: tensor scale = amax / 2688


def e2m1_values() -> np.ndarray:
    """fp64 value of each of the 16 E2M1 codes (bit 3 sign, bits 2-1 the
    exponent with bias 1, bit 0 the mantissa; exponent 0 is subnormal: m x 0.5)."""
    vals = np.empty(16, dtype=np.float64)
    for c in range(16):
        sign = -1.0 if c & 0x8 else 1.0
        e = (c >> 1) & 0x3
        m = c & 0x1
        vals[c] = sign * (m * 0.5 if e == 0 else (1.0 + m / 2.0) * 2.0 ** (e - 1))
    return vals


def round_to_e2m1(v) -> np.ndarray:
    """Codes of the E2M1 values nearest to v (ties to the even code, i.e. the
    one whose mantissa bit is 0), magnitudes above 6 saturating to 6; -0
    encodes as +0."""
    v = np.asarray(v, dtype=np.float64)
    grid = e2m1_values()[:8]                        # 0, 0.5, 1, 1.5, 2, 3, 4, 6
    a = np.minimum(np.abs(v), E2M1_MAX)
    d = np.abs(a[..., None] - grid)                 # distance to every magnitude
    best = d.min(axis=-1, keepdims=True)
    cand = d == best                                # one, or two on a tie
    even = cand & (np.arange(8) % 2 == 0)
    mag = np.where(even.any(axis=-1), even.argmax(axis=-1), cand.argmax(axis=-1))
    return np.where((v < 0) & (mag > 0), mag | 0x8, mag).astype(np.uint8)


def nvfp4_quantize(w):
    """Quantise one matrix (fp32-representable values, last axis a multiple
    of 16 along the reduction dimension) to NVFP4.

    Returns (codes uint8 [..., K] one E2M1 code per value, scales uint8
    [..., K/16] E4M3 codes, tensor scale as np.float32).  All arithmetic is
    fp32 with round to nearest: g = amax / 2688 (1 for an all-zero matrix);
    per block s = round_to_e4m3((amax_block / 6) / g); each element
    round_to_e2m1(w / (s * g)), or code 0 where s * g is 0."""
    w = np.asarray(w, dtype=np.float32)
    K = w.shape[-1]
    if K % NV_BLOCK:
        raise ValueError("the quantised axis must be a multiple of 16")
    amax_t = np.float32(np.abs(w).max()) if w.size else np.float32(0)
    g = amax_t / NV_TENSOR_DIV if amax_t > 0 else np.float32(1)
    blocks = w.reshape(*w.shape[:-1], K // NV_BLOCK, NV_BLOCK)
    amax_b = np.abs(blocks).max(axis=-1).astype(np.float32)
    s = (amax_b / np.float32(E2M1_MAX)) / g                          # fp32, in this order
    s_q = round_to_e4m3(s.astype(np.float64)).astype(np.float32)      # exact in fp32
    positive = e4m3_values()[:0x7F]
    scale_codes = np.searchsorted(positive, s_q.astype(np.float64)).astype(np.uint8)
    denom = (s_q * g).astype(np.float32)                             # fp32 product
    with np.errstate(divide="ignore", invalid="ignore"):
        x = np.where(denom[..., None] > 0, blocks / denom[..., None], np.float32(0))
    codes = round_to_e2m1(x.astype(np.float32).astype(np.float64))
    return codes.reshape(w.shape), scale_codes, np.float32(g)


def nvfp4_dequantize(codes, scales, tensor_scale) -> np.ndarray:
    """E2M1 value x E4M3 block scale x tensor scale, in fp64 (exact)."""
    codes = np.asarray(codes, dtype=np.uint8)
    K = codes.shape[-1]
    vals = e2m1_values()[codes].reshape(*codes.shape[:-1], K // NV_BLOCK, NV_BLOCK)
    s = e4m3_values()[np.asarray(scales, dtype=np.uint8)]
    return (vals * s[..., None] * np.float64(tensor_scale)).reshape(codes.shape)


# --------------------------------------------------------------------------
# Grouping rows by expert: counts, offsets, stable permutation
# --------------------------------------------------------------------------

def permute(ids, E: int):
    """Counting sort of the T*k assignments by expert, stable in t*k+j order.

    Returns (counts [E], offsets [E+1], perm [T*k], slot_pos [T,k]) where
    perm[p] is the flat assignment index t*k+j stored at row p of the grouped
    layout and slot_pos[t, j] is the row that holds assignment (t, j).
    """
    ids = np.asarray(ids)
    T, k = ids.shape
    flat = ids.reshape(-1)
    counts = np.zeros(E, dtype=np.int64)
    for e in flat:
        if not 0 <= e < E:
            raise ValueError("expert id out of range")
        counts[e] += 1
    offsets = np.zeros(E + 1, dtype=np.int64)
    for e in range(E):
        offsets[e + 1] = offsets[e] + counts[e]
    next_row = offsets[:-1].copy()
    perm = np.empty(T * k, dtype=np.int64)
    slot_pos = np.empty(T * k, dtype=np.int64)
    for f in range(T * k):  # ascending flat index: equal keys keep their order
        e = flat[f]
        p = next_row[e]
        next_row[e] += 1
        perm[p] = f
        slot_pos[f] = p
    return counts, offsets, perm, slot_pos.reshape(T, k)


# --------------------------------------------------------------------------
# Expert FFN (SwiGLU, three matrices)
# --------------------------------------------------------------------------

def _weight_values(w) -> np.ndarray:
    """Expert weights given as bf16 bit patterns (uint16), or as exact values
    (float64, e.g. dequantised NVFP4 weights, which bf16 cannot hold)."""
    w = np.asarray(w)
    return w if w.dtype == np.float64 else bf16_bits_to_f64(w)


def mxfp8_round_rows(v) -> np.ndarray:
    """v quantised to MXFP8 along its last axis and dequantised: the values an
    MXFP8 activation operand stands for."""
    codes, scales = mxfp8_quantize(v)
    return mxfp8_dequantize(codes, scales)


def swiglu_ffn(x_rows, w_gate_up_bits, w_down_bits, act_mxfp8: bool = False) -> np.ndarray:
    """One expert on a block of rows: fp64, with h rounded once to bf16.

    x_rows: [m, d] fp64.  w_gate_up: [2I, d] bf16 bits (or fp64 values), rows
    [0, I) = gate and rows [I, 2I) = up.  w_down: [d, I] likewise.  Returns
    y [m, d] fp64.  act_mxfp8: x and the bf16 h are quantised to MXFP8 (runs
    of 32 along d and along I) before their products.
    """
    w_gu = _weight_values(w_gate_up_bits)
    w_d = _weight_values(w_down_bits)
    I = w_gu.shape[0] // 2
    if act_mxfp8:
        x_rows = mxfp8_round_rows(x_rows)
    gate = x_rows @ w_gu[:I].T
    up = x_rows @ w_gu[I:].T
    with np.errstate(over="ignore"):
        silu = gate / (1.0 + np.exp(-gate))
    h = round_to_bf16(silu * up)
    if act_mxfp8:
        h = mxfp8_round_rows(h)
    return h @ w_d.T


def expert_ffn(x_perm, offsets, w_gate_up, w_down, act_mxfp8: bool = False) -> np.ndarray:
    """Grouped expert FFN: rows [offsets[e], offsets[e+1]) go through expert e.

    x_perm: [rows, d] fp64 (exact bf16 values).  Returns y [rows, d] fp64.
    """
    x_perm = np.asarray(x_perm, dtype=np.float64)
    rows, d = x_perm.shape
    E = len(offsets) - 1
    y = np.zeros((rows, d), dtype=np.float64)
    for e in range(E):
        r0, r1 = int(offsets[e]), int(offsets[e + 1])
        if r1 > r0:
            y[r0:r1] = swiglu_ffn(x_perm[r0:r1], w_gate_up[e], w_down[e], act_mxfp8)
    return y


# --------------------------------------------------------------------------
# Combine
# --------------------------------------------------------------------------

def combine(y, slot_pos, gates, y_shared=None) -> np.ndarray:
    """out[t] = sum_j gates[t,j] * y[slot_pos[t,j]] (+ y_shared[t]), fp64."""
    slot_pos = np.asarray(slot_pos)
    T, k = slot_pos.shape
    out = np.zeros((T, y.shape[1]), dtype=np.float64)
    for j in range(k):
        out += np.asarray(gates)[:, j:j + 1] * y[slot_pos[:, j]]
    if y_shared is not None:
        out += y_shared
    return out


# --------------------------------------------------------------------------
# The whole layer
# --------------------------------------------------------------------------

def forward(x_bits, w_router, w_gate_up, w_down, top_k: int, router_bias=None,
            w_gate_up_shared=None, w_down_shared=None,
            bias_for_selection_only: bool = False, act_mxfp8: bool = False) -> dict:
    """Route -> group -> expert FFN -> combine, every intermediate returned.
    act_mxfp8: the expert GEMMs' token operands in MXFP8 (see swiglu_ffn)."""
    x_bits = np.asarray(x_bits, dtype=np.uint16)
    T = x_bits.shape[0]
    E = np.asarray(w_router).shape[0]
    ids, gates, logits = route(x_bits, w_router, top_k, router_bias, bias_for_selection_only)
    counts, offsets, perm, slot_pos = permute(ids, E)
    x = bf16_bits_to_f64(x_bits)
    x_perm = x[perm // top_k]
    y = expert_ffn(x_perm, offsets, w_gate_up, w_down, act_mxfp8)
    y_shared = None
    if w_gate_up_shared is not None:
        y_shared = swiglu_ffn(x, w_gate_up_shared, w_down_shared, act_mxfp8)
    out = combine(y, slot_pos, gates, y_shared)
    return dict(ids=ids, gates=gates, logits=logits, counts=counts,
                offsets=offsets, perm=perm, slot_pos=slot_pos, y=y,
                y_shared=y_shared, out=out, T=T)


def forward_tokens(x_bits, tokens, ids, gates, w_gate_up, w_down,
                   w_gate_up_shared=None, w_down_shared=None,
                   act_mxfp8: bool = False) -> np.ndarray:
    """Layer output for selected tokens only, given their routing.

    The same per-expert arithmetic as forward(), applied to the selected rows:
    out[t] = sum_j gates[t,j] * FFN_{ids[t,j]}(x[t]) (+ FFN_shared(x[t])).
    Used for sampled checks at sizes where the full layer is too slow here.
    ids/gates are [T,k] routing tables (from route()); tokens index into them.
    """
    tokens = np.asarray(tokens, dtype=np.int64)
    x = bf16_bits_to_f64(np.asarray(x_bits)[tokens])
    ids = np.asarray(ids)[tokens]
    gates = np.asarray(gates)[tokens]
    out = np.zeros_like(x)
    for e in np.unique(ids):
        rows, slots = np.nonzero(ids == e)
        y = swiglu_ffn(x[rows], w_gate_up[e], w_down[e], act_mxfp8)
        out[rows] += gates[rows, slots][:, None] * y
    if w_gate_up_shared is not None:
        out += swiglu_ffn(x, w_gate_up_shared, w_down_shared, act_mxfp8)
    return out
