"""Checks that pin the CPU oracle to facts other than itself.

Each check takes the oracle module as an argument and raises AssertionError on
a mismatch, so the same checks run against the real oracle (test_oracle_pins)
and against copies with a planted mistake (test_oracle_mutations), where at
least one of them must fail.

What pins what:
  bf16 decode / rounding ....... torch's own bf16 conversions (library routine)
  router logits ................ one-hot tokens: logits are columns of W_r (closed form)
  top-k set .................... brute force over all k-subsets (max logit sum)
  tie-break .................... duplicated router rows give exact ties
  gates ........................ k = E: scipy softmax; k = 1: exactly 1; subset-softmax identity
  selection-only bias .......... k = E: scipy softmax of the unbiased logits; k = 2 with a
                                 dominant bias: the forced expert plus the unbiased argmax,
                                 gates = scipy expit of the unbiased logit difference
  grouping ..................... numpy's stable argsort / bincount (library routines)
  SwiGLU expert ................ a hand-computed one-element example; torch silu dense FFN
  whole layer .................. brute-force dense form: every expert on every token,
                                 masked by the routing (no grouping, no permutation)
  shared expert, linearity ..... identical experts, exact power-of-two scaling
  MXFP8 ........................ E4M3 decode and rounding against torch.float8_e4m3fn; block
                                 scales from numpy frexp; codes against torch's conversion of the
                                 scaled, clamped block; exact round trip of representable values
  MXFP8 activations ............ one expert, every token routed to it: the layer equals a dense
                                 FFN whose x and bf16 h are micro-scaled independently (frexp
                                 scales, torch's E4M3 conversion); quantising twice = once
"""

from __future__ import annotations

import itertools
import math

import numpy as np
import scipy.special
import torch


def _rng(seed):
    return np.random.default_rng(seed)


def _bf16_bits_from_f32(v):
    t = torch.from_numpy(np.asarray(v, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def _random_layer(seed, T, d, E, I, scale_x=1.0):
    r = _rng(seed)
    x = _bf16_bits_from_f32(r.standard_normal((T, d)) * scale_x)
    wr = _bf16_bits_from_f32(r.standard_normal((E, d)) / math.sqrt(d))
    wgu = _bf16_bits_from_f32(r.standard_normal((E, 2 * I, d)) / math.sqrt(d))
    wd = _bf16_bits_from_f32(r.standard_normal((E, d, I)) / math.sqrt(I))
    return x, wr, wgu, wd


def _dec(bits):
    """bf16 bits -> float64 through torch (independent of the oracle)."""
    t = torch.from_numpy(np.asarray(bits, dtype=np.uint16).view(np.int16)).view(torch.bfloat16)
    return t.to(torch.float64).numpy()


def _dense_ffn_torch(o, x64, wgu_bits, wd_bits):
    """Textbook SwiGLU with torch's silu; h rounded by the (separately pinned)
    oracle bf16 rounding."""
    wgu = torch.from_numpy(_dec(wgu_bits))
    wd = torch.from_numpy(_dec(wd_bits))
    I = wgu.shape[0] // 2
    x = torch.from_numpy(x64)
    h = torch.nn.functional.silu(x @ wgu[:I].T) * (x @ wgu[I:].T)
    h = torch.from_numpy(o.round_to_bf16(h.numpy()))
    return (h @ wd.T).numpy()


def _rel(a, b):
    return float(np.abs(a - b).max() / max(np.abs(b).max(), 1e-300))


# ---------------------------------------------------------------- bf16

def check_bf16_decode(o):
    r = _rng(1)
    bits = r.integers(0, 1 << 16, size=20000, dtype=np.uint32).astype(np.uint16)
    exp = (bits >> 7) & 0xFF
    bits = bits[exp != 0xFF]  # finite values only
    assert np.array_equal(o.bf16_bits_to_f64(bits), _dec(bits))


def check_bf16_round(o):
    r = _rng(2)
    v = np.concatenate([
        r.standard_normal(20000),
        r.standard_normal(2000) * 1e-39,   # bf16 subnormal range
        r.standard_normal(2000) * 1e30,
        [0.0, -0.0, 1.0, -1.5],
    ]).astype(np.float32)
    # exact midpoints between adjacent bf16 values: ties must go to even
    base = _bf16_bits_from_f32(r.standard_normal(4000))
    lo = (base.astype(np.uint32) << 16).view(np.float32)
    hi = ((base.astype(np.uint32) + 1) << 16).view(np.float32)
    mid = ((lo.astype(np.float64) + hi.astype(np.float64)) / 2).astype(np.float32)
    v = np.concatenate([v, mid[np.isfinite(mid)]])
    want = torch.from_numpy(v).to(torch.bfloat16).to(torch.float64).numpy()
    got = o.round_to_bf16(v.astype(np.float64))
    assert np.array_equal(got, want)
    assert np.array_equal(o.f64_to_bf16_bits(v.astype(np.float64)), _bf16_bits_from_f32(v))


# ---------------------------------------------------------------- router

def check_logits_one_hot(o):
    r = _rng(3)
    T, d, E = 12, 64, 8
    hot = r.integers(0, d, size=T)
    x = np.zeros((T, d), dtype=np.float32)
    x[np.arange(T), hot] = 1.0
    wr = _bf16_bits_from_f32(r.standard_normal((E, d)))
    bias = r.standard_normal(E).astype(np.float32)
    L = o.router_logits(_bf16_bits_from_f32(x), wr, bias)
    want = _dec(wr)[:, hot].T + bias.astype(np.float64)[None, :]
    assert np.array_equal(L, want)


def check_topk_brute_force(o):
    for (E, k, seed) in [(8, 1, 4), (8, 2, 5), (8, 3, 6), (6, 6, 7), (9, 4, 8)]:
        x, wr, _, _ = _random_layer(seed, 24, 64, E, 8)
        ids, gates, L = o.route(x, wr, k)
        for t in range(24):
            best = max(itertools.combinations(range(E), k),
                       key=lambda s: sum(L[t, list(s)]))
            assert list(ids[t]) == list(best), (E, k, t)


def check_tie_break(o):
    r = _rng(9)
    d, E, k = 64, 6, 2
    x = _bf16_bits_from_f32(np.abs(r.standard_normal((5, d))))
    w = np.zeros((E, d), dtype=np.float32)
    w[0] = 1.0            # largest logit
    w[2] = 0.5            # tied for second place with expert 5
    w[5] = 0.5
    w[1] = w[3] = w[4] = -1.0
    ids, gates, _ = o.route(x, _bf16_bits_from_f32(w), k)
    assert (ids == np.array([0, 2])).all()
    # all logits equal: the k lowest indices win, equal gates
    ids, gates, _ = o.route(x, _bf16_bits_from_f32(np.zeros((E, d), np.float32)), 3)
    assert (ids == np.array([0, 1, 2])).all()
    assert np.allclose(gates, 1.0 / 3.0, rtol=0, atol=1e-15)


def check_gates(o):
    x, wr, _, _ = _random_layer(10, 32, 64, 8, 8)
    ids, gates, L = o.route(x, wr, 8)          # k = E: the full softmax
    assert (ids == np.arange(8)).all()
    assert np.allclose(gates, scipy.special.softmax(L, axis=1), rtol=1e-13, atol=0)
    ids, gates, L = o.route(x, wr, 1)          # k = 1: gate is exactly one
    assert (gates == 1.0).all()
    assert (ids[:, 0] == np.argmax(L, axis=1)).all()
    bias = _rng(11).standard_normal(8).astype(np.float32) * 3
    ids, gates, L = o.route(x, wr, 3, bias)
    assert np.allclose(gates.sum(axis=1), 1.0, rtol=0, atol=1e-14)
    sel = np.take_along_axis(L, ids.astype(np.int64), axis=1)
    assert np.allclose(gates, scipy.special.softmax(sel, axis=1), rtol=1e-13, atol=0)
    # the chosen k beat every other expert
    for t in range(L.shape[0]):
        rest = np.setdiff1d(np.arange(8), ids[t])
        assert L[t, ids[t]].min() >= L[t, rest].max()


def check_selection_only_bias(o):
    x, wr, _, _ = _random_layer(13, 24, 64, 8, 8)
    bias = _rng(14).standard_normal(8).astype(np.float32) * 3
    L0 = _dec(x) @ _dec(wr).T                      # unbiased logits, computed here
    # k = E: every expert chosen, gates = the softmax of the unbiased logits
    ids, gates, _ = o.route(x, wr, 8, bias, True)
    assert (ids == np.arange(8)).all()
    assert np.allclose(gates, scipy.special.softmax(L0, axis=1), rtol=1e-12, atol=0)
    # the biased variant differs (the bias is large), so the check discriminates
    _, gates_b, _ = o.route(x, wr, 8, bias, False)
    assert np.abs(gates_b - gates).max() > 1e-3
    # k = 2 with a dominant bias on expert 5: expert 5 is always chosen with the
    # unbiased argmax of the others; the gates are a logistic of the unbiased gap
    big = np.zeros(8, dtype=np.float32)
    big[5] = 1e4
    ids, gates, _ = o.route(x, wr, 2, big, True)
    for t in range(L0.shape[0]):
        others = [e for e in range(8) if e != 5]
        second = others[int(np.argmax(L0[t, others]))]
        assert sorted(ids[t].tolist()) == sorted([5, second])
        g5 = gates[t, list(ids[t]).index(5)]
        assert abs(g5 - scipy.special.expit(L0[t, 5] - L0[t, second])) < 1e-12
    # the selection itself is the biased one
    ids_sel, _, _ = o.route(x, wr, 3, bias, True)
    ids_b, _, _ = o.route(x, wr, 3, bias, False)
    assert (ids_sel == ids_b).all()


def check_mxfp8(o):
    # decode of every code = torch's float8_e4m3fn decode
    ref = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn)
    ref = ref.to(torch.float64).numpy()
    mine = o.e4m3_values()
    assert np.array_equal(np.isnan(mine), np.isnan(ref))
    assert np.array_equal(mine[~np.isnan(ref)], ref[~np.isnan(ref)])
    # rounding = torch's conversion (nearest, ties to even) on [-448, 448], incl. subnormals and ties
    r = _rng(15)
    v = np.concatenate([r.uniform(-448, 448, 4000), r.uniform(-2**-5, 2**-5, 4000),
                        np.arange(-64, 65) * 2.0 ** -10, np.arange(-14, 14) * 2.0 ** 5 + 2.0 ** 4])
    v = v.astype(np.float32).astype(np.float64)
    torch_r = torch.from_numpy(v).to(torch.float32).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(o.round_to_e4m3(v), torch_r)
    # quantisation of blocks with a spread of magnitudes
    w = (r.standard_normal((6, 128)) * np.exp(r.uniform(-8, 4, (6, 1)))).astype(np.float32)
    w[2, 32:64] = 0.0                                   # an all-zero block
    w[3, :32] = 3.5 * 2.0 ** r.integers(-6, 5, 32)       # on the block's grid: exactly representable
    codes, scales = o.mxfp8_quantize(w.astype(np.float64))
    blocks = w.astype(np.float64).reshape(6, 4, 32)
    amax = np.abs(blocks).max(axis=-1)
    mant, expo = np.frexp(amax)                          # amax = mant * 2^expo, mant in [0.5, 1)
    xexp = np.where(amax > 0, expo - 1 - 8, -127)
    assert np.array_equal(scales.astype(np.int64), np.where(amax > 0, xexp + 127, 0))
    scaled = np.clip(blocks / 2.0 ** xexp[..., None], -448, 448).astype(np.float32)
    ref_codes = torch.from_numpy(scaled).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    ref_codes = np.where(ref_codes == 0x80, 0, ref_codes)   # -0 encodes as +0
    assert np.array_equal(codes.reshape(6, 4, 32), ref_codes)
    back = o.mxfp8_dequantize(codes, scales)
    assert np.array_equal(back[3, :32], w[3, :32].astype(np.float64))   # exact round trip
    assert (back[2, 32:64] == 0).all()
    nz = amax > 0
    top = np.abs(o.e4m3_values()[codes.reshape(6, 4, 32)]).max(axis=-1)
    assert ((top[nz] >= 256) & (top[nz] <= 448)).all()   # the largest maps into the top binade


def _mx_round_torch(v):
    """MXFP8 quantise-dequantise of [m, K] rows in runs of 32 along K, without
    the oracle: numpy frexp for the block exponent, torch for the E4M3 rounding."""
    m, K = v.shape
    blocks = v.reshape(m, K // 32, 32)
    amax = np.abs(blocks).max(axis=-1)
    _, expo = np.frexp(amax)
    xexp = np.where(amax > 0, expo - 1 - 8, -127).astype(np.float64)
    scaled = np.clip(blocks / 2.0 ** xexp[..., None], -448, 448).astype(np.float32)
    q = torch.from_numpy(scaled).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    return (q * 2.0 ** xexp[..., None]).reshape(m, K)


def check_act_mxfp8(o):
    T, d, I = 32, 64, 64
    r = _rng(21)
    x = _bf16_bits_from_f32(r.standard_normal((T, d)) * np.exp(r.uniform(-3, 3, (T, 1))))
    wr = _bf16_bits_from_f32(r.standard_normal((1, d)))
    wgu = _bf16_bits_from_f32(r.standard_normal((1, 2 * I, d)) / 8)
    wd = _bf16_bits_from_f32(r.standard_normal((1, d, I)) / 8)
    got = o.forward(x, wr, wgu, wd, 1, act_mxfp8=True)["out"]
    # independent dense form: x and h micro-scaled by _mx_round_torch, h rounded to bf16 by torch
    xq = _mx_round_torch(_dec(x))
    g = xq @ _dec(wgu[0][:I]).T
    u = xq @ _dec(wgu[0][I:]).T
    with np.errstate(over="ignore"):
        h = torch.from_numpy(g / (1.0 + np.exp(-g)) * u).to(torch.bfloat16).to(torch.float64).numpy()
    ref = _mx_round_torch(h) @ _dec(wd[0]).T
    assert _rel(got, ref) < 1e-12
    # the quantisation changes the layer (so the check above sees it) ...
    plain = o.forward(x, wr, wgu, wd, 1)["out"]
    assert _rel(plain, ref) > 1e-4
    # ... and values already on the MXFP8 grid go through unchanged
    once = o.mxfp8_round_rows(_dec(x))
    assert np.array_equal(once, xq)
    assert np.array_equal(o.mxfp8_round_rows(once), once)


def check_nvfp4(o):
    """E2M1 grid and rounding, NVFP4 scales and codes."""
    vals = o.e2m1_values()
    pos = vals[:8]
    # a float format's positive codes increase with the code; 16 codes, sign in bit 3
    assert np.all(np.diff(pos) > 0) and pos[0] == 0 and pos[-1] == 6.0
    assert np.array_equal(vals[8:], -pos) and np.sum(vals == 0) == 2
    # each magnitude has at most two significant bits and is a multiple of 0.5
    m, _ = np.frexp(pos[1:])
    assert set(np.round(m * 4).astype(int)) <= {2, 3}
    assert np.array_equal(np.round(pos * 2), pos * 2)
    # decode then round is the identity (+0 for -0)
    codes = np.arange(16)
    back = o.round_to_e2m1(vals)
    assert np.array_equal(back, np.where(codes == 8, 0, codes))
    # rounding = nearest by brute force; exact midpoints go to the code with mantissa bit 0
    r = _rng(31)
    v = np.concatenate([r.uniform(-7, 7, 4000), (pos[:-1] + pos[1:]) / 2,
                        -(pos[:-1] + pos[1:]) / 2, [6.5, -100.0, 1e-9]])
    got = o.round_to_e2m1(v)
    for x, c in zip(v, got):
        a = min(abs(x), 6.0)
        dist = np.abs(pos - a)
        near = np.flatnonzero(dist == dist.min())
        want = near[0] if len(near) == 1 else [n for n in near if n % 2 == 0][0]
        if x < 0 and want > 0:
            want |= 8
        assert c == want, (x, c, want)
    # quantisation: scales through torch's E4M3 conversion, codes by nearest search
    w = (r.standard_normal((6, 64)) * np.exp(r.uniform(-6, 2, (6, 1)))).astype(np.float32)
    w[1, 16:32] = 0.0                                            # an all-zero block
    codes, scales, g = o.nvfp4_quantize(w)
    amax = np.float32(np.abs(w).max())
    assert g == amax / np.float32(2688.0)
    amax_b = np.abs(w.reshape(6, 4, 16)).max(axis=-1).astype(np.float32)
    s = torch.from_numpy((amax_b / np.float32(6.0)) / g).to(torch.float8_e4m3fn)
    assert np.array_equal(scales, s.view(torch.uint8).numpy())
    s_val = s.to(torch.float64).numpy().astype(np.float32)
    denom = (s_val * g).astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        x = np.where(denom[..., None] > 0, w.reshape(6, 4, 16) / denom[..., None], 0).astype(np.float32)
    assert np.array_equal(codes.reshape(6, 4, 16), o.round_to_e2m1(x.astype(np.float64)))
    assert (codes.reshape(6, 4, 16)[1, 1] == 0).all() and scales[1, 1] == 0
    # the largest magnitude of every non-zero block lands on 6 (its scale is within 1/16)
    top = np.abs(o.e2m1_values()[codes.reshape(6, 4, 16)]).max(axis=-1)
    assert np.all(top[amax_b > 0] == 6.0)
    # error bound: half an E2M1 step (at most 1) times the block's scale
    deq = o.nvfp4_dequantize(codes, scales, g)
    step = np.where(np.abs(x) < 2, 0.5, np.where(np.abs(x) < 4, 1.0, 2.0))
    assert np.all(np.abs(deq - w.reshape(6, 64)) <= (0.5 * step * denom[..., None]).reshape(6, 64) * (1 + 1e-6))
    # values on the grid come back exactly: a block whose largest element is 6 x s x 2^-10
    # (s an E4M3 value, one block with s = 448 so that the tensor scale is 2^-10; two
    # blocks with subnormal E4M3 scales, 2^-8 and 3 x 2^-9)
    bs = np.array([[448.0, 0.75, 2.0 ** -8], [13.0, 2.0 ** -3, 3 * 2.0 ** -9]])
    grid = o.e2m1_values()[r.integers(0, 16, (2, 3, 16))] * bs[..., None] * 2.0 ** -10
    grid[..., 0] = 6 * bs * 2.0 ** -10
    grid = grid.reshape(2, 48)
    c2, s2, g2 = o.nvfp4_quantize(grid.astype(np.float32))
    assert g2 == np.float32(2.0 ** -10)
    assert np.array_equal(o.e4m3_values()[s2], bs)
    assert np.array_equal(o.nvfp4_dequantize(c2, s2, g2), grid)
    # an all-zero matrix: tensor scale 1, every code and scale 0
    c3, s3, g3 = o.nvfp4_quantize(np.zeros((2, 32), np.float32))
    assert g3 == 1.0 and not c3.any() and not s3.any()


# ---------------------------------------------------------------- grouping

def check_permute(o):
    r = _rng(12)
    for (T, E, k) in [(50, 8, 2), (37, 16, 4), (1, 5, 5), (200, 64, 8)]:
        ids = np.stack([np.sort(r.choice(E, size=k, replace=False)) for _ in range(T)])
        ids[: T // 3] = np.sort(r.choice(max(k, E // 2), size=k, replace=False))  # skew
        counts, offsets, perm, slot_pos = o.permute(ids, E)
        flat = ids.reshape(-1)
        assert np.array_equal(counts, np.bincount(flat, minlength=E))
        assert counts.sum() == T * k
        assert np.array_equal(offsets, np.concatenate([[0], np.cumsum(counts)]))
        assert np.array_equal(perm, np.argsort(flat, kind="stable"))
        inv = np.empty(T * k, dtype=np.int64)
        inv[perm] = np.arange(T * k)
        assert np.array_equal(slot_pos.reshape(-1), inv)


# ---------------------------------------------------------------- expert FFN

SWIGLU_HAND = [
    # (gate pre-activation G, up U, expected bf16 h)
    # h = G / (1 + exp(-G)) * U rounded to bf16 by hand:
    # G=2, U=3: 5.28478...; bf16 spacing in [4,8) is 2^-5 -> 169 * 2^-5 = 5.28125
    (2.0, 3.0, 5.28125),
    # G=-2, U=3: -0.715217...; spacing in [0.5,1) is 2^-8 -> -183 * 2^-8 = -0.71484375
    (-2.0, 3.0, -0.71484375),
    # G=0: silu(0) = 0 whatever U is
    (0.0, 7.0, 0.0),
]


def check_swiglu_hand_example(o):
    d = 64
    for (G, U, h) in SWIGLU_HAND:
        wgu = np.zeros((2, d), dtype=np.float32)
        wgu[0, 0] = G
        wgu[1, 0] = U
        wd = np.zeros((d, 1), dtype=np.float32)
        wd[0, 0] = 1.0
        wd[5, 0] = -2.0
        x = np.zeros((1, d))
        x[0, 0] = 1.0
        y = o.swiglu_ffn(x, _bf16_bits_from_f32(wgu), _bf16_bits_from_f32(wd))
        want = np.zeros((1, d))
        want[0, 0] = h
        want[0, 5] = -2.0 * h
        assert np.array_equal(y, want), (G, U, y[0, :6])


def check_single_expert_is_dense_ffn(o):
    T, d, E, I = 24, 64, 6, 32
    x, wr, wgu, wd = _random_layer(13, T, d, E, I)
    bias = np.zeros(E, dtype=np.float32)
    bias[2] = 1e4                                  # every token picks expert 2
    res = o.forward(x, wr, wgu, wd, 1, router_bias=bias)
    assert (res["ids"] == 2).all() and (res["gates"] == 1.0).all()
    want = _dense_ffn_torch(o, _dec(x), wgu[2], wd[2])
    assert _rel(res["out"], want) < 1e-12


def check_identical_experts(o):
    T, d, E, I = 20, 64, 8, 32
    x, wr, wgu, wd = _random_layer(14, T, d, E, I)
    wgu = np.broadcast_to(wgu[3], wgu.shape).copy()
    wd = np.broadcast_to(wd[3], wd.shape).copy()
    res = o.forward(x, wr, wgu, wd, 3)
    want = _dense_ffn_torch(o, _dec(x), wgu[0], wd[0])
    assert _rel(res["out"], want) < 1e-12
    # an always-on shared expert equal to them doubles the output
    res = o.forward(x, wr, wgu, wd, 3, w_gate_up_shared=wgu[0], w_down_shared=wd[0])
    assert _rel(res["out"], 2 * want) < 1e-12


def _brute_force_layer(o, x, wr, wgu, wd, k, bias=None):
    """Every expert on every token, masked by the routing: no grouping step."""
    xd = torch.from_numpy(_dec(x))
    L = (xd @ torch.from_numpy(_dec(wr)).T).numpy()
    if bias is not None:
        L = L + np.asarray(bias, np.float64)[None, :]
    T, E = L.shape
    order = np.lexsort((np.tile(np.arange(E), (T, 1)), -L), axis=1)[:, :k]
    mask = np.zeros((T, E))
    np.put_along_axis(mask, order, 1.0, axis=1)
    g = np.where(mask > 0, scipy.special.softmax(np.where(mask > 0, L, -np.inf), axis=1), 0.0)
    out = np.zeros((T, x.shape[1]))
    for e in range(E):
        out += g[:, e:e + 1] * _dense_ffn_torch(o, xd.numpy(), wgu[e], wd[e])
    return out


def check_brute_force_layer(o):
    for (T, d, E, I, k, seed) in [(40, 64, 8, 32, 2, 15), (33, 128, 16, 64, 4, 16)]:
        x, wr, wgu, wd = _random_layer(seed, T, d, E, I)
        bias = _rng(seed).standard_normal(E).astype(np.float32)
        res = o.forward(x, wr, wgu, wd, k, router_bias=bias)
        want = _brute_force_layer(o, x, wr, wgu, wd, k, bias)
        assert _rel(res["out"], want) < 1e-12


def check_down_scaling(o):
    T, d, E, I = 16, 64, 8, 32
    x, wr, wgu, wd = _random_layer(17, T, d, E, I)
    a = o.forward(x, wr, wgu, wd, 2)["out"]
    wd2 = _bf16_bits_from_f32(_dec(wd) * 2.0)
    b = o.forward(x, wr, wgu, wd2, 2)["out"]
    assert np.array_equal(b, 2.0 * a)


def check_forward_tokens(o):
    T, d, E, I, k = 30, 64, 8, 32, 3
    x, wr, wgu, wd = _random_layer(18, T, d, E, I)
    r = _rng(18)
    wgus = _bf16_bits_from_f32(r.standard_normal((2 * I, d)) / 8)
    wds = _bf16_bits_from_f32(r.standard_normal((d, I)) / 6)
    res = o.forward(x, wr, wgu, wd, k, w_gate_up_shared=wgus, w_down_shared=wds)
    toks = [0, 7, 29, 13]
    part = o.forward_tokens(x, toks, res["ids"], res["gates"], wgu, wd, wgus, wds)
    assert _rel(part, res["out"][toks]) < 1e-13


ALL_CHECKS = [
    check_bf16_decode, check_bf16_round, check_logits_one_hot,
    check_topk_brute_force, check_tie_break, check_gates, check_selection_only_bias, check_mxfp8,
    check_act_mxfp8,
    check_nvfp4,
    check_permute,
    check_swiglu_hand_example, check_single_expert_is_dense_ffn,
    check_identical_experts, check_brute_force_layer, check_down_scaling,
    check_forward_tokens,
]
