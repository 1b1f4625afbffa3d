"""Planted mistakes in a copy of the oracle must be caught by the pins.

Each mutation loads a fresh copy of the oracle module, replaces one function
with a plausibly wrong version (a dropped term, a flipped sign, a swapped or
transposed operand, a wrong index or order) and runs every pin check; at least
one must fail.  This runs on the CPU only and never touches the real module.
"""

import importlib.util
import os

import numpy as np
import pytest

from tests import oracle_pins

ORACLE_FILE = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                           "oracle", "moe_oracle.py")


def _fresh_copy():
    spec = importlib.util.spec_from_file_location("oracle_mutant", ORACLE_FILE)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _m_silu_sign(o):
    def swiglu_ffn(x_rows, wgu, wd, act_mxfp8=False):
        wgu = o.bf16_bits_to_f64(wgu); wd = o.bf16_bits_to_f64(wd)
        I = wgu.shape[0] // 2
        g = x_rows @ wgu[:I].T; u = x_rows @ wgu[I:].T
        with np.errstate(over="ignore"):
            h = o.round_to_bf16(g / (1.0 + np.exp(g)) * u)
        return h @ wd.T
    o.swiglu_ffn = swiglu_ffn


def _m_gate_up_swapped(o):
    def swiglu_ffn(x_rows, wgu, wd, act_mxfp8=False):
        wgu = o.bf16_bits_to_f64(wgu); wd = o.bf16_bits_to_f64(wd)
        I = wgu.shape[0] // 2
        u = x_rows @ wgu[:I].T; g = x_rows @ wgu[I:].T
        with np.errstate(over="ignore"):
            h = o.round_to_bf16(g / (1.0 + np.exp(-g)) * u)
        return h @ wd.T
    o.swiglu_ffn = swiglu_ffn


def _m_no_h_rounding(o):
    def swiglu_ffn(x_rows, wgu, wd, act_mxfp8=False):
        wgu = o.bf16_bits_to_f64(wgu); wd = o.bf16_bits_to_f64(wd)
        I = wgu.shape[0] // 2
        g = x_rows @ wgu[:I].T; u = x_rows @ wgu[I:].T
        with np.errstate(over="ignore"):
            h = g / (1.0 + np.exp(-g)) * u
        return h @ wd.T
    o.swiglu_ffn = swiglu_ffn


def _m_down_transposed(o):
    def swiglu_ffn(x_rows, wgu, wd, act_mxfp8=False):
        wgu = o.bf16_bits_to_f64(wgu); wd = o.bf16_bits_to_f64(wd)
        I = wgu.shape[0] // 2
        g = x_rows @ wgu[:I].T; u = x_rows @ wgu[I:].T
        with np.errstate(over="ignore"):
            h = o.round_to_bf16(g / (1.0 + np.exp(-g)) * u)
        w = wd.reshape(wd.shape[1], wd.shape[0]).T  # wrong memory order
        return h @ w.T
    o.swiglu_ffn = swiglu_ffn


def _m_tie_high_index(o):
    def select_top_k(row, k):
        E = len(row)
        ranked = sorted(range(E), key=lambda e: (-row[e], -e))
        return sorted(ranked[:k])
    o.select_top_k = select_top_k


def _m_slots_by_logit(o):
    def select_top_k(row, k):
        E = len(row)
        return sorted(range(E), key=lambda e: (-row[e], e))[:k]
    o.select_top_k = select_top_k


def _m_no_renormalise(o):
    orig = o.route

    def route(x, wr, k, bias=None, sel_only=False):
        ids, gates, L = orig(x, wr, k, bias, sel_only)
        p = np.exp(L - L.max(axis=1, keepdims=True))
        p = p / p.sum(axis=1, keepdims=True)
        return ids, np.take_along_axis(p, ids.astype(np.int64), axis=1), L
    o.route = route


def _m_bias_dropped(o):
    orig = o.router_logits
    o.router_logits = lambda x, w, b=None: orig(x, w, None)


def _m_bf16_round_truncates(o):
    def round_to_bf16(x):
        x = np.asarray(x, dtype=np.float64)
        _, e = np.frexp(x)
        s = np.ldexp(1.0, np.maximum(e, -125) - 8)
        return np.trunc(x / s) * s
    o.round_to_bf16 = round_to_bf16


def _m_bf16_decode_shift(o):
    def bf16_bits_to_f64(bits):
        b = np.asarray(bits, dtype=np.uint16)
        return (b.astype(np.uint32) << np.uint32(15)).view(np.float32).astype(np.float64)
    o.bf16_bits_to_f64 = bf16_bits_to_f64


def _m_unstable_permute(o):
    def permute(ids, E):
        ids = np.asarray(ids); T, k = ids.shape
        flat = ids.reshape(-1)
        counts = np.bincount(flat, minlength=E).astype(np.int64)
        offsets = np.concatenate([[0], np.cumsum(counts)])
        nxt = offsets[1:].copy()
        perm = np.empty(T * k, np.int64); slot = np.empty(T * k, np.int64)
        for f in range(T * k):          # fills each range from the back
            e = flat[f]; nxt[e] -= 1
            perm[nxt[e]] = f; slot[f] = nxt[e]
        return counts, offsets, perm, slot.reshape(T, k)
    o.permute = permute


def _m_gather_wrong_index(o):
    orig_forward = o.forward

    def forward(x_bits, wr, wgu, wd, k, router_bias=None, w_gate_up_shared=None, w_down_shared=None,
                bias_for_selection_only=False, act_mxfp8=False):
        x_bits = np.asarray(x_bits, dtype=np.uint16)
        ids, gates, logits = o.route(x_bits, wr, k, router_bias, bias_for_selection_only)
        counts, offsets, perm, slot_pos = o.permute(ids, np.asarray(wr).shape[0])
        x = o.bf16_bits_to_f64(x_bits)
        x_perm = x[(perm % k) % x.shape[0]]       # token index taken modulo k
        y = o.expert_ffn(x_perm, offsets, wgu, wd, act_mxfp8)
        ys = (o.swiglu_ffn(x, w_gate_up_shared, w_down_shared, act_mxfp8)
              if w_gate_up_shared is not None else None)
        out = o.combine(y, slot_pos, gates, ys)
        return dict(ids=ids, gates=gates, logits=logits, counts=counts, offsets=offsets,
                    perm=perm, slot_pos=slot_pos, y=y, y_shared=ys, out=out, T=x.shape[0])
    assert orig_forward
    o.forward = forward


def _m_combine_ignores_gates(o):
    def combine(y, slot_pos, gates, y_shared=None):
        slot_pos = np.asarray(slot_pos)
        out = y[slot_pos].sum(axis=1)
        return out + y_shared if y_shared is not None else out
    o.combine = combine


def _m_combine_drops_shared(o):
    orig = o.combine
    o.combine = lambda y, s, g, ys=None: orig(y, s, g, None)


def _m_expert_shift(o):
    def expert_ffn(x_perm, offsets, wgu, wd, act_mxfp8=False):
        x_perm = np.asarray(x_perm, dtype=np.float64)
        E = len(offsets) - 1
        y = np.zeros_like(x_perm)
        for e in range(E):
            r0, r1 = int(offsets[e]), int(offsets[e + 1])
            if r1 > r0:
                y[r0:r1] = o.swiglu_ffn(x_perm[r0:r1], wgu[(e + 1) % E], wd[(e + 1) % E])
        return y
    o.expert_ffn = expert_ffn


def _m_forward_tokens_no_gate(o):
    def forward_tokens(x_bits, tokens, ids, gates, wgu, wd, wgus=None, wds=None, act_mxfp8=False):
        tokens = np.asarray(tokens)
        x = o.bf16_bits_to_f64(np.asarray(x_bits)[tokens])
        ids = np.asarray(ids)[tokens]
        out = np.zeros_like(x)
        for e in np.unique(ids):
            rows, _ = np.nonzero(ids == e)
            out[rows] += o.swiglu_ffn(x[rows], wgu[e], wd[e])
        if wgus is not None:
            out += o.swiglu_ffn(x, wgus, wds)
        return out
    o.forward_tokens = forward_tokens


def _m_selection_only_ignored(o):
    orig = o.route
    o.route = lambda x, wr, k, bias=None, sel_only=False: orig(x, wr, k, bias, False)


def _m_selection_only_unbiased_pick(o):
    orig = o.route

    def route(x, wr, k, bias=None, sel_only=False):
        if not sel_only:
            return orig(x, wr, k, bias, False)
        ids, gates, L = orig(x, wr, k, None, False)   # picks on the unbiased logits too
        return ids, gates, L
    o.route = route


def _m_mx_scale_off_by_one(o):
    o.E4M3_EMAX = 7


def _m_mx_truncates(o):
    orig = o.round_to_e4m3

    def round_to_e4m3(v):
        v = np.clip(np.asarray(v, dtype=np.float64), -448.0, 448.0)
        a = np.abs(v)
        with np.errstate(divide="ignore"):
            e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
        q = np.where(a >= 2.0 ** -6, 2.0 ** (np.maximum(e, -6) - 3), 2.0 ** -9)
        return np.floor(a / q) * q * np.sign(v)
    assert orig
    o.round_to_e4m3 = round_to_e4m3


def _m_mx_no_clamp(o):
    o.E4M3_MAX = 512.0


def _m_nv_no_tensor_scale(o):
    o.NV_TENSOR_DIV = np.float32(1.0)


def _m_nv_e2m1_truncates(o):
    def round_to_e2m1(v):
        v = np.asarray(v, dtype=np.float64)
        grid = o.e2m1_values()[:8]
        a = np.minimum(np.abs(v), 6.0)
        mag = np.searchsorted(grid, a, side="right") - 1   # the grid value at or below
        return np.where((v < 0) & (mag > 0), mag | 0x8, mag).astype(np.uint8)
    o.round_to_e2m1 = round_to_e2m1


def _m_nv_ties_away(o):
    def round_to_e2m1(v):
        v = np.asarray(v, dtype=np.float64)
        grid = o.e2m1_values()[:8]
        a = np.minimum(np.abs(v), 6.0)
        d = np.abs(a[..., None] - grid)
        best = d.min(axis=-1, keepdims=True)
        mag = 7 - np.argmax((d == best)[..., ::-1], axis=-1)   # the larger of a tie
        return np.where((v < 0) & (mag > 0), mag | 0x8, mag).astype(np.uint8)
    o.round_to_e2m1 = round_to_e2m1


def _m_nv_block_32(o):
    o.NV_BLOCK = 32


def _act_swiglu(o, quant_x, quant_h):
    """A swiglu_ffn whose activation quantisation steps are the given ones."""
    def swiglu_ffn(x_rows, wgu, wd, act_mxfp8=False):
        wgu = o.bf16_bits_to_f64(wgu); wd = o.bf16_bits_to_f64(wd)
        I = wgu.shape[0] // 2
        if act_mxfp8:
            x_rows = quant_x(x_rows)
        g = x_rows @ wgu[:I].T; u = x_rows @ wgu[I:].T
        with np.errstate(over="ignore"):
            h = g / (1.0 + np.exp(-g)) * u
        h = quant_h(h) if act_mxfp8 else o.round_to_bf16(h)
        return h @ wd.T
    return swiglu_ffn


def _m_act_h_before_round(o):
    # h micro-scaled before its bf16 rounding instead of after
    o.swiglu_ffn = _act_swiglu(o, o.mxfp8_round_rows,
                               lambda h: o.round_to_bf16(o.mxfp8_round_rows(h)))


def _m_act_x_skipped(o):
    o.swiglu_ffn = _act_swiglu(o, lambda x: x,
                               lambda h: o.mxfp8_round_rows(o.round_to_bf16(h)))


def _m_act_token_axis(o):
    # x's runs of 32 taken along the tokens instead of along d
    o.swiglu_ffn = _act_swiglu(o, lambda x: o.mxfp8_round_rows(x.T).T,
                               lambda h: o.mxfp8_round_rows(o.round_to_bf16(h)))


MUTATIONS = [
    _m_silu_sign, _m_gate_up_swapped, _m_no_h_rounding, _m_down_transposed,
    _m_tie_high_index, _m_slots_by_logit, _m_no_renormalise, _m_bias_dropped,
    _m_bf16_round_truncates, _m_bf16_decode_shift, _m_unstable_permute,
    _m_gather_wrong_index, _m_combine_ignores_gates, _m_combine_drops_shared,
    _m_expert_shift, _m_forward_tokens_no_gate, _m_selection_only_ignored,
    _m_selection_only_unbiased_pick, _m_mx_scale_off_by_one, _m_mx_truncates, _m_mx_no_clamp,
    _m_nv_no_tensor_scale, _m_nv_e2m1_truncates, _m_nv_ties_away, _m_nv_block_32,
    _m_act_h_before_round, _m_act_x_skipped, _m_act_token_axis,
]


@pytest.mark.parametrize("mutate", MUTATIONS, ids=lambda m: m.__name__[3:])
def test_planted_mistake_is_caught(mutate):
    o = _fresh_copy()
    mutate(o)
    caught = []
    for check in oracle_pins.ALL_CHECKS:
        try:
            check(o)
        except TypeError as exc:  # a mutant with the wrong signature proves nothing
            raise AssertionError(f"{mutate.__name__} does not fit {check.__name__}: {exc}")
        except Exception as exc:  # AssertionError, or a shape error the mistake causes
            caught.append((check.__name__, type(exc).__name__))
    assert caught, f"no pin catches {mutate.__name__}"
