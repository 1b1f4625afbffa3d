"""Full-size workloads, run exactly as the benchmark runs them (one
moe_forward call on the default workspace), checked against the oracle:
routing for every token, counts / offsets / permutation bit for bit, and the
whole layer output -- every element of every token except the listed
near-ties -- against the oracle's fp64 layer (one pass over the experts,
each expert's weights fetched once)."""

import numpy as np
import pytest
import torch

import oracle
from mixture_experts_layer_20_gb300 import counters
from mixture_experts_layer_20_gb300 import workloads as W
from tests import oracle_pool
from tests.gpu_util import ExpertsStreamed, assert_layer_close, compare_routing, f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    from mixture_experts_layer_20_gb300 import binding
    return binding


@pytest.mark.parametrize("name", [W.TINY, W.DECODE, W.PREFILL, W.SKEWED, W.DEEPSEEK])
def test_full_size_whole_layer(moe, name, report):
    w = W.WORKLOADS[name]
    p = W.make_weights(w, device="cuda")
    x = W.make_x(w, device="cuda")
    ws = moe.new_workspace(w.T, w.d, w.E, w.I, w.top_k, w.I_shared)
    out = moe.moe_forward(x, p["w_router"], p["w_gate_up"], p["w_down"], w.top_k, ws=ws,
                          router_bias=p["router_bias"], w_gate_up_shared=p["w_gate_up_shared"],
                          w_down_shared=p["w_down_shared"])
    assert moe.moe_get_device_status(ws) == moe.MOE_OK
    v = moe.workspace_views(ws, w.T, w.d, w.E, w.I, w.top_k, w.I_shared)
    bias = None if p["router_bias"] is None else p["router_bias"].cpu().numpy()
    ids_ref, gates_ref, logits = oracle.route(W.to_bits(x), W.to_bits(p["w_router"]), w.top_k, bias)
    ids = v["topk_ids"].cpu().numpy()
    differ = compare_routing(ids, v["topk_gates"].cpu().numpy(), ids_ref, gates_ref, logits, w.top_k)
    report(f"{name}: {differ.size} near-tie tokens routed differently: {differ.tolist()}")

    counts = v["expert_counts"].cpu().numpy()
    assert counts.sum() == w.T * w.top_k
    if differ.size == 0:
        c_ref, o_ref, p_ref, s_ref = oracle.permute(ids_ref, w.E)
        assert np.array_equal(counts, c_ref)
        assert np.array_equal(v["expert_offsets"].cpu().numpy(), o_ref)
        assert np.array_equal(v["perm"].cpu().numpy(), p_ref)
        assert np.array_equal(v["slot_pos"].cpu().numpy(), s_ref)
    else:  # the grouping is still the exact stable grouping of the GPU's own ids
        c_ref, o_ref, p_ref, s_ref = oracle.permute(ids, w.E)
        assert np.array_equal(v["perm"].cpu().numpy(), p_ref)
    if name == W.DECODE:
        active = int((counts > 0).sum())
        expect = counters.expected_active_experts(w.E, w.top_k, w.T)
        assert 120 <= active <= 128, (active, expect)

    tokens = np.setdiff1d(np.arange(w.T), differ)   # every token but the near-ties
    ref = oracle.forward_tokens(
        W.to_bits(x), tokens, ids_ref, gates_ref, ExpertsStreamed(p["w_gate_up"]),
        ExpertsStreamed(p["w_down"]),
        None if p["w_gate_up_shared"] is None else W.to_bits(p["w_gate_up_shared"]),
        None if p["w_down_shared"] is None else W.to_bits(p["w_down_shared"]))
    got = f64(out[torch.as_tensor(tokens, device="cuda")])
    assert got.shape == (w.T - differ.size, w.d)
    max_rel, mean_rel = assert_layer_close(got, ref, name)
    report(f"{name}: whole layer, {tokens.size} of {w.T} tokens x {w.d} columns: "
          f"max_rel={max_rel:.3e} mean_rel={mean_rel:.3e}")


@pytest.mark.parametrize("fmt", ["mxfp8", "nvfp4", "mxfp8_a8"])
def test_full_size_decode_quantised_weights(moe, fmt, report):
    """The decode workload with MXFP8 / NVFP4 expert weights (mxfp8_a8: MXFP8
    tokens too), as the benchmark runs it: routing for every token, and every
    token's output (all 64 x 4096 values but near-ties) against the oracle on
    its own quantisation of the experts' weights (and tokens)."""
    w = W.WORKLOADS[W.DECODE]
    p = W.make_weights(w, device="cuda")
    x = W.make_x(w, device="cuda")
    a8 = fmt == "mxfp8_a8"
    ws = moe.new_workspace(w.T, w.d, w.E, w.I, w.top_k, act_mxfp8=a8)
    if fmt in ("mxfp8", "mxfp8_a8"):
        out = moe.moe_forward_mxfp8(x, p["w_router"], moe.moe_mxfp8_quantize(p["w_gate_up"]),
                                    moe.moe_mxfp8_quantize(p["w_down"]), w.top_k, ws=ws,
                                    act_mxfp8=a8)
    else:
        out = moe.moe_forward_nvfp4(x, p["w_router"], moe.moe_nvfp4_quantize(p["w_gate_up"]),
                                    moe.moe_nvfp4_quantize(p["w_down"]), w.top_k, ws=ws)
    assert moe.moe_get_device_status(ws) == moe.MOE_OK
    v = moe.workspace_views(ws, w.T, w.d, w.E, w.I, w.top_k)
    ids_ref, gates_ref, logits = oracle.route(W.to_bits(x), W.to_bits(p["w_router"]), w.top_k)
    differ = compare_routing(v["topk_ids"].cpu().numpy(), v["topk_gates"].cpu().numpy(),
                             ids_ref, gates_ref, logits, w.top_k)
    tokens = np.setdiff1d(np.arange(w.T), differ)
    # the oracle quantises each expert itself; experts run in host worker processes
    ref = oracle_pool.layer_out(
        W.to_bits(x), ids_ref, gates_ref, w.E,
        lambda e: (W.to_bits(p["w_gate_up"][e]), W.to_bits(p["w_down"][e])), fmt=fmt)[tokens]
    got = f64(out[torch.as_tensor(tokens, device="cuda")])
    assert got.shape == (w.T - differ.size, w.d)
    max_rel, mean_rel = assert_layer_close(got, ref, f"decode {fmt}")
    report(f"decode {fmt}: whole layer, {tokens.size} of {w.T} tokens: "
          f"max_rel={max_rel:.3e} mean_rel={mean_rel:.3e}")
