"""The whole layer as one kernel launch (moe_forward_ext_t.single_launch),
through the C ABI, against the oracle: routing bit for bit except near-ties
(its router sums 128-wide ranges of d), counts / offsets / permutation of its
own routing bit for bit, y and out within the layer tolerance.  Also: the
same layer as the multi-launch path, repeated launches (the grid-barrier
counters return to zero), a forced barrier timeout that returns
MOE_ERR_TIMEOUT and leaves the next call correct, and a captured graph."""

import numpy as np
import pytest
import torch

import oracle
from mixture_experts_layer_20_gb300 import workloads as W
from tests.gpu_util import ExpertsOnHost, assert_layer_close, compare_routing, f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    from mixture_experts_layer_20_gb300 import binding
    return binding


def _run(moe, w, p, x, ws=None, **kw):
    ws = ws if ws is not None else moe.new_workspace(w.T, w.d, w.E, w.I, w.top_k)
    out = moe.moe_forward(x, p["w_router"], p["w_gate_up"], p["w_down"], w.top_k, ws=ws,
                          router_bias=p["router_bias"], single_launch=True, **kw)
    return out, ws


CASES = [
    # T, d, E, k, I, zipf, selection-only bias
    (64, 512, 32, 8, 256, False, False),    # 16 rows per expert: some experts in two passes
    (1, 256, 8, 2, 128, False, False),      # one token
    (64, 4096, 128, 8, 1536, False, False), # the Qwen3-235B-A22B decode layer's shapes
    (80, 384, 20, 4, 128, True, False),     # E not a multiple of 16, router bias
    (40, 768, 256, 8, 384, True, True),     # 256 experts, bias used for selection only
    (16, 256, 8, 8, 128, False, False),     # k = E
    (17, 640, 16, 1, 256, False, False),    # k = 1: gate exactly 1
    (512, 256, 256, 8, 128, False, False),  # the limits: T k = 4096, 16 rows per expert
]


@pytest.mark.parametrize("T,d,E,k,I,zipf,sel", CASES)
def test_single_launch_matches_oracle(moe, T, d, E, k, I, zipf, sel):
    w = W.Workload("fused", T, d, E, k, I, zipf_bias=zipf, seed=T + d + E)
    p = W.make_weights(w, device="cuda")
    x = W.make_x(w, device="cuda")
    out, ws = _run(moe, w, p, x, bias_selection_only=sel)
    assert moe.moe_get_device_status(ws) == moe.MOE_OK
    v = moe.workspace_views(ws, T, d, E, I, k)
    bias = None if p["router_bias"] is None else p["router_bias"].cpu().numpy()
    ids_ref, gates_ref, logits = oracle.route(W.to_bits(x), W.to_bits(p["w_router"]), k, bias,
                                              bias_for_selection_only=sel)
    ids = v["topk_ids"].cpu().numpy()
    differ = compare_routing(ids, v["topk_gates"].cpu().numpy(), ids_ref, gates_ref, logits, k)
    # the grouping of the kernel's own routing, bit for bit
    c_ref, o_ref, p_ref, s_ref = oracle.permute(ids, E)
    assert np.array_equal(v["expert_counts"].cpu().numpy(), c_ref)
    assert np.array_equal(v["expert_offsets"].cpu().numpy(), o_ref)
    assert np.array_equal(v["perm"].cpu().numpy(), p_ref)
    assert np.array_equal(v["slot_pos"].cpu().numpy(), s_ref)
    # y of the kernel's own grouping, and out on the tokens routed as the oracle did
    xb = W.to_bits(x)
    y_ref = oracle.expert_ffn(oracle.bf16_bits_to_f64(xb)[p_ref // k], o_ref,
                              ExpertsOnHost(p["w_gate_up"]), ExpertsOnHost(p["w_down"]))
    assert_layer_close(f64(v["y"]), y_ref, "y")
    tokens = np.setdiff1d(np.arange(T), differ)
    ref = oracle.forward_tokens(xb, tokens, ids_ref, gates_ref, ExpertsOnHost(p["w_gate_up"]),
                                ExpertsOnHost(p["w_down"]))
    max_rel, mean_rel = assert_layer_close(f64(out)[tokens], ref, "out")
    print(f"single launch T={T} d={d} E={E} k={k}: max_rel={max_rel:.2e} "
          f"mean_rel={mean_rel:.2e} near-ties {differ.tolist()}")


def test_single_launch_agrees_with_multi_launch_and_repeats(moe):
    w = W.Workload("fused_rep", 64, 1024, 64, 8, 512, seed=5)
    p = W.make_weights(w, device="cuda")
    x = W.make_x(w, device="cuda")
    ws = moe.new_workspace(w.T, w.d, w.E, w.I, w.top_k)
    first, _ = _run(moe, w, p, x, ws=ws)
    first = first.clone()
    for _ in range(5):  # the barrier words return to zero after every launch
        again, _ = _run(moe, w, p, x, ws=ws)
        assert torch.equal(again, first)
    assert moe.moe_get_device_status(ws) == moe.MOE_OK
    multi = moe.moe_forward(x, p["w_router"], p["w_gate_up"], p["w_down"], w.top_k)
    assert_layer_close(f64(first), f64(multi), "single vs multi launch")


def test_single_launch_barrier_timeout_is_reported_and_recovers(moe):
    w = W.Workload("fused_tmo", 64, 512, 32, 8, 256, seed=9)
    p = W.make_weights(w, device="cuda")
    x = W.make_x(w, device="cuda")
    ws = moe.new_workspace(w.T, w.d, w.E, w.I, w.top_k)
    good, _ = _run(moe, w, p, x, ws=ws)
    good = good.clone()
    assert moe.moe_get_device_status(ws) == moe.MOE_OK
    moe.moe_set_wait_timeout_ns(1)  # a barrier not already complete gives up at once
    try:
        _run(moe, w, p, x, ws=ws)
        st = moe.moe_get_device_status(ws)
    finally:
        moe.moe_set_wait_timeout_ns(0)
    assert st == moe.MOE_ERR_TIMEOUT
    again, _ = _run(moe, w, p, x, ws=ws)
    assert moe.moe_get_device_status(ws) == moe.MOE_OK
    assert torch.equal(again, good)


def test_single_launch_graph_replay(moe):
    w = W.Workload("fused_graph", 64, 512, 32, 8, 256, seed=11)
    p = W.make_weights(w, device="cuda")
    x = W.make_x(w, device="cuda")
    ws = moe.new_workspace(w.T, w.d, w.E, w.I, w.top_k)
    want, _ = _run(moe, w, p, x, ws=ws)
    want = want.clone()
    out = torch.empty_like(want)
    g = moe.ForwardGraph(x, p["w_router"], p["w_gate_up"], p["w_down"], w.top_k, out, ws,
                         single_launch=True)
    n0 = moe.moe_launch_count()
    g.launch()
    torch.cuda.synchronize()
    assert moe.moe_launch_count() - n0 == 1  # one kernel per replay
    assert torch.equal(out, want)
    g.close()


def test_single_launch_rejects_unsupported(moe):
    w = W.Workload("fused_bad", 600, 512, 8, 4, 256, seed=3)  # 300 rows per expert: not decode
    p = W.make_weights(w, device="cuda")
    x = W.make_x(w, device="cuda")
    with pytest.raises(RuntimeError, match="UNSUPPORTED"):
        _run(moe, w, p, x)


def test_single_launch_zero_tokens(moe):
    """An empty batch launches nothing and returns an empty output."""
    w = W.Workload("fused0", 4, 256, 8, 2, 128, seed=3)
    p = W.make_weights(w, device="cuda")
    x = W.make_x(w, device="cuda")[:0]
    out = moe.moe_forward(x, p["w_router"], p["w_gate_up"], p["w_down"], 2, single_launch=True)
    torch.cuda.synchronize()
    assert out.shape == (0, 256)
