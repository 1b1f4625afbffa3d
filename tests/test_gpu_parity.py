"""CUDA path (through the C ABI) against the fp64 CPU oracle, step by step and
for the whole layer, at sizes the oracle finishes in seconds that span several
tiles with ragged tails, plus the method's edge cases."""

import numpy as np
import pytest
import torch

import oracle
from mixture_experts_layer_20_gb300 import workloads as W
from tests.gpu_util import (ExpertsOnHost, assert_layer_close, compare_routing, f64,
                            layer_error)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    from mixture_experts_layer_20_gb300 import binding
    return binding


def _layer(T, d, E, k, I, I_shared=0, zipf=False, seed=0):
    w = W.Workload("custom", T, d, E, k, I, I_shared=I_shared, zipf_bias=zipf, seed=seed)
    p = W.make_weights(w, device="cuda")
    x = W.make_x(w, device="cuda")
    return w, x, p


def _oracle_forward(x, p, k):
    return oracle.forward(
        W.to_bits(x), W.to_bits(p["w_router"]), ExpertsOnHost(p["w_gate_up"]),
        ExpertsOnHost(p["w_down"]), k,
        router_bias=None if p["router_bias"] is None else p["router_bias"].cpu().numpy(),
        w_gate_up_shared=None if p["w_gate_up_shared"] is None else W.to_bits(p["w_gate_up_shared"]),
        w_down_shared=None if p["w_down_shared"] is None else W.to_bits(p["w_down_shared"]))


# ------------------------------------------------------------------ route

ROUTE_CASES = [
    # T, d, E, k, bias
    (64, 256, 8, 2, False),      # the tiny layer
    (129, 512, 8, 8, False),     # k = E: full softmax; ragged second tile
    (300, 512, 20, 3, True),     # E not a multiple of 16, with bias
    (1, 256, 8, 1, False),       # one token, k = 1
    (513, 1024, 128, 8, False),  # Qwen3 expert count
    (200, 512, 256, 8, True),    # maximum expert count
    (2100, 1024, 128, 8, False), # 17 token tiles, one tile per K range
    # 16 token tiles or more with many experts: one logits pass per tile over all K ranges
    (2048, 640, 256, 8, True),   # expert chunks to fill the SMs; a 128-wide last K range
    (1921, 512, 256, 3, True),   # exactly 16 tiles
    (5000, 1024, 256, 8, False), # 40 tiles: three chunks of 96 experts, the last one partial
]


@pytest.mark.parametrize("T,d,E,k,bias", ROUTE_CASES)
def test_route(moe, T, d, E, k, bias):
    w, x, p = _layer(T, d, E, k, 64, zipf=bias, seed=T)
    ids, gates = moe.moe_route(x, p["w_router"], k, router_bias=p["router_bias"])
    torch.cuda.synchronize()
    ids_ref, gates_ref, logits = oracle.route(
        W.to_bits(x), W.to_bits(p["w_router"]), k,
        None if p["router_bias"] is None else p["router_bias"].cpu().numpy())
    compare_routing(ids.cpu().numpy(), gates.cpu().numpy(), ids_ref, gates_ref, logits, k)
    assert torch.allclose(gates.sum(1), torch.ones(T, device="cuda"), atol=1e-6)
    if k == 1:
        assert (gates == 1.0).all()


def test_route_does_not_depend_on_the_batch(moe):
    """A token's routing is the same in a large batch (logits in one pass per
    tile) and alone with a few others (one tile per K range): bit for bit."""
    w, x, p = _layer(2304, 1024, 256, 8, 64, zipf=True, seed=5)
    ids, gates = moe.moe_route(x, p["w_router"], 8, router_bias=p["router_bias"])
    ids_s, gates_s = moe.moe_route(x[:100].contiguous(), p["w_router"], 8,
                                   router_bias=p["router_bias"])
    torch.cuda.synchronize()
    assert torch.equal(ids[:100], ids_s) and torch.equal(gates[:100], gates_s)


def test_route_ties(moe):
    """Exactly tied logits: the lower expert index wins (duplicated router rows)."""
    T, d, E, k = 40, 256, 16, 2
    x = W.make_x(W.Workload("t", T, d, E, k, 64), device="cuda").abs()
    wr = torch.full((E, d), -0.01, dtype=torch.bfloat16, device="cuda")
    wr[3] = 0.02
    wr[9] = 0.01
    wr[12] = 0.01   # tied with 9 for second place
    ids, gates = moe.moe_route(x, wr, k)
    assert (ids.cpu() == torch.tensor([3, 9], dtype=torch.int32)).all()


@pytest.mark.parametrize("T,d,E,k", [(300, 512, 20, 3), (129, 1024, 128, 8), (40, 256, 256, 8)])
def test_route_bias_selection_only(moe, T, d, E, k):
    """The bias picks the experts; the gates come from the unbiased logits."""
    w, x, p = _layer(T, d, E, k, 64, zipf=True, seed=T + 1)
    bias = p["router_bias"]
    ids, gates = moe.moe_route(x, p["w_router"], k, router_bias=bias, bias_selection_only=True)
    torch.cuda.synchronize()
    ids_ref, gates_ref, logits = oracle.route(W.to_bits(x), W.to_bits(p["w_router"]), k,
                                              bias.cpu().numpy(), bias_for_selection_only=True)
    compare_routing(ids.cpu().numpy(), gates.cpu().numpy(), ids_ref, gates_ref, logits, k)
    # the same selection as the biased router, other gates
    ids_b, gates_b = moe.moe_route(x, p["w_router"], k, router_bias=bias)
    assert torch.equal(ids, ids_b)
    assert not torch.equal(gates, gates_b)


# ------------------------------------------------------------------ permute

PERMUTE_CASES = [
    (64, 8, 2), (1, 8, 8), (1500, 128, 8), (4096, 256, 8), (777, 16, 4), (5000, 64, 1),
    (512, 128, 8),    # 4096 assignments: the largest single-CTA grouping
    (9000, 200, 8),   # 72000 assignments: 18 chunks of the multi-CTA path
]


@pytest.mark.parametrize("T,E,k", PERMUTE_CASES)
def test_permute(moe, T, E, k):
    ids, _ = W.random_routing(T, E, k, seed=T + E)
    ids[: T // 3] = ids[0]                        # a hot set of experts, others thin or empty
    d = 128
    x = W.make_x(W.Workload("p", T, d, E, k, 64), device="cuda")
    counts, offsets, perm, slot_pos, x_perm = moe.moe_permute(ids.cuda(), E, x=x)
    torch.cuda.synchronize()
    c_ref, o_ref, p_ref, s_ref = oracle.permute(ids.numpy(), E)
    assert np.array_equal(counts.cpu().numpy(), c_ref)
    assert np.array_equal(offsets.cpu().numpy(), o_ref)
    assert np.array_equal(perm.cpu().numpy(), p_ref)
    assert np.array_equal(slot_pos.cpu().numpy(), s_ref)
    xb = W.to_bits(x)
    assert np.array_equal(W.to_bits(x_perm), xb[p_ref // k])


def test_permute_without_gather(moe):
    ids, _ = W.random_routing(300, 32, 4, seed=5)
    counts, offsets, perm, slot_pos, x_perm = moe.moe_permute(ids.cuda(), 32)
    assert x_perm is None
    _, o_ref, p_ref, _ = oracle.permute(ids.numpy(), 32)
    assert np.array_equal(perm.cpu().numpy(), p_ref)


# ------------------------------------------------------------------ expert FFN

FFN_CASES = [
    # rows per expert, d, I
    ([40, 0, 200, 1, 129, 0, 3, 128], 256, 128),
    ([300, 17, 0, 64], 512, 384),     # I not a multiple of 128: ragged N tile
    ([1], 256, 64),
    ([130, 250, 5, 0, 0, 0, 1, 90, 60, 33, 7, 256], 768, 192),
    # >= 256 rows per expert: several token chunks per expert (up to 256
    # tokens each, sharing the expert's 16-row units) mixed with small ones
    ([600, 257, 512, 513, 16, 1000, 0, 300], 256, 128),
    ([700, 300, 260], 512, 384),
    # d = 64: one pipeline stage per gate_up tile, 256 experts x 8 slabs = 2048
    # tiles (~27 per CTA pair), so the producer runs several tiles ahead of the
    # MMA issuer and the ring of tile sizes between them wraps
    ([8, 0, 24, 9] * 64, 64, 1024),
]


@pytest.mark.parametrize("counts,d,I", FFN_CASES)
def test_expert_ffn(moe, counts, d, I):
    E = len(counts)
    rows = sum(counts)
    w = W.Workload("f", rows, d, E, 1, I, seed=rows)
    p = W.make_weights(w, device="cuda")
    x_perm = W.make_x(w, device="cuda")
    offsets = torch.tensor(np.concatenate([[0], np.cumsum(counts)]), dtype=torch.int32, device="cuda")
    y = moe.moe_expert_ffn(x_perm, offsets, p["w_gate_up"], p["w_down"])
    torch.cuda.synchronize()
    y_ref = oracle.expert_ffn(f64(x_perm), offsets.cpu().numpy(), ExpertsOnHost(p["w_gate_up"]),
                              ExpertsOnHost(p["w_down"]))
    assert_layer_close(f64(y), y_ref, "expert_ffn y")


# ------------------------------------------------------------------ combine

@pytest.mark.parametrize("T,d,k,shared", [(64, 256, 2, False), (333, 1024, 8, True),
                                          (1, 7168, 8, True), (100, 64, 1, False)])
def test_combine(moe, T, d, k, shared):
    g = torch.Generator(device="cuda").manual_seed(T * 7 + k)
    rows = T * k
    y = torch.randn((rows, d), generator=g, device="cuda").half()
    slot_pos = torch.randperm(rows, generator=g, device="cuda").to(torch.int32).view(T, k)
    _, gates = W.random_routing(T, max(k, 8), k, seed=T)
    gates = gates.cuda()
    ys = torch.randn((T, d), generator=g, device="cuda").half() if shared else None
    out = moe.moe_combine(y, slot_pos, gates, y_shared=ys)
    torch.cuda.synchronize()
    ref = oracle.combine(f64(y), slot_pos.cpu().numpy(), f64(gates),
                         f64(ys) if shared else None)
    got = f64(out)
    # one bf16 rounding of an fp32 sum: within half a bf16 ulp plus fp32 noise
    assert (np.abs(got - ref) <= np.abs(ref) * 2.0**-8 + 1e-5).all()
    assert_layer_close(got, ref, "combine")


# ------------------------------------------------------------------ whole layer

FORWARD_CASES = [
    # T, d, E, k, I, I_shared, zipf
    (64, 256, 8, 2, 128, 0, False),       # the tiny layer
    (300, 512, 16, 4, 384, 0, True),      # several tiles, ragged tails, biased router
    (17, 256, 8, 2, 128, 0, False),
    (1, 512, 32, 8, 256, 0, False),
    (250, 1024, 64, 6, 256, 256, False),  # with an always-on shared expert
    (130, 768, 256, 8, 128, 128, False),  # 256 experts, most with zero or one row
    # more than 4096 rows and 128 per expert: grouping by count and scatter kernels,
    # x_perm written by the gather kernel
    (1500, 512, 16, 4, 384, 0, True),     # biased router: hot experts with many chunks
    (2100, 256, 8, 2, 128, 0, False),     # 4200 rows: a last 16-row unit of 8 rows
    (1100, 1024, 64, 8, 256, 256, False),  # with a shared expert
]


@pytest.mark.parametrize("T,d,E,k,I,Is,zipf", FORWARD_CASES)
def test_forward(moe, T, d, E, k, I, Is, zipf):
    w, x, p = _layer(T, d, E, k, I, I_shared=Is, zipf=zipf, seed=T + E)
    ws = moe.new_workspace(T, d, E, I, k, Is)
    out = moe.moe_forward(x, p["w_router"], p["w_gate_up"], p["w_down"], k, ws=ws,
                          router_bias=p["router_bias"], w_gate_up_shared=p["w_gate_up_shared"],
                          w_down_shared=p["w_down_shared"])
    assert moe.moe_get_device_status(ws) == moe.MOE_OK
    v = moe.workspace_views(ws, T, d, E, I, k, Is)
    ref = _oracle_forward(x, p, k)
    differ = compare_routing(v["topk_ids"].cpu().numpy(), v["topk_gates"].cpu().numpy(),
                             ref["ids"], ref["gates"], ref["logits"], k)
    assert differ.size == 0   # no near-ties expected at these sizes
    assert np.array_equal(v["expert_counts"].cpu().numpy(), ref["counts"])
    assert np.array_equal(v["expert_offsets"].cpu().numpy(), ref["offsets"])
    assert np.array_equal(v["perm"].cpu().numpy(), ref["perm"])
    assert np.array_equal(v["slot_pos"].cpu().numpy(), ref["slot_pos"])
    if T * k > 128 * E:  # x_perm written (fewer rows: gate_up gathers them from x itself)
        assert torch.equal(v["x_perm"], x[v["perm"].long() // k])
    assert_layer_close(f64(v["y"]), ref["y"], "y")
    assert_layer_close(f64(out), ref["out"], "out")


FP32_Y_CASES = [
    # T, d, E, k, I, I_shared, zipf
    (300, 512, 16, 4, 384, 0, True),      # tile GEMMs on x_perm
    (48, 256, 8, 2, 128, 128, False),     # decode-sized (rows gathered from x), shared expert
]


@pytest.mark.parametrize("T,d,E,k,I,Is,zipf", FP32_Y_CASES)
def test_forward_fp32_y(moe, T, d, E, k, I, Is, zipf):
    """y kept in fp32 (moe_forward_ext_t.y_fp32): the same routing, y and out
    within the layer tolerance of the oracle, and out close to the fp16-y
    layer's (the difference is fp16 rounding of y, relative to the largest
    output: a sum that nearly cancels may differ by more than its own ulp)."""
    w, x, p = _layer(T, d, E, k, I, I_shared=Is, zipf=zipf, seed=T + E + 1)
    kw = dict(router_bias=p["router_bias"], w_gate_up_shared=p["w_gate_up_shared"],
              w_down_shared=p["w_down_shared"])
    ws = moe.new_workspace(T, d, E, I, k, Is, y_fp32=True)
    assert ws.numel() > moe.moe_workspace_size(T, d, E, I, k, Is)
    out = moe.moe_forward(x, p["w_router"], p["w_gate_up"], p["w_down"], k, ws=ws, y_fp32=True,
                          **kw)
    assert moe.moe_get_device_status(ws) == moe.MOE_OK
    v = moe.workspace_views(ws, T, d, E, I, k, Is, y_fp32=True)
    assert v["y"].dtype == torch.float32
    ref = _oracle_forward(x, p, k)
    differ = compare_routing(v["topk_ids"].cpu().numpy(), v["topk_gates"].cpu().numpy(),
                             ref["ids"], ref["gates"], ref["logits"], k)
    assert differ.size == 0
    assert_layer_close(f64(v["y"]), ref["y"], "y")
    assert_layer_close(f64(out), ref["out"], "out")
    out16 = moe.moe_forward(x, p["w_router"], p["w_gate_up"], p["w_down"], k, **kw)
    torch.cuda.synchronize()
    a, b = f64(out), f64(out16)
    assert np.abs(a - b).max() <= np.abs(b).max() * 2.0**-6  # about one bf16 ulp at the top


def test_forward_fp32_y_needs_its_workspace(moe):
    w, x, p = _layer(64, 256, 8, 2, 128, seed=3)
    with pytest.raises(RuntimeError):
        moe.moe_forward(x, p["w_router"], p["w_gate_up"], p["w_down"], 2,
                        ws=moe.new_workspace(64, 256, 8, 128, 2), y_fp32=True)
    with pytest.raises(RuntimeError):
        moe.moe_forward(x, p["w_router"], p["w_gate_up"], p["w_down"], 2, y_fp32=True,
                        single_launch=True)


def test_forward_bias_selection_only(moe):
    T, d, E, k, I = 250, 512, 16, 4, 256
    w, x, p = _layer(T, d, E, k, I, zipf=True, seed=21)
    ws = moe.new_workspace(T, d, E, I, k)
    out = moe.moe_forward(x, p["w_router"], p["w_gate_up"], p["w_down"], k, ws=ws,
                          router_bias=p["router_bias"], bias_selection_only=True)
    assert moe.moe_get_device_status(ws) == moe.MOE_OK
    v = moe.workspace_views(ws, T, d, E, I, k)
    ref = oracle.forward(W.to_bits(x), W.to_bits(p["w_router"]), ExpertsOnHost(p["w_gate_up"]),
                         ExpertsOnHost(p["w_down"]), k, router_bias=p["router_bias"].cpu().numpy(),
                         bias_for_selection_only=True)
    differ = compare_routing(v["topk_ids"].cpu().numpy(), v["topk_gates"].cpu().numpy(),
                             ref["ids"], ref["gates"], ref["logits"], k)
    assert differ.size == 0
    assert_layer_close(f64(out), ref["out"], "out")


def test_single_expert_is_dense_ffn(moe):
    """k = 1 and a dominant bias: every token goes to one expert with gate 1."""
    T, d, E, k, I = 200, 512, 8, 1, 256
    w, x, p = _layer(T, d, E, k, I, seed=3)
    bias = torch.zeros(E, device="cuda")
    bias[5] = 1e4
    out = moe.moe_forward(x, p["w_router"], p["w_gate_up"], p["w_down"], k, router_bias=bias)
    torch.cuda.synchronize()
    ref = oracle.swiglu_ffn(f64(x), W.to_bits(p["w_gate_up"][5]), W.to_bits(p["w_down"][5]))
    assert_layer_close(f64(out), ref, "dense")


def test_deterministic_and_row_independent(moe):
    T, d, E, k, I = 600, 512, 32, 4, 256
    w, x, p = _layer(T, d, E, k, I, seed=11)
    a = moe.moe_forward(x, p["w_router"], p["w_gate_up"], p["w_down"], k)
    b = moe.moe_forward(x, p["w_router"], p["w_gate_up"], p["w_down"], k)
    assert torch.equal(a, b)
    part = moe.moe_forward(x[:37].contiguous(), p["w_router"], p["w_gate_up"], p["w_down"], k)
    assert torch.equal(part, a[:37])
    # doubling W_down doubles every output exactly
    c = moe.moe_forward(x, p["w_router"], p["w_gate_up"], (p["w_down"] * 2).contiguous(), k)
    assert torch.equal(c, a * 2)


def test_zero_tokens(moe):
    w, x, p = _layer(4, 256, 8, 2, 128)
    out = moe.moe_forward(x[:0], p["w_router"], p["w_gate_up"], p["w_down"], 2)
    assert out.shape == (0, 256)
