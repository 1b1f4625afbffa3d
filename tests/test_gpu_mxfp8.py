"""MXFP8 weights on the GPU against the oracle: quantisation codes and scales
bit for bit, and the whole layer against the oracle's layer with the weights
it quantised and dequantised itself; with act_mxfp8 (W8A8) the tokens' codes
and scales bit for bit too, and the layer against the oracle's W8A8 layer."""

import numpy as np
import pytest
import torch

import oracle
from mixture_experts_layer_20_gb300 import workloads as W
from tests.gpu_util import assert_layer_close, compare_routing, f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    from mixture_experts_layer_20_gb300 import binding
    return binding


def _oracle_layout(codes, scales_blocks):
    """oracle scales [rows, K/32] -> the library's [K/128, rows, 4]."""
    rows, nb = scales_blocks.shape
    return codes, scales_blocks.reshape(rows, nb // 4, 4).transpose(1, 0, 2)


@pytest.mark.parametrize("shape", [(3, 256, 512), (1, 40, 128), (2, 96, 1536)])
def test_quantize_matches_oracle(moe, shape):
    g = torch.Generator(device="cuda").manual_seed(sum(shape))
    w = torch.randn(shape, generator=g, device="cuda")
    # magnitudes from 2^-40 to 2^20 across rows, an all-zero run and exact powers of two
    w = w * torch.exp2(torch.linspace(-40, 20, shape[1], device="cuda"))[None, :, None]
    w[0, 0, 32:64] = 0.0
    w[0, 1, :32] = 2.0 ** torch.arange(-16, 16, device="cuda", dtype=torch.float32)
    wb = w.to(torch.bfloat16)
    codes, scales = moe.moe_mxfp8_quantize(wb)
    torch.cuda.synchronize()
    K = shape[-1]
    ref_codes, ref_scales = oracle.mxfp8_quantize(
        oracle.bf16_bits_to_f64(W.to_bits(wb)).reshape(-1, K))
    ref_codes, ref_scales = _oracle_layout(ref_codes, ref_scales)
    assert np.array_equal(codes.cpu().numpy().reshape(-1, K), ref_codes)
    assert np.array_equal(scales.cpu().numpy(), ref_scales)


def _dequantised_bits(w):
    """The oracle's own MXFP8 round trip of a bf16 [E, rows, K] weight tensor,
    as bf16 bits (exact: codes times powers of two have four significant bits)."""
    K = w.shape[-1]
    codes, scales = oracle.mxfp8_quantize(oracle.bf16_bits_to_f64(W.to_bits(w)).reshape(-1, K))
    deq = oracle.mxfp8_dequantize(codes, scales).reshape(w.shape)
    bits = oracle.f64_to_bf16_bits(deq)
    assert np.array_equal(oracle.bf16_bits_to_f64(bits), deq)
    return bits


# Layers with at most 8 token rows per expert on average (and d, I multiples
# of 256) take the warp-level small-M kernels; the others the tcgen05 tile
# kernels.
FORWARD_CASES = [
    # T, d, E, k, I, I_shared, zipf
    (64, 512, 32, 8, 256, 0, False),     # 16 rows per expert: tile kernels, 16-row chunks
    (32, 512, 32, 8, 256, 0, False),     # small-M: 8 rows per expert, some in two passes
    (60, 768, 64, 8, 512, 128, True),    # small-M: bias (hot experts: several passes), shared expert
    (600, 512, 8, 4, 384, 0, False),     # ~300 rows per expert: three chunks, six slabs
    (200, 384, 16, 4, 128, 0, True),     # d = 384: the last down slab has one populated half
    (130, 768, 64, 8, 256, 128, True),   # bias and a (bf16) shared expert
    (1, 256, 8, 2, 128, 0, False),       # one token (I = 128: tile kernels)
    (1, 256, 8, 2, 256, 0, False),       # one token, small-M
]


@pytest.mark.parametrize("T,d,E,k,I,Is,zipf", FORWARD_CASES)
def test_forward_mxfp8(moe, T, d, E, k, I, Is, zipf):
    w = W.Workload("mx", T, d, E, k, I, I_shared=Is, zipf_bias=zipf, seed=T + d)
    p = W.make_weights(w, device="cuda")
    x = W.make_x(w, device="cuda")
    mx_gu = moe.moe_mxfp8_quantize(p["w_gate_up"])
    mx_d = moe.moe_mxfp8_quantize(p["w_down"])
    ws = moe.new_workspace(T, d, E, I, k, Is)
    out = moe.moe_forward_mxfp8(x, p["w_router"], mx_gu, mx_d, k, ws=ws,
                                router_bias=p["router_bias"],
                                w_gate_up_shared=p["w_gate_up_shared"],
                                w_down_shared=p["w_down_shared"])
    assert moe.moe_get_device_status(ws) == moe.MOE_OK
    v = moe.workspace_views(ws, T, d, E, I, k, Is)
    ref = oracle.forward(
        W.to_bits(x), W.to_bits(p["w_router"]), _dequantised_bits(p["w_gate_up"]),
        _dequantised_bits(p["w_down"]), k,
        router_bias=None if p["router_bias"] is None else p["router_bias"].cpu().numpy(),
        w_gate_up_shared=None if p["w_gate_up_shared"] is None else W.to_bits(p["w_gate_up_shared"]),
        w_down_shared=None if p["w_down_shared"] is None else W.to_bits(p["w_down_shared"]))
    differ = compare_routing(v["topk_ids"].cpu().numpy(), v["topk_gates"].cpu().numpy(),
                             ref["ids"], ref["gates"], ref["logits"], k)
    assert differ.size == 0
    assert_layer_close(f64(v["y"]), ref["y"], "y")
    assert_layer_close(f64(out), ref["out"], "out")


@pytest.mark.parametrize("T", [96, 32])  # tile kernels (24 rows per expert); small-M (8)
def test_forward_mxfp8_extreme_codes(moe, T):
    """Subnormal E4M3 codes (tiny weights inside a block) and scales above
    2^7 (the converter's general path) still match the oracle."""
    d, E, k, I = 512, 8, 2, 256
    w = W.Workload("mx_extreme", T, d, E, k, I, seed=77)
    p = W.make_weights(w, device="cuda")
    x = W.make_x(w, device="cuda")
    wgu = p["w_gate_up"].clone()
    wgu[1, :, 0::32] *= 2.0 ** -14          # one value per run far below the run maximum
    wgu[2, I:] *= 2.0 ** -20                # expert 2's up rows: h, and so y, scaled back
    wd = p["w_down"].clone()
    wd[2] *= 2.0 ** 20                      # run maxima near 2^19: scale bytes above 134
    mx_gu = moe.moe_mxfp8_quantize(wgu)
    mx_d = moe.moe_mxfp8_quantize(wd)
    assert int(mx_d[1].max()) > 134
    assert bool(((mx_gu[0][1] & 0x78) == 0).any())   # exponent field 0: subnormal codes
    out = moe.moe_forward_mxfp8(x, p["w_router"], mx_gu, mx_d, k)
    torch.cuda.synchronize()
    ref = oracle.forward(W.to_bits(x), W.to_bits(p["w_router"]), _dequantised_bits(wgu),
                         _dequantised_bits(wd), k)
    assert_layer_close(f64(out), ref["out"], "out")


def test_mxfp8_zero_tokens(moe):
    """An empty batch launches nothing and returns an empty output."""
    w = W.Workload("mxfp80", 4, 256, 8, 2, 256, seed=3)
    p = W.make_weights(w, device="cuda")
    x = W.make_x(w, device="cuda")[:0]
    out = moe.moe_forward_mxfp8(x, p["w_router"], moe.moe_mxfp8_quantize(p["w_gate_up"]),
                               moe.moe_mxfp8_quantize(p["w_down"]), 2)
    torch.cuda.synchronize()
    assert out.shape == (0, 256)


@pytest.mark.parametrize("T,d,E,k,I,Is", [(32, 512, 32, 8, 256, 0),     # small-M kernels
                                          (600, 512, 8, 4, 256, 128)])  # tile kernels, shared expert
def test_forward_mxfp8_fp32_y(moe, T, d, E, k, I, Is):
    """y kept in fp32 (moe_forward_ext_t.y_fp32) with MXFP8 weights."""
    w = W.Workload("mxfp832", T, d, E, k, I, I_shared=Is, seed=T + 3)
    p = W.make_weights(w, device="cuda")
    x = W.make_x(w, device="cuda")
    q_gu = moe.moe_mxfp8_quantize(p["w_gate_up"])
    q_d = moe.moe_mxfp8_quantize(p["w_down"])
    ws = moe.new_workspace(T, d, E, I, k, Is, y_fp32=True)
    out = moe.moe_forward_mxfp8(x, p["w_router"], q_gu, q_d, k, ws=ws, y_fp32=True,
                              w_gate_up_shared=p["w_gate_up_shared"],
                              w_down_shared=p["w_down_shared"])
    assert moe.moe_get_device_status(ws) == moe.MOE_OK
    v = moe.workspace_views(ws, T, d, E, I, k, Is, y_fp32=True)
    ref = oracle.forward(
        W.to_bits(x), W.to_bits(p["w_router"]), _dequantised_bits(p["w_gate_up"]), _dequantised_bits(p["w_down"]), k,
        w_gate_up_shared=None if p["w_gate_up_shared"] is None else W.to_bits(p["w_gate_up_shared"]),
        w_down_shared=None if p["w_down_shared"] is None else W.to_bits(p["w_down_shared"]))
    differ = compare_routing(v["topk_ids"].cpu().numpy(), v["topk_gates"].cpu().numpy(),
                             ref["ids"], ref["gates"], ref["logits"], k)
    assert differ.size == 0
    assert_layer_close(f64(v["y"]), ref["y"], "y")
    assert_layer_close(f64(out), ref["out"], "out")


# ---------------------------------------------------------------- W8A8 (act_mxfp8)

def _unpermute_act(codes):
    """Token codes [rows, K] in the GEMMs' order (byte 64 t + 8 r + j of a
    256-wide chunk holds value 32 r + 4 t + (j & 3) + 16 (j >> 2)) -> value order."""
    rows, K = codes.shape
    # [.., t, r, jh, jl] -> values [.., r, jh, t, jl]
    return codes.reshape(rows, K // 256, 4, 8, 2, 4).transpose(0, 1, 3, 4, 2, 5).reshape(rows, K)


def _forward_a8(moe, T, d, E, k, I, zipf, seed):
    w = W.Workload("mxa8", T, d, E, k, I, zipf_bias=zipf, seed=seed)
    p = W.make_weights(w, device="cuda")
    x = W.make_x(w, device="cuda")
    ws = moe.new_workspace(T, d, E, I, k, act_mxfp8=True)
    out = moe.moe_forward_mxfp8(x, p["w_router"], moe.moe_mxfp8_quantize(p["w_gate_up"]),
                                moe.moe_mxfp8_quantize(p["w_down"]), k, ws=ws,
                                router_bias=p["router_bias"], act_mxfp8=True)
    assert moe.moe_get_device_status(ws) == moe.MOE_OK
    return w, p, x, out, moe.workspace_views(ws, T, d, E, I, k, act_mxfp8=True)


A8_CASES = [
    # T, d, E, k, I, zipf: at most 8 rows per expert on average (the small-M kernels)
    (32, 512, 32, 8, 256, False),
    (60, 768, 64, 8, 512, True),      # biased router: hot experts take several passes of 8
    (17, 1024, 16, 4, 512, False),
    (1, 256, 8, 2, 256, False),
]


@pytest.mark.parametrize("T,d,E,k,I,zipf", A8_CASES)
def test_forward_mxfp8_act(moe, T, d, E, k, I, zipf):
    """W8A8: the tokens x and h quantised bit for bit like the oracle, and the
    layer against the oracle's layer with MXFP8 weights and tokens."""
    w, p, x, out, v = _forward_a8(moe, T, d, E, k, I, zipf, seed=T + 5 * d)
    xc, xs = oracle.mxfp8_quantize(oracle.bf16_bits_to_f64(W.to_bits(x)))
    assert np.array_equal(_unpermute_act(v["act_x"].cpu().numpy()), xc)
    assert np.array_equal(v["act_x_scales"].cpu().numpy(), xs)
    hc, hs = oracle.mxfp8_quantize(oracle.bf16_bits_to_f64(W.to_bits(v["h"])))
    assert np.array_equal(_unpermute_act(v["act_h"].cpu().numpy()), hc)
    assert np.array_equal(v["act_h_scales"].cpu().numpy(), hs)
    ref = oracle.forward(
        W.to_bits(x), W.to_bits(p["w_router"]), _dequantised_bits(p["w_gate_up"]),
        _dequantised_bits(p["w_down"]), k,
        router_bias=None if p["router_bias"] is None else p["router_bias"].cpu().numpy(),
        act_mxfp8=True)
    differ = compare_routing(v["topk_ids"].cpu().numpy(), v["topk_gates"].cpu().numpy(),
                             ref["ids"], ref["gates"], ref["logits"], k)
    assert differ.size == 0
    assert_layer_close(f64(v["y"]), ref["y"], "y")
    assert_layer_close(f64(out), ref["out"], "out")


def test_forward_mxfp8_act_unsupported(moe):
    """W8A8 outside decode sizes, or with a shared expert, is refused on the
    host before anything runs."""
    w = W.Workload("mxa8u", 64, 512, 8, 4, 256, I_shared=128, seed=9)   # 32 rows per expert
    p = W.make_weights(w, device="cuda")
    x = W.make_x(w, device="cuda")
    q_gu = moe.moe_mxfp8_quantize(p["w_gate_up"])
    q_d = moe.moe_mxfp8_quantize(p["w_down"])
    with pytest.raises(RuntimeError, match="act_mxfp8"):
        moe.moe_forward_mxfp8(x, p["w_router"], q_gu, q_d, 4, act_mxfp8=True)
    with pytest.raises(RuntimeError, match="act_mxfp8"):
        moe.moe_forward_mxfp8(x[:8], p["w_router"], q_gu, q_d, 4, act_mxfp8=True,
                              w_gate_up_shared=p["w_gate_up_shared"],
                              w_down_shared=p["w_down_shared"])


def test_forward_mxfp8_act_extreme_scales(moe):
    """Tokens scaled by 2^-70 (scale bytes below 64, h underflowing to bf16
    subnormals and zeros) still match the oracle's W8A8 layer; the other
    tokens share experts with them."""
    T, d, E, k, I = 32, 512, 16, 4, 256
    w = W.Workload("mxa8x", T, d, E, k, I, seed=123)
    p = W.make_weights(w, device="cuda")
    x = W.make_x(w, device="cuda")
    x[::3] = (x[::3].float() * 2.0 ** -70).to(torch.bfloat16)
    ws = moe.new_workspace(T, d, E, I, k, act_mxfp8=True)
    out = moe.moe_forward_mxfp8(x, p["w_router"], moe.moe_mxfp8_quantize(p["w_gate_up"]),
                                moe.moe_mxfp8_quantize(p["w_down"]), k, ws=ws, act_mxfp8=True)
    assert moe.moe_get_device_status(ws) == moe.MOE_OK
    v = moe.workspace_views(ws, T, d, E, I, k, act_mxfp8=True)
    assert int(v["act_x_scales"].min()) < 64
    xc, xs = oracle.mxfp8_quantize(oracle.bf16_bits_to_f64(W.to_bits(x)))
    assert np.array_equal(_unpermute_act(v["act_x"].cpu().numpy()), xc)
    assert np.array_equal(v["act_x_scales"].cpu().numpy(), xs)
    ref = oracle.forward(W.to_bits(x), W.to_bits(p["w_router"]), _dequantised_bits(p["w_gate_up"]),
                         _dequantised_bits(p["w_down"]), k, act_mxfp8=True)
    differ = compare_routing(v["topk_ids"].cpu().numpy(), v["topk_gates"].cpu().numpy(),
                             ref["ids"], ref["gates"], ref["logits"], k)
    keep = np.setdiff1d(np.arange(T), differ)
    assert_layer_close(f64(out)[keep], ref["out"][keep], "out")


def test_forward_mxfp8_act_fp32_y(moe):
    """W8A8 with y kept in fp32 (y_fp32): the fp32 expert outputs and the layer
    against the oracle's W8A8 layer, and out equal to the fp16-y run's within
    the layer tolerance (only y's storage differs)."""
    T, d, E, k, I = 32, 512, 32, 8, 256
    w = W.Workload("mxa8y", T, d, E, k, I, seed=77)
    p = W.make_weights(w, device="cuda")
    x = W.make_x(w, device="cuda")
    q_gu = moe.moe_mxfp8_quantize(p["w_gate_up"])
    q_d = moe.moe_mxfp8_quantize(p["w_down"])
    ws = moe.new_workspace(T, d, E, I, k, y_fp32=True, act_mxfp8=True)
    out = moe.moe_forward_mxfp8(x, p["w_router"], q_gu, q_d, k, ws=ws, y_fp32=True,
                                act_mxfp8=True)
    assert moe.moe_get_device_status(ws) == moe.MOE_OK
    v = moe.workspace_views(ws, T, d, E, I, k, y_fp32=True, act_mxfp8=True)
    assert v["y"].dtype == torch.float32
    ref = oracle.forward(W.to_bits(x), W.to_bits(p["w_router"]), _dequantised_bits(p["w_gate_up"]),
                         _dequantised_bits(p["w_down"]), k, act_mxfp8=True)
    differ = compare_routing(v["topk_ids"].cpu().numpy(), v["topk_gates"].cpu().numpy(),
                             ref["ids"], ref["gates"], ref["logits"], k)
    assert differ.size == 0
    assert_layer_close(f64(v["y"]), ref["y"], "y")
    assert_layer_close(f64(out), ref["out"], "out")
    out16 = moe.moe_forward_mxfp8(x, p["w_router"], q_gu, q_d, k, act_mxfp8=True)
    assert_layer_close(f64(out16), f64(out), "fp16 y against fp32 y")
