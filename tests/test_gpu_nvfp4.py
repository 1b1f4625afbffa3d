"""NVFP4 expert weights: the GPU quantisation against the oracle's (bit for
bit: codes, block scales and tensor scales), and the whole layer with NVFP4
weights against the oracle run on the same dequantised weights."""

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


def _oracle_quantize(w):
    """The oracle's NVFP4 of a bf16 [G, rows, K] tensor in the library's layout:
    packed codes [G*rows, K/2], scales [K/256, G*rows, 16], tensor scales [G]."""
    G, rows, K = w.shape
    vals = oracle.bf16_bits_to_f64(W.to_bits(w)).astype(np.float32)
    codes, scales, tsc = [], [], []
    for g in range(G):
        c, s, t = oracle.nvfp4_quantize(vals[g])
        codes.append((c[:, 0::2] | (c[:, 1::2] << 4)).astype(np.uint8))
        scales.append(s)
        tsc.append(t)
    codes = np.concatenate(codes)
    scales = np.concatenate(scales).reshape(G * rows, K // 256, 16).transpose(1, 0, 2)
    return codes, scales, np.array(tsc, dtype=np.float32)


def _dequantised(w):
    """The oracle's NVFP4 round trip of a bf16 [E, rows, K] weight tensor, one
    matrix per expert, as exact fp64 values."""
    vals = oracle.bf16_bits_to_f64(W.to_bits(w)).astype(np.float32)
    out = np.empty(vals.shape, dtype=np.float64)
    for e in range(vals.shape[0]):
        out[e] = oracle.nvfp4_dequantize(*oracle.nvfp4_quantize(vals[e]))
    return out


@pytest.mark.parametrize("shape", [(2, 64, 512), (1, 48, 256), (3, 96, 1536)])
def test_quantize_matches_oracle(moe, shape):
    g = torch.Generator(device="cuda").manual_seed(sum(shape) + 1)
    w = torch.randn(shape, generator=g, device="cuda")
    # magnitudes from 2^-30 to 2^10 across rows, an all-zero block, tiny blocks far
    # below the matrix maximum (their scales underflow E4M3), exact powers of two
    w = w * torch.exp2(torch.linspace(-30, 10, shape[1], device="cuda"))[None, :, None]
    w[0, 0, 16:32] = 0.0
    w[0, -1, :16] = 2.0 ** torch.arange(-8, 8, device="cuda", dtype=torch.float32)
    wb = w.to(torch.bfloat16)
    codes, scales, tsc = moe.moe_nvfp4_quantize(wb)
    torch.cuda.synchronize()
    rc, rs, rt = _oracle_quantize(wb)
    assert np.array_equal(codes.cpu().numpy(), rc)
    assert np.array_equal(scales.cpu().numpy(), rs)
    assert np.array_equal(tsc.cpu().numpy().view(np.uint32), rt.view(np.uint32))


def test_quantize_all_zero_matrix(moe):
    wb = torch.zeros((2, 32, 256), dtype=torch.bfloat16, device="cuda")
    wb[1, 3, 5] = 1.5
    codes, scales, tsc = moe.moe_nvfp4_quantize(wb)
    rc, rs, rt = _oracle_quantize(wb)
    assert tsc[0].item() == 1.0
    assert np.array_equal(codes.cpu().numpy(), rc) and np.array_equal(scales.cpu().numpy(), rs)
    assert np.array_equal(tsc.cpu().numpy(), rt)


# Layers with at most 8 token rows per expert on average take the warp-level
# small-M kernels; the others the tcgen05 tile kernels.
FORWARD_CASES = [
    # T, d, E, k, I, I_shared, zipf
    (64, 512, 32, 8, 256, 0, False),     # 16 rows per expert: tile kernels, 16-row chunks
    (32, 512, 32, 8, 256, 0, False),     # small-M: 8 rows per expert, some in two passes
    (32, 1024, 32, 8, 512, 256, True),   # small-M: bias (hot experts: several passes), shared expert
    (600, 512, 8, 4, 512, 0, False),     # ~300 rows per expert: three chunks
    (200, 768, 16, 4, 256, 0, True),     # d = 768: three 128-row down slabs
    (130, 1024, 32, 8, 256, 256, True),  # bias and a (bf16) shared expert
    (1, 256, 8, 2, 256, 0, False),       # one token
]


@pytest.mark.parametrize("T,d,E,k,I,Is,zipf", FORWARD_CASES)
def test_forward_nvfp4(moe, T, d, E, k, I, Is, zipf):
    w = W.Workload("nv", T, d, E, k, I, I_shared=Is, zipf_bias=zipf, seed=T + d + 1)
    p = W.make_weights(w, device="cuda")
    x = W.make_x(w, device="cuda")
    nv_gu = moe.moe_nvfp4_quantize(p["w_gate_up"])
    nv_d = moe.moe_nvfp4_quantize(p["w_down"])
    ws = moe.new_workspace(T, d, E, I, k, Is)
    out = moe.moe_forward_nvfp4(x, p["w_router"], nv_gu, nv_d, k, ws=ws,
                                router_bias=p["router_bias"],
                                w_gate_up_shared=p["w_gate_up_shared"],
                                w_down_shared=p["w_down_shared"])
    assert moe.moe_get_device_status(ws) == moe.MOE_OK
    v = moe.workspace_views(ws, T, d, E, I, k, Is)
    ref = oracle.forward(
        W.to_bits(x), W.to_bits(p["w_router"]), _dequantised(p["w_gate_up"]),
        _dequantised(p["w_down"]), k,
        router_bias=None if p["router_bias"] is None else p["router_bias"].cpu().numpy(),
        w_gate_up_shared=None if p["w_gate_up_shared"] is None else W.to_bits(p["w_gate_up_shared"]),
        w_down_shared=None if p["w_down_shared"] is None else W.to_bits(p["w_down_shared"]))
    differ = compare_routing(v["topk_ids"].cpu().numpy(), v["topk_gates"].cpu().numpy(),
                             ref["ids"], ref["gates"], ref["logits"], k)
    assert differ.size == 0
    assert_layer_close(f64(v["y"]), ref["y"], "y")
    assert_layer_close(f64(out), ref["out"], "out")


def test_nvfp4_rejects_unaligned_dims(moe):
    w = W.Workload("nv_bad", 16, 384, 4, 2, 256, seed=3)   # d = 384 is not a multiple of 256
    p = W.make_weights(w, device="cuda")
    x = W.make_x(w, device="cuda")
    nv_d = moe.moe_nvfp4_quantize(torch.zeros((4, 384, 256), dtype=torch.bfloat16, device="cuda"))
    fake_gu = (torch.zeros((8 * 256, 192), dtype=torch.uint8, device="cuda"),
               torch.zeros((1, 8 * 256, 16), dtype=torch.uint8, device="cuda"),
               torch.ones((4,), dtype=torch.float32, device="cuda"))
    with pytest.raises(RuntimeError, match="UNSUPPORTED"):
        moe.moe_forward_nvfp4(x, p["w_router"], fake_gu, nv_d, 2)


def test_forward_nvfp4_subnormal_block_scales(moe):
    """Small-M path with blocks whose E4M3 scale is subnormal: every 16-value
    block of the weights is multiplied by a power of ten down to 1e-6, so that
    the smallest blocks' scales (448 x block amax / tensor amax) fall below
    the E4M3 normal range 2^-6, and every code magnitude, 0.5 included, occurs."""
    T, d, E, k, I = 32, 512, 16, 4, 256
    w = W.Workload("nv_sub", T, d, E, k, I, seed=7)
    p = W.make_weights(w, device="cuda")
    x = W.make_x(w, device="cuda")
    g = torch.Generator().manual_seed(11)

    def spread(t):
        rows, K = t.shape[-2], t.shape[-1]
        f = 10.0 ** -torch.randint(0, 7, (t.shape[0], rows, K // 16, 1), generator=g)
        t32 = t.float().cpu().reshape(t.shape[0], rows, K // 16, 16) * f
        return t32.reshape(t.shape).to(torch.bfloat16).to(t.device)

    wgu, wd = spread(p["w_gate_up"]), spread(p["w_down"])
    nv_gu, nv_d = moe.moe_nvfp4_quantize(wgu), moe.moe_nvfp4_quantize(wd)
    sc = np.concatenate([nv_gu[1].cpu().numpy().ravel(), nv_d[1].cpu().numpy().ravel()])
    assert (((sc & 0x78) == 0) & ((sc & 0x07) != 0)).any()  # subnormal scales occur
    ws = moe.new_workspace(T, d, E, I, k, 0)
    out = moe.moe_forward_nvfp4(x, p["w_router"], nv_gu, nv_d, k, ws=ws)
    assert moe.moe_get_device_status(ws) == moe.MOE_OK
    v = moe.workspace_views(ws, T, d, E, I, k, 0)
    ref = oracle.forward(W.to_bits(x), W.to_bits(p["w_router"]), _dequantised(wgu),
                         _dequantised(wd), k)
    differ = compare_routing(v["topk_ids"].cpu().numpy(), v["topk_gates"].cpu().numpy(),
                             ref["ids"], ref["gates"], ref["logits"], k)
    assert differ.size == 0
    assert_layer_close(f64(v["y"]), ref["y"], "y")
    assert_layer_close(f64(out), ref["out"], "out")


def test_nvfp4_zero_tokens(moe):
    """An empty batch launches nothing and returns an empty output."""
    w = W.Workload("nvfp40", 4, 256, 8, 2, 256, seed=3)
    p = W.make_weights(w, device="cuda")
    x = W.make_x(w, device="cuda")[:0]
    out = moe.moe_forward_nvfp4(x, p["w_router"], moe.moe_nvfp4_quantize(p["w_gate_up"]),
                               moe.moe_nvfp4_quantize(p["w_down"]), 2)
    torch.cuda.synchronize()
    assert out.shape == (0, 256)


@pytest.mark.parametrize("T,d,E,k,I,Is", [(32, 512, 32, 8, 256, 0),     # small-M kernels
                                          (600, 512, 8, 4, 256, 128)])  # tile kernels, shared expert
def test_forward_nvfp4_fp32_y(moe, T, d, E, k, I, Is):
    """y kept in fp32 (moe_forward_ext_t.y_fp32) with NVFP4 weights."""
    w = W.Workload("nvfp432", T, d, E, k, I, I_shared=Is, seed=T + 3)
    p = W.make_weights(w, device="cuda")
    x = W.make_x(w, device="cuda")
    q_gu = moe.moe_nvfp4_quantize(p["w_gate_up"])
    q_d = moe.moe_nvfp4_quantize(p["w_down"])
    ws = moe.new_workspace(T, d, E, I, k, Is, y_fp32=True)
    out = moe.moe_forward_nvfp4(x, p["w_router"], q_gu, q_d, k, ws=ws, y_fp32=True,
                              w_gate_up_shared=p["w_gate_up_shared"],
                              w_down_shared=p["w_down_shared"])
    assert moe.moe_get_device_status(ws) == moe.MOE_OK
    v = moe.workspace_views(ws, T, d, E, I, k, Is, y_fp32=True)
    ref = oracle.forward(
        W.to_bits(x), W.to_bits(p["w_router"]), _dequantised(p["w_gate_up"]), _dequantised(p["w_down"]), k,
        w_gate_up_shared=None if p["w_gate_up_shared"] is None else W.to_bits(p["w_gate_up_shared"]),
        w_down_shared=None if p["w_down_shared"] is None else W.to_bits(p["w_down_shared"]))
    differ = compare_routing(v["topk_ids"].cpu().numpy(), v["topk_gates"].cpu().numpy(),
                             ref["ids"], ref["gates"], ref["logits"], k)
    assert differ.size == 0
    assert_layer_close(f64(v["y"]), ref["y"], "y")
    assert_layer_close(f64(out), ref["out"], "out")
