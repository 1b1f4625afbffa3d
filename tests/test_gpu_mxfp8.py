"""MXFP8 weights on the GPU against the oracle: quantisation codes and scales
bit for bit."""

import numpy as np
import pytest
import torch

import oracle
from mixture_experts_layer_20_gb300 import workloads as W

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
