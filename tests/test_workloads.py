"""The seeded synthetic workloads: shapes, value laws and the skewed routing."""

import math

import numpy as np
import pytest
import torch

import oracle
from mixture_experts_layer_20_gb300 import workloads as W


def test_workload_table():
    t = W.WORKLOADS
    assert t[W.TINY].T == 64 and t[W.TINY].d == 256 and t[W.TINY].E == 8
    assert t[W.DECODE].rows == 512
    assert t[W.PREFILL].rows * 1.0 / t[W.PREFILL].E == 375.0
    assert t[W.DEEPSEEK].I_shared == 2048 and t[W.DEEPSEEK].E == 256
    assert t[W.SKEWED].zipf_bias


def test_generation_is_seeded_and_shaped():
    w = W.WORKLOADS[W.TINY]
    a = W.make_weights(w)
    b = W.make_weights(w)
    for k in ("w_router", "w_gate_up", "w_down"):
        assert torch.equal(a[k], b[k])
        assert a[k].dtype == torch.bfloat16
    assert a["w_gate_up"].shape == (8, 256, 256)
    assert a["w_down"].shape == (8, 256, 128)
    x = W.make_x(w)
    assert x.shape == (64, 256)
    assert torch.equal(x, W.make_x(w))
    # the law: std 1/sqrt(fan_in)
    assert abs(a["w_gate_up"].float().std().item() * math.sqrt(256) - 1) < 0.02
    assert abs(a["w_down"].float().std().item() * math.sqrt(128) - 1) < 0.02
    assert abs(x.float().std().item() - 1) < 0.03


def test_skewed_routing_top8_share():
    """The log-rank bias puts about half of all assignments on 8 experts."""
    w = W.WORKLOADS[W.SKEWED]
    x = W.make_x(w)
    wr, bias = W.make_router(w)
    ids, gates, logits = oracle.route(W.to_bits(x), W.to_bits(wr), w.top_k, bias.numpy())
    counts = np.bincount(ids.reshape(-1), minlength=w.E)
    share = np.sort(counts)[::-1][:8].sum() / (w.T * w.top_k)
    assert 0.45 <= share <= 0.55, share
    assert counts.max() <= w.T   # a token picks an expert at most once


def test_random_routing_valid():
    ids, gates = W.random_routing(100, 16, 4, seed=3)
    assert ids.shape == (100, 4)
    for row in ids.tolist():
        assert row == sorted(set(row)) and len(row) == 4
    assert torch.allclose(gates.sum(1), torch.ones(100), atol=1e-6)
