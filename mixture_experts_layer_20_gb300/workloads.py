"""Seeded synthetic inputs for the MoE FFN layer.

This module only draws random numbers: it holds none of the layer's
arithmetic, so both the CUDA path and the CPU oracle can consume what it makes.

Value recipe (the same for every workload):
  x          ~ N(0, 1)                 -> bf16 (round to nearest even)
  W_router   ~ N(0, std 1/sqrt(d))     -> bf16, shape [E, d]
  W_gate_up  ~ N(0, std 1/sqrt(d))     -> bf16, shape [E, 2I, d]; rows [0,I) gate, [I,2I) up
  W_down     ~ N(0, std 1/sqrt(I))     -> bf16, shape [E, d, I]
  shared expert (if any): same laws, shapes [2I_s, d] and [d, I_s]
  router bias (skewed workload only): b_e = -beta * ln(r_e), r a seeded random
      permutation of the ranks 1..E, beta = ZIPF_BETA (fp32)

Each tensor has its own generator stream, seeded from (seed, tensor id), so a
tensor's values do not depend on which other tensors were drawn.  Large weight
tensors are drawn one expert at a time to bound temporary memory.
"""

from __future__ import annotations

import dataclasses
import math

import torch

# Log-rank ("Zipf-shaped") router bias strength for the skewed workload.  With
# unit-variance logits this puts about half of all T*k assignments on the 8
# most popular experts; the realised share is checked by a test.
ZIPF_BETA = 0.8

_TENSOR_IDS = {"x": 1, "w_router": 2, "w_gate_up": 3, "w_down": 4,
               "router_bias": 5, "w_gate_up_shared": 6, "w_down_shared": 7}


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    T: int          # tokens
    d: int          # hidden size
    E: int          # routed experts
    top_k: int      # experts per token
    I: int          # expert intermediate size
    I_shared: int = 0       # always-on shared expert's intermediate size (0 = none)
    zipf_bias: bool = False  # per-expert router bias with a log-rank law
    seed: int = 0

    @property
    def rows(self) -> int:
        return self.T * self.top_k

    def with_tokens(self, T: int) -> "Workload":
        return dataclasses.replace(self, T=T)


WORKLOADS = {
    w.name: w for w in [
        # tiny layer for full parity
        Workload("tiny_T64_d256_E8_k2_I128", 64, 256, 8, 2, 128),
        # Qwen3-235B-A22B MoE layer, decode batch of 64 tokens (weight-streaming)
        Workload("qwen3_235b_decode_T64", 64, 4096, 128, 8, 1536),
        # the same layer, ~6000-token prefill (375 rows per expert on average)
        Workload("qwen3_235b_prefill_T6000", 6000, 4096, 128, 8, 1536),
        # the same layer with a Zipf-shaped router bias (load-imbalanced)
        Workload("qwen3_235b_skewed_T4096", 4096, 4096, 128, 8, 1536, zipf_bias=True),
        # DeepSeek-V3-like layer: 256 routed experts + 1 shared expert
        Workload("deepseek_v3_like_T8192", 8192, 7168, 256, 8, 2048, I_shared=2048),
    ]
}

TINY = "tiny_T64_d256_E8_k2_I128"
DECODE = "qwen3_235b_decode_T64"
PREFILL = "qwen3_235b_prefill_T6000"
SKEWED = "qwen3_235b_skewed_T4096"
DEEPSEEK = "deepseek_v3_like_T8192"


def _generator(seed: int, tensor: str, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed * 1000 + _TENSOR_IDS[tensor])
    return g


def _normal_bf16(shape, std, gen, device, chunk_dim0=False):
    if not chunk_dim0:
        v = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
        return (v * std).to(torch.bfloat16)
    out = torch.empty(shape, device=device, dtype=torch.bfloat16)
    for i in range(shape[0]):
        v = torch.randn(shape[1:], generator=gen, device=device, dtype=torch.float32)
        out[i] = (v * std).to(torch.bfloat16)
    return out


def make_x(w: Workload, device="cpu") -> torch.Tensor:
    return _normal_bf16((w.T, w.d), 1.0, _generator(w.seed, "x", device), device)


def make_router(w: Workload, device="cpu"):
    """Router weights [E, d] (bf16) and the router bias [E] (fp32, or None)."""
    w_router = _normal_bf16((w.E, w.d), 1.0 / math.sqrt(w.d),
                            _generator(w.seed, "w_router", device), device)
    bias = None
    if w.zipf_bias:
        g = _generator(w.seed, "router_bias", device)
        ranks = torch.randperm(w.E, generator=g, device=device).to(torch.float64) + 1.0
        bias = (-ZIPF_BETA * torch.log(ranks)).to(torch.float32)
    return w_router, bias


def make_weights(w: Workload, device="cpu") -> dict:
    """Router, expert and shared-expert weights (+ router bias) of a workload."""
    d, E, I = w.d, w.E, w.I
    w_router, bias = make_router(w, device)
    p = {
        "w_router": w_router,
        "w_gate_up": _normal_bf16((E, 2 * I, d), 1.0 / math.sqrt(d),
                                  _generator(w.seed, "w_gate_up", device), device, True),
        "w_down": _normal_bf16((E, d, I), 1.0 / math.sqrt(I),
                               _generator(w.seed, "w_down", device), device, True),
        "router_bias": bias,
        "w_gate_up_shared": None,
        "w_down_shared": None,
    }
    if w.I_shared:
        Is = w.I_shared
        p["w_gate_up_shared"] = _normal_bf16((2 * Is, d), 1.0 / math.sqrt(d),
                                             _generator(w.seed, "w_gate_up_shared", device), device)
        p["w_down_shared"] = _normal_bf16((d, Is), 1.0 / math.sqrt(Is),
                                          _generator(w.seed, "w_down_shared", device), device)
    return p


def random_routing(T: int, E: int, top_k: int, seed: int = 0, device="cpu"):
    """A valid routing table: k distinct experts per token (ascending) + gates.

    Used to drive the grouping and combine steps on their own.  Gates are
    positive and sum to one per token.
    """
    g = torch.Generator(device="cpu")
    g.manual_seed(seed * 1000 + 11)
    scores = torch.rand((T, E), generator=g)
    ids = torch.topk(scores, top_k, dim=1).indices.sort(dim=1).values.to(torch.int32)
    raw = torch.rand((T, top_k), generator=g, dtype=torch.float64) + 0.05
    gates = (raw / raw.sum(dim=1, keepdim=True)).to(torch.float32)
    return ids.to(device), gates.to(device)


def to_bits(t: torch.Tensor):
    """Raw bf16 bit patterns of a bf16 tensor as a numpy uint16 array (host)."""
    import numpy as np
    assert t.dtype == torch.bfloat16
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
