"""Shared helpers of the GPU parity tests: tolerances and comparisons.

The bar for floating-point outputs of the layer (and of the expert FFN's y):
    max|gpu - oracle| <= 1e-2 * max|oracle|
    sum|gpu - oracle| / sum|oracle| <= 2e-3      (mean relative error)
Routing ids, counts, offsets and the permutation are compared bit for bit,
except tokens whose fp64 logit margin between the k-th and (k+1)-th expert is
below 1e-4: those may route differently in fp32 and are listed, not failed.
"""

from __future__ import annotations

import numpy as np
import torch

import oracle
from mixture_experts_layer_20_gb300 import workloads as W

MAX_REL = 1e-2
MEAN_REL = 2e-3
NEAR_TIE = 1e-4
GATE_ATOL = 1e-5


def f64(t: torch.Tensor) -> np.ndarray:
    """Exact fp64 values of a bf16 or fp32 device tensor."""
    if t.dtype == torch.bfloat16:
        return oracle.bf16_bits_to_f64(W.to_bits(t))
    return t.detach().cpu().to(torch.float64).numpy()


def layer_error(gpu: np.ndarray, ref: np.ndarray):
    err = np.abs(gpu - ref)
    return float(err.max() / np.abs(ref).max()), float(err.sum() / np.abs(ref).sum())


def assert_layer_close(gpu: np.ndarray, ref: np.ndarray, what: str):
    max_rel, mean_rel = layer_error(gpu, ref)
    assert max_rel <= MAX_REL and mean_rel <= MEAN_REL, \
        f"{what}: max_rel={max_rel:.3e} mean_rel={mean_rel:.3e}"
    return max_rel, mean_rel


def boundary_margin(logits: np.ndarray, k: int) -> np.ndarray:
    """fp64 gap between the k-th and (k+1)-th largest logit of each token."""
    if k >= logits.shape[1]:
        return np.full(logits.shape[0], np.inf)
    s = -np.sort(-logits, axis=1)
    return s[:, k - 1] - s[:, k]


def compare_routing(ids_gpu, gates_gpu, ids_ref, gates_ref, logits, k):
    """Bit-exact ids except near-ties; gates within GATE_ATOL where ids agree.
    Returns the indices of tokens that routed differently (all near-ties)."""
    ids_gpu = np.asarray(ids_gpu)
    differ = ~(ids_gpu == ids_ref).all(axis=1)
    near = boundary_margin(logits, k) < NEAR_TIE
    bad = np.nonzero(differ & ~near)[0]
    assert bad.size == 0, f"routing differs on tokens {bad[:10]} with margins >= {NEAR_TIE}"
    same = ~differ
    if same.any():
        gerr = np.abs(np.asarray(gates_gpu, np.float64)[same] - gates_ref[same]).max()
        assert gerr <= GATE_ATOL, f"gate error {gerr:.3e}"
    return np.nonzero(differ)[0]


class ExpertsOnHost:
    """Lazy per-expert host copies of a [E, ...] bf16 device weight tensor."""

    def __init__(self, t: torch.Tensor):
        self.t = t
        self.cache = {}

    def __getitem__(self, e):
        e = int(e)
        if e not in self.cache:
            self.cache[e] = W.to_bits(self.t[e])
        return self.cache[e]


class ExpertsStreamed:
    """Per-expert host copies of a [E, ...] bf16 device weight tensor, made on
    each access and not kept (a whole-layer oracle pass reads each expert
    once; keeping them would hold every expert's weights in host memory)."""

    def __init__(self, t: torch.Tensor):
        self.t = t

    def __getitem__(self, e):
        return W.to_bits(self.t[int(e)])
