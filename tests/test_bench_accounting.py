"""bench.py's per-launch work accounting (the roofline's numerators): FLOPs
and algorithmic bytes of each kernel, each operand and result counted once,
weights only for experts that received rows, y in fp16."""

import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from mixture_experts_layer_20_gb300 import counters  # noqa: E402
from mixture_experts_layer_20_gb300 import workloads as W  # noqa: E402


def test_expert_gemms_and_combine():
    w = W.WORKLOADS["qwen3_235b_prefill_T6000"]
    T, d, E, k, I = w.T, w.d, w.E, w.top_k, w.I
    rows = T * k
    counts = [rows // E] * E
    fl_gu, by = bench.kernel_work("moe_gate_up_swiglu", w, counts)
    assert fl_gu == 4 * rows * d * I
    assert by == E * 2 * I * d * 2 + rows * d * 2 + rows * I * 2
    fl_dn, by = bench.kernel_work("moe_down", w, counts)
    assert fl_dn == 2 * rows * d * I
    assert by == E * d * I * 2 + rows * I * 2 + rows * d * 2          # y: fp16
    assert fl_gu + fl_dn == counters.expert_flops(T, k, d, I)         # 6 d I per assignment
    _, by = bench.kernel_work("moe_combine", w, counts)
    assert by == rows * d * 2 + T * d * 2 + rows * 8                   # y fp16, out bf16, ids+gates
    _, by = bench.kernel_work("moe_permute_gather", w, counts)
    assert by == rows * d * 2 + T * d * 2 + rows * 4


def test_untouched_experts_are_not_counted():
    w = W.WORKLOADS["qwen3_235b_decode_T64"]
    d, I, rows = w.d, w.I, w.T * w.top_k
    counts = [0] * 64 + [rows // 64] * 64
    _, by = bench.kernel_work("moe_down", w, counts)
    assert by == 64 * d * I * 2 + rows * I * 2 + rows * d * 2
    _, by_mx = bench.kernel_work("moe_down_mxfp8", w, counts)
    assert by_mx == int(64 * d * I * bench.MX_BYTES) + rows * I * 2 + rows * d * 2
    _, by_nv = bench.kernel_work("moe_down_nvfp4", w, counts)
    assert by_nv == int(64 * d * I * bench.NV_BYTES) + rows * I * 2 + rows * d * 2


def test_small_m_and_single_launch_accounting():
    """The small-M kernels do the tile kernels' work; the single-launch layer
    counts the whole layer: every expert FLOP, the router and the combine,
    and the layer's algorithmic bytes."""
    w = W.WORKLOADS["qwen3_235b_decode_T64"]
    T, d, E, k, I = w.T, w.d, w.E, w.top_k, w.I
    counts = [T * k // 64] * 64 + [0] * 64
    for fmt in ("mxfp8", "nvfp4"):
        for kind in ("gate_up_swiglu", "down"):
            assert bench.kernel_work(f"moe_{kind}_{fmt}_smallm", w, counts) == \
                bench.kernel_work(f"moe_{kind}_{fmt}", w, counts)
    fl, by = bench.kernel_work("moe_decode_fused", w, counts)
    assert fl == counters.expert_flops(T, k, d, I) + counters.router_flops(T, d, E) + 2 * T * k * d
    assert by == counters.algorithmic_bytes(counts, T, d, E, I)
