"""Work counters and row-count invariants against the pages' worked numbers."""

import json
import os

import numpy as np
import pytest

from mixture_experts_layer_20_gb300 import counters

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden",
                                     "pages_worked_numbers.json")))


def test_expert_size():
    g = GOLDEN["qwen3_expert_params"]
    assert counters.expert_params(g["d"], g["I"]) == g["value"]
    assert counters.expert_bytes(4096, 1536) == GOLDEN["qwen3_expert_bf16_mib"]["value"] * 2**20
    g = GOLDEN["qwen3_layer_all_experts_gib"]
    assert g["E"] * counters.expert_bytes(4096, 1536) == g["value"] * 2**30


def test_flops():
    g = GOLDEN["decode_64_tokens_top8_gflop"]
    f = counters.expert_flops(g["T"], g["top_k"], 4096, 1536)
    assert round(f / 1e9, 1) == g["value"]
    assert counters.expert_flops(1, 1, 4096, 1536) == GOLDEN["flops_per_assignment"]["value"]
    # F_e(m) = 2 m P_e
    assert counters.expert_flops(7, 1, 4096, 1536) == 2 * 7 * counters.expert_params(4096, 1536)


def test_expected_active_experts():
    g = GOLDEN["expected_active_experts"]
    u = counters.expected_active_experts(g["E"], g["K"], g["M"])
    assert round(u) == g["value_approx"]
    assert round(u * counters.expert_bytes(4096, 1536) / 2**30, 2) == g["ideal_read_gib_approx"]


def test_rows_per_expert_means():
    g = GOLDEN["prefill_rows_per_expert"]
    assert g["tokens"] * g["top_k"] / g["E"] == g["value"]
    g = GOLDEN["ep_rows_per_expert"]
    assert g["n"] * g["k"] / g["E"] == g["value"]
    g = GOLDEN["decode_64_tokens_uniform_rows_per_expert"]
    assert 64 * 8 / 128 == g["value"] and 64 * 8 / 8 == g["concentrated_rows"]


def test_padding_example():
    g = GOLDEN["grouped_gemm_padding"]
    assert sum(g["rows"]) == g["useful"]
    assert counters.padded_rows(g["rows"], g["tile"]) == g["padded_to_tile"]
    assert counters.padded_rows_to_max(g["rows"]) == g["padded_to_max"]
    assert counters.padded_rows(g["rows"], g["tile"]) / g["useful"] == g["ratio_tile"]


def test_touched_bytes():
    counts = [4, 0, 3, 0, 1]
    assert counters.touched_weight_bytes(counts, 64, 32) == 3 * 3 * 64 * 32 * 2
    b = counters.algorithmic_bytes(counts, T=2, d=64, E=5, I=32, I_shared=16)
    assert b == 3 * 3 * 64 * 32 * 2 + 5 * 64 * 2 + 2 * 2 * 64 * 2 + 3 * 64 * 16 * 2
