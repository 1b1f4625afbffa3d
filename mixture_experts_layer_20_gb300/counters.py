"""Algorithmic work counters of the MoE FFN layer (FLOPs, bytes, padding).

These define the numerators of every throughput and roofline figure, so they
count only what the method needs, never what an implementation wastes:

* FLOPs: 2 per multiply-add.  An expert is three d x I matrices, P_e = 3 d I
  parameters, and m rows cost F_e(m) = 2 m P_e ('Chapter 9. Distributed
  inference', section 9.3.2), i.e. 6 d I per token-expert assignment (section
  9.4.1).  The router's 2 T d E is listed separately.
* Bytes: expert weights that the batch touches (an expert with zero rows is
  never read), the router weights, the input x and the output, all bf16.
  Intermediates (grouped x, h, y) are implementation traffic, not algorithmic.
* Padding: rows a grouped GEMM computes beyond the useful ones when every
  expert's rows are rounded up to the tile (section 9.4.3).
"""

from __future__ import annotations

import math


def expert_params(d: int, I: int) -> int:
    """P_e: parameters of one SwiGLU expert (gate, up and down: three d x I)."""
    return 3 * d * I


def expert_bytes(d: int, I: int, bytes_per_elem: int = 2) -> int:
    return expert_params(d, I) * bytes_per_elem


def expert_flops(T: int, top_k: int, d: int, I: int, I_shared: int = 0) -> int:
    """Matrix FLOPs of the experts: T*k assignments at 6 d I each (+ shared)."""
    return T * top_k * 6 * d * I + T * 6 * d * I_shared


def router_flops(T: int, d: int, E: int) -> int:
    return 2 * T * d * E


def expected_active_experts(E: int, K: int, M: int) -> float:
    """E[U] = E (1 - (1 - K/E)^M) for M tokens each picking K of E experts
    uniformly ('Chapter 9. Distributed inference', section 9.3.3)."""
    return E * (1.0 - (1.0 - K / E) ** M)


def touched_weight_bytes(counts, d: int, I: int) -> int:
    """Bytes of the expert weights that a batch with these row counts reads."""
    return sum(1 for c in counts if c > 0) * expert_bytes(d, I)


def algorithmic_bytes(counts, T: int, d: int, E: int, I: int, I_shared: int = 0) -> int:
    """Touched expert weights + router weights + x + out (+ shared expert)."""
    b = touched_weight_bytes(counts, d, I)
    b += E * d * 2          # router weights
    b += 2 * T * d * 2      # x in, out
    if I_shared:
        b += expert_bytes(d, I_shared)
    return b


def padded_rows(counts, tile: int) -> int:
    """Rows computed when every non-empty expert is padded up to the tile."""
    return sum(int(math.ceil(c / tile)) * tile for c in counts if c > 0)


def padded_rows_to_max(counts) -> int:
    """Rows computed when every expert is padded to the largest expert."""
    return len(counts) * max(counts)
