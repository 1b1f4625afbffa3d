"""Per-expert oracle work spread over host processes, for the full-size checks.

The oracle's expert FFN treats experts independently ('Chapter 9. Distributed
inference', section 9.3.4: each expert multiplies its own rows), so a layer's
y can be formed expert by expert in worker processes and combined with the
oracle's own combine.  Workers are started with "spawn" (never forked from a
process that has touched the GPU) and run only oracle code on host arrays.
"""

from __future__ import annotations

import concurrent.futures as cf
import multiprocessing as mp
import os

import numpy as np

import oracle


def _expert_y(args):
    """y rows of one expert: the oracle's SwiGLU FFN on the oracle's own
    quantise-dequantise round trip of the expert's bf16 weights (fmt "mxfp8",
    "nvfp4"; "mxfp8_a8": MXFP8 weights and tokens) or on the bf16 weights
    themselves (fmt None)."""
    fmt, x_rows, gu_bits, d_bits = args

    def weights(bits):
        if fmt is None:
            return bits
        vals = oracle.bf16_bits_to_f64(bits)
        if fmt in ("mxfp8", "mxfp8_a8"):
            return oracle.f64_to_bf16_bits(oracle.mxfp8_dequantize(*oracle.mxfp8_quantize(vals)))
        return oracle.nvfp4_dequantize(*oracle.nvfp4_quantize(vals.astype(np.float32)))

    return oracle.swiglu_ffn(x_rows, weights(gu_bits), weights(d_bits), act_mxfp8=fmt == "mxfp8_a8")


def layer_out(x_bits, ids, gates, E, expert_bits, fmt=None, processes=None):
    """The oracle's layer output [T, d] for the given routing: permute, one
    expert FFN per active expert (in worker processes), combine.
    expert_bits(e) -> (w_gate_up bits [2I, d], w_down bits [d, I])."""
    T, k = ids.shape
    counts, offsets, perm, slot_pos = oracle.permute(ids, E)
    x_perm = oracle.bf16_bits_to_f64(np.asarray(x_bits))[perm // k]
    active = [e for e in range(E) if counts[e] > 0]
    y = np.zeros((T * k, x_perm.shape[1]), dtype=np.float64)
    n = processes or min(16, os.cpu_count() or 1)
    # a worker that dies raises BrokenProcessPool here instead of being
    # respawned; at most 2n experts' weights are in flight at a time
    with cf.ProcessPoolExecutor(n, mp_context=mp.get_context("spawn")) as pool:
        for w0 in range(0, len(active), 2 * n):
            window = active[w0:w0 + 2 * n]
            futs = [pool.submit(_expert_y, (fmt, x_perm[offsets[e]:offsets[e + 1]],
                                            *expert_bits(e))) for e in window]
            for e, f in zip(window, futs):
                y[offsets[e]:offsets[e + 1]] = f.result()
    return oracle.combine(y, slot_pos, gates)
