"""The process-pool composition of the oracle used by the full-size GPU
checks (permute, one expert FFN per worker, combine) gives exactly the
oracle's own layer."""

import numpy as np

import oracle
from tests import oracle_pool


def test_pool_layer_equals_oracle_forward():
    rng = np.random.default_rng(0)
    T, d, E, k, I = 40, 256, 8, 2, 128
    bits = oracle.f64_to_bf16_bits
    x = bits(rng.standard_normal((T, d)))
    wr = bits(rng.standard_normal((E, d)) / 16)
    gu = bits(rng.standard_normal((E, 2 * I, d)) / 16)
    dn = bits(rng.standard_normal((E, d, I)) / 11)
    ref = oracle.forward(x, wr, gu, dn, k)
    out = oracle_pool.layer_out(x, ref["ids"], ref["gates"], E, lambda e: (gu[e], dn[e]),
                                processes=2)
    assert np.array_equal(out, ref["out"])
