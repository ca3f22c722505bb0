"""The process-pool form of the oracle used by the full-size GPU parity tests
gives exactly the serial oracle's values (CPU only)."""

from __future__ import annotations

import numpy as np

import oracle
import oracle_pool
from exact_attention_63_gb300 import inputs


def test_pool_matches_serial_oracle():
    w = inputs.custom(2, 3, 300, 260, 64, True, seed=5)
    q, k, v = inputs.make_inputs(w)
    O1, L1 = oracle_pool.attention_forward_pool(q, k, v, w.scale, w.causal, workers=2)
    O2, L2 = oracle.attention_forward(q, k, v, w.scale, w.causal)
    assert O1.shape == O2.shape and L1.shape == L2.shape
    assert np.array_equal(O1, O2) and np.array_equal(L1, L2)


def test_backward_pool_matches_serial_oracle():
    w = inputs.custom(2, 2, 200, 200, 64, True, seed=6)
    q, k, v = inputs.make_inputs(w)
    import torch
    g = torch.randn(q.shape, generator=torch.Generator().manual_seed(7)).to(torch.bfloat16)
    got = oracle_pool.attention_backward_pool(q, k, v, g, w.scale, w.causal, workers=2)
    ref = oracle.attention_backward(q, k, v, g, w.scale, w.causal)
    for a, b in zip(got, ref):
        assert a.shape == b.shape and np.array_equal(a, b)
