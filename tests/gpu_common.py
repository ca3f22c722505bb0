"""Shared helpers of the GPU tests: the library, tolerance checks, sampling."""

from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from exact_attention_63_gb300 import attn, inputs

# The parity bar: |O_gpu − O_ref| ≤ 1e-2 + 1e-2·|O_ref| elementwise and
# |LSE_gpu − LSE_ref| ≤ 1e-3 (absolute, natural log).
O_ATOL, O_RTOL, LSE_ATOL = 1e-2, 1e-2, 1e-3


def need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    attn.lib()


def run(w, q, k, v, **kw):
    dev = torch.device("cuda:0")
    o, lse = attn.attn_fwd(q.to(dev), k.to(dev), v.to(dev), causal=w.causal, scale=w.scale, **kw)
    torch.cuda.synchronize()
    assert attn.get_status() == 0
    return o, lse


def f64(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def assert_close(o, lse, O_ref, L_ref, what=""):
    o64 = o if isinstance(o, np.ndarray) else f64(o)
    l64 = lse if isinstance(lse, np.ndarray) else f64(lse)
    assert np.all(np.isfinite(o64)) and np.all(np.isfinite(l64)), f"{what}: non-finite output"
    excess = np.abs(o64 - O_ref) - (O_ATOL + O_RTOL * np.abs(O_ref))
    n_bad = int((excess > 0).sum())
    assert n_bad == 0, f"{what}: {n_bad} O elements out of tolerance (max excess {excess.max():.3e})"
    dl = np.abs(l64 - L_ref)
    assert dl.max() <= LSE_ATOL, f"{what}: max |dLSE| = {dl.max():.3e}"
    return float(np.abs(o64 - O_ref).max()), float(dl.max())


def sample_rows(w, n_heads=6, seed=0):
    """(b, h, rows) samples: tile edges, the first and last rows, random rows."""
    r = np.random.default_rng(1000 + seed)
    out = []
    fixed = sorted({0, 1, 127, 128, 255, 256, w.Sq // 2, w.Sq - 129, w.Sq - 128, w.Sq - 2, w.Sq - 1} &
                   set(range(w.Sq)))
    for i in range(n_heads):
        b = int(r.integers(w.B)) if i else 0
        h = int(r.integers(w.H)) if i else 0
        if i == n_heads - 1:
            b, h = w.B - 1, w.H - 1
        rows = sorted(set(fixed) | set(int(x) for x in r.integers(0, w.Sq, size=6)))
        out.append((b, h, np.array(rows)))
    return out
