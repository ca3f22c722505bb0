"""Seeded random shapes through every entry point, against the oracle.

The other GPU tests pick their shapes by hand (tile edges, ragged tails, the
bench's workloads).  These draw them: batch, heads (grouped key/value heads
included), query and key lengths that fall anywhere against the 128-row
tiles and 128-key blocks, both head dims, causal masks of both alignments,
peaky logits; packed sequences with empty ones; FP8 inputs; and gradients.
The draws are fixed by their seeds, so a failure names a reproducible case.
Each case is checked with the bar of its own suite.
"""

from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from exact_attention_63_gb300 import attn, inputs
from gpu_common import assert_close, f64, need_gpu
from test_bwd_gpu import check as check_grad, grads
from test_fp8_gpu import _check as check_fp8
from test_varlen_gpu import check as check_varlen

pytestmark = pytest.mark.gpu


def _dense_cases(n: int, seed: int, d_choices=(64, 128), max_len: int = 700, aligns=("top-left", "bottom-right")):
    r = np.random.default_rng(seed)
    out = []
    for i in range(n):
        d = int(r.choice(d_choices))
        h_kv = int(r.choice([1, 2, 4]))
        H = h_kv * int(r.choice([1, 2, 3]))
        B = int(r.integers(1, 4))
        Sq, Sk = int(r.integers(1, max_len)), int(r.integers(1, max_len))
        causal = bool(r.integers(2))
        align = str(r.choice(list(aligns))) if causal else "top-left"
        sigma = float(r.choice([1.0, 3.0]))
        out.append(inputs.custom(B, H, Sq, Sk, d, causal, sigma_qk=sigma, seed=seed * 100 + i,
                                 H_kv=h_kv if h_kv != H else 0, causal_align=align,
                                 name=f"rand{seed}_{i}_b{B}h{H}kv{h_kv}_q{Sq}k{Sk}_d{d}"
                                      f"{'_causal_' + align if causal else ''}"))
    return out


def _offset(w):
    return (w.Sk - w.Sq) if (w.causal and w.causal_align == "bottom-right") else 0


@pytest.mark.parametrize("w", _dense_cases(48, 7) + _dense_cases(6, 11, max_len=2500), ids=lambda w: w.name)
def test_forward_random_shapes(w):
    """attn_fwd (grouped heads, both causal alignments) on every element; rows
    that see no key (bottom-right with Sq > Sk) must give O = 0, LSE = −inf."""
    need_gpu()
    q, k, v = inputs.make_inputs(w)
    dev = torch.device("cuda:0")
    o, lse = attn.attn_fwd(q.to(dev), k.to(dev), v.to(dev), causal=w.causal, scale=w.scale,
                           causal_align=w.causal_align)
    torch.cuda.synchronize()
    assert attn.get_status() == 0
    O_ref, L_ref = oracle.attention_forward(q, k, v, w.scale, w.causal, causal_offset=_offset(w))
    o64, l64 = f64(o), f64(lse)                      # [B, Sq, H, d], [B, H, Sq]
    unseen = ~np.isfinite(L_ref)
    assert np.array_equal(unseen, np.isneginf(l64)), f"{w.name}: LSE −inf pattern differs"
    ot = np.transpose(o64, (0, 2, 1, 3))             # [B, H, Sq, d]
    rt = np.transpose(O_ref, (0, 2, 1, 3))
    if unseen.any():
        assert np.all(ot[unseen] == 0.0), f"{w.name}: rows without keys are not zero"
    seen = ~unseen
    assert_close(ot[seen], l64[seen], rt[seen], L_ref[seen], w.name)


def _varlen_cases(n: int, seed: int):
    r = np.random.default_rng(seed)
    out = []
    for i in range(n):
        n_seq = int(r.integers(1, 13))
        lens_q = [int(x) for x in r.integers(0, 420, size=n_seq)]
        lens_k = lens_q if r.integers(2) else [int(x) for x in r.integers(0, 420, size=n_seq)]
        if max(lens_q) == 0:
            lens_q[0] = 1
        d = int(r.choice([64, 128]))
        h_kv = int(r.choice([1, 2]))
        H = h_kv * int(r.choice([1, 2]))
        causal = bool(r.integers(2))
        align = str(r.choice(["top-left", "bottom-right"])) if causal else "top-left"
        out.append((f"randvl{seed}_{i}_n{n_seq}_h{H}kv{h_kv}_d{d}{'_causal_' + align if causal else ''}",
                    lens_q, lens_k, H, h_kv, d, causal, align, seed * 100 + i))
    return out


@pytest.mark.parametrize("case", _varlen_cases(20, 8), ids=lambda c: c[0])
def test_varlen_random_shapes(case):
    """attn_fwd_varlen on random length mixes (empty sequences included)."""
    need_gpu()
    name, lens_q, lens_k, H, H_kv, d, causal, align, seed = case
    q, k, v, cu_q, cu_k = inputs.make_varlen_inputs(lens_q, lens_k, H, H_kv, d, seed)
    dev = torch.device("cuda:0")
    o, lse = attn.attn_fwd_varlen(q.to(dev), k.to(dev), v.to(dev), cu_q.to(dev), cu_k.to(dev),
                                  max(max(lens_q), 1), causal=causal, causal_align=align)
    torch.cuda.synchronize()
    assert attn.get_status() == 0
    O_ref, L_ref = oracle.attention_varlen(q, k, v, cu_q.numpy(), cu_k.numpy(), 1.0 / np.sqrt(d), causal,
                                           bottom_right=(align == "bottom-right"))
    check_varlen(o, lse, O_ref, L_ref, name)


@pytest.mark.parametrize("w", [w for w in _dense_cases(24, 9, d_choices=(128,), aligns=("top-left",))
                               if not w.H_kv], ids=lambda w: w.name)
def test_fp8_random_shapes(w):
    """attn_fwd_fp8 (dense heads, top-left causal) within the E4M3 bound."""
    need_gpu()
    q8, k8, v8, dq, dk, dv = inputs.make_fp8_inputs(w)
    o, lse = attn.attn_fwd_fp8(q8.cuda(), k8.cuda(), v8.cuda(), dq, dk, dv, causal=w.causal, scale=w.scale)
    torch.cuda.synchronize()
    assert attn.get_status() == 0
    check_fp8(w, o, lse, q8, k8, v8, dq, dk, dv)


@pytest.mark.parametrize("w", _dense_cases(16, 10, max_len=420), ids=lambda w: w.name)
def test_backward_random_shapes(w):
    """attn_bwd (grouped heads, both causal alignments) on every element of
    dQ, dK, dV."""
    need_gpu()
    q, k, v = inputs.make_inputs(w)
    g = torch.Generator().manual_seed(w.seed + 4000)
    dout = torch.randn(q.shape, generator=g).to(torch.bfloat16)
    dq, dk, dv = grads(w, q, k, v, dout)
    rq, rk, rv = oracle.attention_backward(q, k, v, dout, w.scale, w.causal, causal_offset=_offset(w))
    check_grad("dq", dq, rq, w.name)
    check_grad("dk", dk, rk, w.name)
    check_grad("dv", dv, rv, w.name)
