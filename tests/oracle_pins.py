"""Pins that tie the CPU oracle to something other than itself.

Each ``pin_*`` function raises AssertionError when the oracle is wrong.  They
are collected by ``test_oracle.py`` and re-run against deliberately broken
oracles by ``test_oracle_mutants.py`` (every planted mistake must trip at
least one pin).

Sources of truth used here, none of which is the oracle's own code:
  * brute force in pure Python (math.fsum / math.exp) on tiny inputs;
  * the online-softmax recurrence restated independently from the Python
    simulator of "FlashAttention-4 em Blackwell B200 …" (section 4, its
    ``online_softmax_accumulate`` step, which keeps O normalised), extended
    with a causal mask and run with several block sizes;
  * closed forms (tests/golden/closed_form_cases.json) and invariants that
    follow from the definition: rows of P sum to 1, constant V, a single key,
    causal row 0, Q = 0, key shift, key permutation;
  * scipy.special.softmax / logsumexp on the same score matrix.
"""

from __future__ import annotations

import json
import math
import os

import numpy as np
from scipy import special

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "closed_form_cases.json")
TOL = 1e-12


def _rng(seed):
    return np.random.default_rng(seed)


def _bf16_like(a):
    """Round float64 values to the bf16 grid (RNE) so inputs look like the GPU's."""
    f = np.asarray(a, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    u = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16) << 16
    return u.astype(np.uint32).view(np.float32).astype(np.float64)


def rand_head(seed, Sq, Sk, d, sigma=1.0):
    r = _rng(seed)
    q = _bf16_like(r.standard_normal((Sq, d)) * sigma)
    k = _bf16_like(r.standard_normal((Sk, d)) * sigma)
    v = _bf16_like(r.standard_normal((Sk, d)))
    return q, k, v


# ---------------------------------------------------------------- brute force
def brute_force_head(q, k, v, scale, causal, offset=0):
    """Pure-Python attention for one head (lists of floats, math.fsum); causal
    rows see keys j ≤ i + offset."""
    Sq, Sk, d = len(q), len(k), len(v[0])
    O, LSE = [], []
    for i in range(Sq):
        vis = [j for j in range(Sk) if (not causal) or j <= i + offset]
        if not vis:
            O.append([0.0] * d)
            LSE.append(-math.inf)
            continue
        s = {j: scale * math.fsum(q[i][c] * k[j][c] for c in range(len(q[i]))) for j in vis}
        m = max(s.values())
        e = {j: math.exp(s[j] - m) for j in vis}
        tot = math.fsum(e.values())
        O.append([math.fsum(e[j] * v[j][c] for j in vis) / tot for c in range(d)])
        LSE.append(m + math.log(tot))
    return np.array(O), np.array(LSE)


def pin_brute_force_tiny():
    cases = [(1, 1, 8, False), (2, 2, 8, True), (3, 3, 16, True), (5, 5, 16, False),
             (17, 17, 64, True), (17, 9, 64, False), (4, 7, 8, False), (7, 4, 8, True)]
    for n, (Sq, Sk, d, causal) in enumerate(cases):
        q, k, v = rand_head(100 + n, Sq, Sk, d, sigma=2.0)
        scale = 1.0 / math.sqrt(d)
        O, L = oracle.attention_head(q, k, v, scale, causal)
        Ob, Lb = brute_force_head(q.tolist(), k.tolist(), v.tolist(), scale, causal)
        assert O.shape == Ob.shape and L.shape == Lb.shape
        fin = np.isfinite(Lb)
        assert np.array_equal(fin, np.isfinite(L)), (Sq, Sk, causal)
        assert np.max(np.abs(O - Ob)) <= TOL, (Sq, Sk, causal)
        assert np.max(np.abs(L[fin] - Lb[fin])) <= TOL, (Sq, Sk, causal)


def pin_brute_force_d64_130():
    # 130 rows = one full 128-row tile plus a ragged tail of 2.
    for causal in (False, True):
        q, k, v = rand_head(7 if causal else 8, 130, 130, 64)
        O, L = oracle.attention_head(q, k, v, 0.125, causal)
        Ob, Lb = brute_force_head(q.tolist(), k.tolist(), v.tolist(), 0.125, causal)
        assert np.max(np.abs(O - Ob)) <= TOL
        assert np.max(np.abs(L - Lb)) <= TOL


# ----------------------------------------------------------- online recurrence
def online_recurrence_head(q, k, v, scale, causal, block):
    """The simulator's per-block update, restated in float64 with a causal mask.

    Per key block: m_new = max(m, rowmax); a = exp(m − m_new) (0 when m = −inf);
    p = exp(s − m_new); l_new = a·l + Σp; O_new = (a·l·O + p·V) / l_new.
    """
    Sq, Sk = q.shape[0], k.shape[0]
    m = np.full(Sq, -np.inf)
    l = np.zeros(Sq)
    O = np.zeros((Sq, v.shape[1]))
    rows = np.arange(Sq)[:, None]
    for j0 in range(0, Sk, block):
        kb, vb = k[j0:j0 + block], v[j0:j0 + block]
        s = scale * (q @ kb.T)
        if causal:
            s = np.where(np.arange(j0, j0 + kb.shape[0])[None, :] <= rows, s, -np.inf)
        rowmax = s.max(axis=1)
        m_new = np.maximum(m, rowmax)
        a = np.where(np.isfinite(m), np.exp(m - np.where(np.isfinite(m_new), m_new, 0.0)), 0.0)
        p = np.where(np.isfinite(m_new)[:, None], np.exp(s - np.where(np.isfinite(m_new), m_new, 0.0)[:, None]), 0.0)
        l_new = a * l + p.sum(axis=1)
        safe = np.where(l_new != 0, l_new, 1.0)
        O = ((a * l)[:, None] * O + p @ vb) / safe[:, None]
        m, l = m_new, l_new
    lse = np.where(l > 0, m + np.log(np.where(l > 0, l, 1.0)), -np.inf)
    return O, lse


def pin_online_recurrence():
    for n, (Sq, Sk, d, causal) in enumerate([(64, 64, 32, False), (64, 64, 32, True),
                                             (200, 300, 64, False), (300, 300, 64, True),
                                             (129, 257, 128, True)]):
        q, k, v = rand_head(200 + n, Sq, Sk, d, sigma=3.0 if n % 2 else 1.0)
        scale = 1.0 / math.sqrt(d)
        O, L = oracle.attention_head(q, k, v, scale, causal)
        for block in (1, 7, 32, 128):
            Or, Lr = online_recurrence_head(q, k, v, scale, causal, block)
            assert np.max(np.abs(O - Or)) <= 1e-12, (n, block)
            assert np.max(np.abs(L - Lr)) <= 1e-12, (n, block)


# ------------------------------------------------------------- library routines
def pin_scipy_softmax_logsumexp():
    for causal in (False, True):
        q, k, v = rand_head(300 + causal, 96, 96, 64, sigma=2.0)
        scale = 0.125
        rows = np.arange(96)
        s = oracle.head_scores(q, k, scale)
        mask = oracle.visible_mask(rows, 96, causal)
        P, M, L = oracle.head_probabilities(s, mask)
        s_lib = scale * np.einsum("ic,jc->ij", q, k)
        s_lib = np.where(np.tril(np.ones((96, 96), bool)) if causal else True, s_lib, -np.inf)
        assert np.max(np.abs(P - special.softmax(s_lib, axis=1))) <= TOL
        O, LSE = oracle.attention_head(q, k, v, scale, causal)
        assert np.max(np.abs(LSE - special.logsumexp(s_lib, axis=1))) <= TOL
        assert np.max(np.abs(O - special.softmax(s_lib, axis=1) @ v)) <= TOL


# ------------------------------------------------------------------ invariants
def pin_rows_sum_to_one():
    for causal in (False, True):
        q, k, _ = rand_head(400 + causal, 150, 150, 64, sigma=3.0)
        P, _, _ = oracle.head_probabilities(oracle.head_scores(q, k, 0.125),
                                            oracle.visible_mask(np.arange(150), 150, causal))
        assert np.max(np.abs(P.sum(axis=1) - 1.0)) <= TOL
        assert np.all(P >= 0)
        if causal:
            assert np.all(P[np.triu(np.ones((150, 150), bool), 1)] == 0)


def pin_constant_v():
    for causal in (False, True):
        q, k, v = rand_head(500 + causal, 70, 70, 64, sigma=2.0)
        c = np.linspace(-3, 3, 64)
        v[:] = c[None, :]
        O, _ = oracle.attention_head(q, k, v, 0.125, causal)
        assert np.max(np.abs(O - c[None, :])) <= TOL


def pin_single_key():
    q, k, v = rand_head(600, 9, 1, 128, sigma=2.0)
    scale = 1.0 / math.sqrt(128)
    for causal in (False, True):
        O, L = oracle.attention_head(q, k, v, scale, causal)
        assert np.max(np.abs(O - v[0][None, :])) <= TOL
        expect = np.array([scale * math.fsum(q[i][c] * k[0][c] for c in range(128)) for i in range(9)])
        assert np.max(np.abs(L - expect)) <= TOL


def pin_causal_row0():
    q, k, v = rand_head(700, 33, 33, 64, sigma=2.0)
    O, L = oracle.attention_head(q, k, v, 0.125, True)
    assert np.max(np.abs(O[0] - v[0])) <= TOL
    assert abs(L[0] - 0.125 * math.fsum(q[0][c] * k[0][c] for c in range(64))) <= TOL
    # Row 1 sees exactly keys 0 and 1 (a two-term softmax).
    s0 = 0.125 * math.fsum(q[1][c] * k[0][c] for c in range(64))
    s1 = 0.125 * math.fsum(q[1][c] * k[1][c] for c in range(64))
    w1 = 1.0 / (1.0 + math.exp(s0 - s1))
    assert np.max(np.abs(O[1] - ((1 - w1) * v[0] + w1 * v[1]))) <= TOL


def pin_zero_q_uniform():
    _, k, v = rand_head(800, 40, 40, 64)
    q = np.zeros((40, 64))
    for causal in (False, True):
        O, L = oracle.attention_head(q, k, v, 0.125, causal)
        for i in range(40):
            n = (i + 1) if causal else 40
            assert np.max(np.abs(O[i] - v[:n].mean(axis=0))) <= TOL
            assert abs(L[i] - math.log(n)) <= TOL


def pin_key_shift():
    for causal in (False, True):
        q, k, v = rand_head(900 + causal, 50, 50, 64)
        w = _rng(901).standard_normal(64)
        O, L = oracle.attention_head(q, k, v, 0.125, causal)
        O2, L2 = oracle.attention_head(q, k + w[None, :], v, 0.125, causal)
        assert np.max(np.abs(O - O2)) <= 1e-11
        assert np.max(np.abs((L2 - L) - 0.125 * (q @ w))) <= 1e-11


def pin_key_permutation():
    q, k, v = rand_head(1000, 60, 60, 64, sigma=2.0)
    perm = _rng(1001).permutation(60)
    O, L = oracle.attention_head(q, k, v, 0.125, False)
    O2, L2 = oracle.attention_head(q, k[perm], v[perm], 0.125, False)
    assert np.max(np.abs(O - O2)) <= TOL
    assert np.max(np.abs(L - L2)) <= TOL


def pin_closed_forms():
    env = {"log": math.log, "tanh": math.tanh, "e": math.e, "exp": math.exp}
    with open(GOLDEN) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        ev = lambda m: np.array([[eval(x, {}, env) for x in row] for row in m], dtype=np.float64)  # noqa: E731
        q, k, v = ev(c["q"]), ev(c["k"]), ev(c["v"])
        O, L = oracle.attention_head(q, k, v, c["scale"], c["causal"])
        assert np.max(np.abs(O - ev(c["o"]))) <= TOL, c["name"]
        assert np.max(np.abs(L - np.array([eval(x, {}, env) for x in c["lse"]]))) <= TOL, c["name"]


def pin_forward_layout():
    """attention_forward maps (batch, seq, head, dim) slices to per-head results."""
    r = _rng(1100)
    B, S, H, d = 2, 19, 3, 64
    q = _bf16_like(r.standard_normal((B, S, H, d)))
    k = _bf16_like(r.standard_normal((B, S + 4, H, d)))
    v = _bf16_like(r.standard_normal((B, S + 4, H, d)))
    O, L = oracle.attention_forward(q, k, v, 0.125, False)
    assert O.shape == (B, S, H, d) and L.shape == (B, H, S)
    for b in range(B):
        for h in range(H):
            Ob, Lb = brute_force_head(q[b, :, h].tolist(), k[b, :, h].tolist(), v[b, :, h].tolist(), 0.125, False)
            assert np.max(np.abs(O[b, :, h] - Ob)) <= TOL
            assert np.max(np.abs(L[b, h] - Lb)) <= TOL


def pin_rows_subset():
    q, k, v = rand_head(1200, 300, 300, 64)
    rows = np.array([0, 1, 127, 128, 255, 299])
    for causal in (False, True):
        O, L = oracle.attention_head(q, k, v, 0.125, causal)
        Os, Ls = oracle.attention_head(q, k, v, 0.125, causal, rows=rows)
        assert np.max(np.abs(O[rows] - Os)) <= TOL and np.max(np.abs(L[rows] - Ls)) <= TOL
        Ob, Lb = brute_force_head(q[rows].tolist(), k.tolist(), v.tolist(), 0.125, False) if not causal else (None, None)
        if not causal:
            assert np.max(np.abs(Os - Ob)) <= TOL and np.max(np.abs(Ls - Lb)) <= TOL


def pin_combine_partials():
    """Merging key-range partials reproduces the whole (non-causal and causal)."""
    for causal in (False, True):
        q, k, v = rand_head(1300 + causal, 80, 200, 64, sigma=2.0)
        O, L = oracle.attention_head(q, k, v, 0.125, causal)
        parts_o, parts_l = [], []
        for a, b in [(0, 50), (50, 51), (51, 130), (130, 200)]:
            rows = np.arange(80)
            mask = oracle.visible_mask(rows, 200, causal)[:, a:b]
            s = 0.125 * np.einsum("ic,jc->ij", q, k[a:b])
            Ob, Lb = brute_force_masked(s, mask, v[a:b])
            parts_o.append(Ob)
            parts_l.append(Lb)
        Oc, Lc = oracle.combine_partials(parts_o, parts_l)
        assert np.max(np.abs(Oc - O)) <= 1e-12 and np.max(np.abs(Lc - L)) <= 1e-12


def brute_force_masked(s, mask, v):
    n = s.shape[0]
    O = np.zeros((n, v.shape[1]))
    L = np.full(n, -np.inf)
    for i in range(n):
        vis = np.nonzero(mask[i])[0]
        if vis.size == 0:
            continue
        m = s[i, vis].max()
        e = np.exp(s[i, vis] - m)
        L[i] = m + math.log(math.fsum(e))
        O[i] = (e @ v[vis]) / math.fsum(e)
    return O, L


# ------------------------------------------------ grouped heads, causal offset
def pin_gqa_brute_force_and_repeat():
    """Grouped-query attention: query head h reads key/value head h // (H/H_kv).
    Checked per head against brute force, and against ordinary attention on
    K/V whose heads are repeated H/H_kv times in place (the usual way a grouped
    model is run on a kernel without grouping)."""
    r = _rng(1400)
    B, S, Sk, H, H_kv, d = 2, 9, 11, 6, 2, 8
    q = _bf16_like(r.standard_normal((B, S, H, d)))
    k = _bf16_like(r.standard_normal((B, Sk, H_kv, d)))
    v = _bf16_like(r.standard_normal((B, Sk, H_kv, d)))
    for causal in (False, True):
        O, L = oracle.attention_forward(q, k, v, 0.3, causal)
        for b in range(B):
            for h in range(H):
                g = h // (H // H_kv)
                Ob, Lb = brute_force_head(q[b, :, h].tolist(), k[b, :, g].tolist(), v[b, :, g].tolist(), 0.3, causal)
                assert np.max(np.abs(O[b, :, h] - Ob)) <= TOL and np.max(np.abs(L[b, h] - Lb)) <= TOL
        Or, Lr = oracle.attention_forward(q, np.repeat(k, H // H_kv, axis=2), np.repeat(v, H // H_kv, axis=2), 0.3,
                                          causal)
        assert np.max(np.abs(O - Or)) <= TOL and np.max(np.abs(L - Lr)) <= TOL
    # MQA (one key/value head): every query head reads it.
    O1, L1 = oracle.attention_forward(q, k[:, :, :1], v[:, :, :1], 0.3, False)
    for h in range(H):
        Ob, Lb = brute_force_head(q[0, :, h].tolist(), k[0, :, 0].tolist(), v[0, :, 0].tolist(), 0.3, False)
        assert np.max(np.abs(O1[0, :, h] - Ob)) <= TOL and np.max(np.abs(L1[0, h] - Lb)) <= TOL


def pin_causal_bottom_right():
    """Bottom-right alignment (key j visible to row i iff j ≤ i + Sk − Sq):
    brute force on tiny shapes, rows without a visible key (Sq > Sk) give
    O = 0 and LSE = −inf, and for Sq ≤ Sk the result equals the last Sq rows of
    the top-left causal result with Q padded in front to Sk rows."""
    for n, (Sq, Sk) in enumerate([(3, 7), (7, 3), (5, 5), (1, 9), (9, 1)]):
        q, k, v = rand_head(1500 + n, Sq, Sk, 8, sigma=2.0)
        off = Sk - Sq
        O, L = oracle.attention_head(q, k, v, 0.4, True, causal_offset=off)
        Ob, Lb = brute_force_head(q.tolist(), k.tolist(), v.tolist(), 0.4, True, offset=off)
        fin = np.isfinite(Lb)
        assert np.array_equal(fin, np.isfinite(L)), (Sq, Sk)
        assert np.array_equal(fin, np.arange(Sq) >= Sq - Sk) if Sq > Sk else fin.all()
        assert np.max(np.abs(O - Ob)) <= TOL and np.max(np.abs(L[fin] - Lb[fin])) <= TOL
        assert np.all(O[~fin] == 0.0)
    q, k, v = rand_head(1510, 40, 100, 16)
    O, L = oracle.attention_head(q, k, v, 0.25, True, causal_offset=60)
    qp = np.concatenate([np.zeros((60, 16)), q])
    Op, Lp = oracle.attention_head(qp, k, v, 0.25, True)
    assert np.max(np.abs(O - Op[60:])) <= TOL and np.max(np.abs(L - Lp[60:])) <= TOL


def pin_rows_grouped_offset():
    """attention_rows agrees with attention_forward on sampled rows, with
    grouped heads and a causal offset."""
    r = _rng(1600)
    B, Sq, Sk, H, H_kv, d = 1, 50, 70, 4, 2, 16
    q = _bf16_like(r.standard_normal((B, Sq, H, d)))
    k = _bf16_like(r.standard_normal((B, Sk, H_kv, d)))
    v = _bf16_like(r.standard_normal((B, Sk, H_kv, d)))
    O, L = oracle.attention_forward(q, k, v, 0.25, True, causal_offset=Sk - Sq)
    rows = np.array([0, 7, 31, 49])
    for h in range(H):
        Os, Ls = oracle.attention_rows(q, k, v, 0.25, True, 0, h, rows, causal_offset=Sk - Sq)
        assert np.max(np.abs(O[0, rows, h] - Os)) <= TOL and np.max(np.abs(L[0, h, rows] - Ls)) <= TOL


# ------------------------------------------------------ packed sequences
def pin_varlen_identities():
    """Packed sequences: each sequence's rows equal the batched forward of that
    sequence alone (B = 1), equal lengths equal the batched forward of the
    reshaped tensors, and empty key or query ranges give O = 0, LSE = −inf."""
    r = _rng(1700)
    H, H_kv, d = 4, 2, 16
    lq = [5, 0, 12, 1, 9]
    lk = [7, 3, 12, 0, 4]
    cu_q, cu_k = np.concatenate([[0], np.cumsum(lq)]), np.concatenate([[0], np.cumsum(lk)])
    q = _bf16_like(r.standard_normal((cu_q[-1], H, d)))
    k = _bf16_like(r.standard_normal((cu_k[-1], H_kv, d)))
    v = _bf16_like(r.standard_normal((cu_k[-1], H_kv, d)))
    for causal, br in ((False, False), (True, False), (True, True)):
        O, L = oracle.attention_varlen(q, k, v, cu_q, cu_k, 0.25, causal, bottom_right=br)
        for s_ in range(len(lq)):
            a, b = cu_q[s_], cu_q[s_ + 1]
            if a == b:
                continue
            if lk[s_] == 0:
                assert np.all(O[a:b] == 0.0) and np.all(np.isneginf(L[:, a:b]))
                continue
            ka, kb = cu_k[s_], cu_k[s_ + 1]
            off = (kb - ka) - (b - a) if (causal and br) else 0
            Ob, Lb = oracle.attention_forward(q[None, a:b], k[None, ka:kb], v[None, ka:kb], 0.25, causal,
                                              causal_offset=off)
            fin = np.isfinite(Lb[0])
            assert np.array_equal(fin, np.isfinite(L[:, a:b]))
            assert np.max(np.abs(O[a:b] - Ob[0])) <= TOL and np.max(np.abs(L[:, a:b][fin] - Lb[0][fin])) <= TOL
            # brute force on one head of this sequence
            h = 3
            g = h // (H // H_kv)
            Oq, Lq = brute_force_head(q[a:b, h].tolist(), k[ka:kb, g].tolist(), v[ka:kb, g].tolist(), 0.25, causal,
                                      offset=off)
            fq = np.isfinite(Lq)
            assert np.max(np.abs(O[a:b, h] - Oq)) <= TOL and np.max(np.abs(L[h, a:b][fq] - Lq[fq])) <= TOL
    # equal lengths: the batched layout
    B, S = 3, 10
    qb = _bf16_like(r.standard_normal((B, S, H, d)))
    kb_ = _bf16_like(r.standard_normal((B, S, H_kv, d)))
    vb = _bf16_like(r.standard_normal((B, S, H_kv, d)))
    cu = np.arange(B + 1) * S
    O, L = oracle.attention_varlen(qb.reshape(B * S, H, d), kb_.reshape(B * S, H_kv, d), vb.reshape(B * S, H_kv, d),
                                   cu, cu, 0.25, True)
    Ob, Lb = oracle.attention_forward(qb, kb_, vb, 0.25, True)
    assert np.max(np.abs(O - Ob.reshape(B * S, H, d))) <= TOL
    assert np.max(np.abs(L - np.transpose(Lb, (1, 0, 2)).reshape(H, B * S))) <= TOL


# ----------------------------------------------------------------- backward
def _torch_grads(q, k, v, dO, scale, causal, offset=0):
    """Reference gradients from torch autograd (float64, CPU) of the plain
    formula softmax(scale·QKᵀ + mask)V: an independent implementation."""
    import torch

    qt, kt, vt = (torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (q, k, v))
    s = scale * qt @ kt.T
    if causal:
        i = torch.arange(q.shape[0])[:, None]
        j = torch.arange(k.shape[0])[None, :]
        s = s.masked_fill(j > i + offset, float("-inf"))
    o = torch.softmax(s, dim=1) @ vt
    (o * torch.tensor(dO, dtype=torch.float64)).sum().backward()
    return qt.grad.numpy(), kt.grad.numpy(), vt.grad.numpy()


def pin_backward_autograd():
    """Backward against torch autograd (float64) of the plain formula."""
    for n, (Sq, Sk, d, causal, off) in enumerate([(9, 9, 8, False, 0), (9, 9, 8, True, 0), (7, 13, 16, True, 6),
                                                  (13, 5, 8, False, 0), (130, 130, 64, True, 0)]):
        q, k, v = rand_head(1800 + n, Sq, Sk, d, sigma=1.5)
        dO = _bf16_like(_rng(1850 + n).standard_normal((Sq, d)))
        dQ, dK, dV, D = oracle.attention_backward_head(q, k, v, dO, 0.3, causal, causal_offset=off)
        tQ, tK, tV = _torch_grads(q, k, v, dO, 0.3, causal, off)
        assert np.max(np.abs(dQ - tQ)) <= 1e-10 and np.max(np.abs(dK - tK)) <= 1e-10
        assert np.max(np.abs(dV - tV)) <= 1e-10


def pin_backward_finite_differences():
    """Central differences of the loss Σ O∘dO on a tiny causal problem."""
    q, k, v = rand_head(1900, 5, 6, 4, sigma=1.0)
    dO = _rng(1901).standard_normal((5, 4))
    dQ, dK, dV, _ = oracle.attention_backward_head(q, k, v, dO, 0.7, True, causal_offset=1)

    def loss(q_, k_, v_):
        O, _ = oracle.attention_head(q_, k_, v_, 0.7, True, causal_offset=1)
        return float((O * dO).sum())

    h = 1e-6
    for (arr, grad) in ((q, dQ), (k, dK), (v, dV)):
        for idx in [(0, 0), (2, 3), (4, 1)]:
            if idx[0] >= arr.shape[0]:
                continue
            a, b = arr.copy(), arr.copy()
            a[idx] += h
            b[idx] -= h
            args_a = [a if arr is x else x for x in (q, k, v)]
            args_b = [b if arr is x else x for x in (q, k, v)]
            fd = (loss(*args_a) - loss(*args_b)) / (2 * h)
            assert abs(fd - grad[idx]) <= 1e-7, (idx, fd, grad[idx])


def pin_backward_identities():
    """D = rowsum(dO ∘ O); Σ_j dS_ij = 0 makes Σ_j dK-contributions vanish:
    adding a constant vector to every key changes nothing, so the key
    gradients sum to zero; each row of P sums to one, so the value
    gradients sum to Σ_i dO_i (every row here sees a key); scaling q by
    (1 + ε) and k by 1/(1 + ε) leaves the scores unchanged, so
    Σ_i ⟨dQ_i, q_i⟩ = Σ_j ⟨dK_j, k_j⟩; the batched call matches the per-head
    one."""
    q, k, v = rand_head(1950, 20, 30, 16, sigma=1.5)
    dO = _rng(1951).standard_normal((20, 16))
    for causal in (False, True):
        dQ, dK, dV, D = oracle.attention_backward_head(q, k, v, dO, 0.25, causal)
        O, _ = oracle.attention_head(q, k, v, 0.25, causal)
        assert np.max(np.abs(D - (dO * O).sum(axis=1))) <= TOL
        assert np.max(np.abs(dK.sum(axis=0))) <= 1e-10
        assert np.max(np.abs(dV.sum(axis=0) - dO.sum(axis=0))) <= 1e-10
        lhs, rhs = float((dQ * q).sum()), float((dK * k).sum())
        assert abs(lhs - rhs) <= 1e-10 * max(1.0, abs(lhs)) and abs(lhs) > 1e-3
    r = _rng(1952)
    qb, kb, vb, db = (_bf16_like(r.standard_normal((2, 11, 3, 8))) for _ in range(4))
    dQ, dK, dV = oracle.attention_backward(qb, kb, vb, db, 0.35, True)
    for b in range(2):
        for h in range(3):
            hq, hk, hv, _ = oracle.attention_backward_head(qb[b, :, h], kb[b, :, h], vb[b, :, h], db[b, :, h], 0.35,
                                                           True)
            assert np.array_equal(dQ[b, :, h], hq) and np.array_equal(dK[b, :, h], hk)
            assert np.array_equal(dV[b, :, h], hv)


def pin_backward_grouped_heads():
    """Grouped heads: the gradients equal those of ordinary attention on K/V
    with each head repeated for its group, with dK and dV summed over the
    group (the chain rule through the repetition)."""
    r = _rng(1960)
    B, S, Sk, H, H_kv, d = 2, 9, 12, 6, 2, 8
    q = _bf16_like(r.standard_normal((B, S, H, d)))
    k = _bf16_like(r.standard_normal((B, Sk, H_kv, d)))
    v = _bf16_like(r.standard_normal((B, Sk, H_kv, d)))
    dO = r.standard_normal((B, S, H, d))
    g = H // H_kv
    for causal, off in ((False, 0), (True, 0), (True, Sk - S)):
        dQ, dK, dV = oracle.attention_backward(q, k, v, dO, 0.3, causal, causal_offset=off)
        rQ, rK, rV = oracle.attention_backward(q, np.repeat(k, g, axis=2), np.repeat(v, g, axis=2), dO, 0.3, causal,
                                               causal_offset=off)
        assert np.max(np.abs(dQ - rQ)) <= TOL
        assert np.max(np.abs(dK - rK.reshape(B, Sk, H_kv, g, d).sum(axis=3))) <= TOL
        assert np.max(np.abs(dV - rV.reshape(B, Sk, H_kv, g, d).sum(axis=3))) <= TOL


def pin_backward_rows_subset():
    """Selected gradient rows equal the same rows of the whole-head backward
    (causal with an offset, and non-causal; 1100 query rows, so the key-row
    sums cross a query chunk)."""
    rng = np.random.default_rng(17)
    Sq, Sk, d = 1100, 260, 8
    q, k, v, dO = (rng.standard_normal((n, d)) for n in (Sq, Sk, Sk, Sq))
    qrows = np.array([0, 1, 127, 128, 150, 1023, 1024, 1099])
    krows = np.array([0, 5, 128, 200, 259])
    for causal, off in ((False, 0), (True, 0), (True, Sk - Sq)):
        dq, dk, dv, _ = oracle.attention_backward_head(q, k, v, dO, 0.3, causal, off)
        rq, rk, rv = oracle.attention_backward_rows(q, k, v, dO, 0.3, causal, qrows, krows, off)
        assert np.allclose(rq, dq[qrows], atol=1e-12)
        assert np.allclose(rk, dk[krows], atol=1e-12)
        assert np.allclose(rv, dv[krows], atol=1e-12)


# ---------------------------------------------------------------- FP8 (E4M3)
def _e4m3_by_hand(b: int) -> float:
    """Decode one E4M3 byte from its fields (1 sign, 4 exponent bits with bias
    7, 3 mantissa bits; exponent 0 is subnormal; 0x7F/0xFF are NaN; no inf)."""
    sign = -1.0 if b & 0x80 else 1.0
    e, m = (b >> 3) & 0xF, b & 0x7
    if e == 0xF and m == 0x7:
        return math.nan
    if e == 0:
        return sign * (m / 8.0) * 2.0 ** -6
    return sign * (1.0 + m / 8.0) * 2.0 ** (e - 7)


def pin_e4m3_decoding():
    import torch

    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    got = oracle.e4m3_to_f64(codes)
    want = np.array([_e4m3_by_hand(b) for b in range(256)])
    assert np.array_equal(np.isnan(got), np.isnan(want))
    ok = ~np.isnan(want)
    assert np.array_equal(got[ok], want[ok])
    assert want[ok].max() == 448.0 and want[ok].min() == -448.0


def _fp8_case(seed, B=1, Sq=5, Sk=7, H=2, d=64):
    import torch

    g = torch.Generator().manual_seed(seed)
    q8 = (torch.randn((B, Sq, H, d), generator=g) * 40).to(torch.float8_e4m3fn)
    k8 = (torch.randn((B, Sk, H, d), generator=g) * 40).to(torch.float8_e4m3fn)
    v8 = (torch.randn((B, Sk, H, d), generator=g) * 40).to(torch.float8_e4m3fn)
    return q8, k8, v8


def pin_fp8_brute_force():
    """The FP8 forward over the hand-decoded values, with the scale factors, by
    pure-Python loops (math.fsum / math.exp)."""
    q8, k8, v8 = _fp8_case(5)
    dq, dk, dv, scale = 0.011, 0.02, 0.007, 0.125
    dec = lambda t: np.vectorize(_e4m3_by_hand)(t.view(__import__("torch").uint8).numpy().astype(np.int64))
    q, k, v = dec(q8) * dq, dec(k8) * dk, dec(v8) * dv
    for causal in (False, True):
        O, L = oracle.attention_forward_fp8(q8, k8, v8, dq, dk, dv, scale, causal)
        B, Sq, H, d = q.shape
        for h in range(H):
            for i in range(Sq):
                keys = [j for j in range(k.shape[1]) if not causal or j <= i]
                s = [scale * math.fsum(q[0, i, h, c] * k[0, j, h, c] for c in range(d)) for j in keys]
                mx = max(s)
                e = [math.exp(x - mx) for x in s]
                tot = math.fsum(e)
                assert abs(L[0, h, i] - (mx + math.log(tot))) <= 1e-12
                for c in range(d):
                    o = math.fsum(e[n] * v[0, j, h, c] for n, j in enumerate(keys)) / tot
                    assert abs(O[0, i, h, c] - o) <= 1e-12


def pin_fp8_scale_factors():
    """descale_q and descale_k act as a factor on the logits, descale_v as a
    factor on O (LSE unchanged)."""
    q8, k8, v8 = _fp8_case(6, Sq=9, Sk=11)
    O1, L1 = oracle.attention_forward_fp8(q8, k8, v8, 0.02, 0.01, 0.5, 0.1, True)
    O2, L2 = oracle.attention_forward_fp8(q8, k8, v8, 0.01, 0.01, 0.5, 0.2, True)
    O3, L3 = oracle.attention_forward_fp8(q8, k8, v8, 0.02, 0.01, 1.5, 0.1, True)
    assert np.allclose(O1, O2, atol=1e-13) and np.allclose(L1, L2, atol=1e-13)
    assert np.allclose(3 * O1, O3, atol=1e-12) and np.allclose(L1, L3, atol=1e-13)
    O4, L4 = oracle.attention_forward_fp8(q8, k8, v8, 0.02, 0.03, 0.5, 0.1, True)
    assert not np.allclose(L1, L4)  # descale_k is not ignored


ALL_PINS = [v for k_, v in sorted(globals().items()) if k_.startswith("pin_") and callable(v)]
