"""FP8 (E4M3) forward against the oracle over the exact E4M3 inputs.

The method ("FlashAttention-3: Pipeline Assíncrono …", section "Estabilidade
em FP8") computes the row's exact maximum first, then p = exp(s − m) ≤ 1 and
O = P·V with P rounded to E4M3 under the static scale 448.  Everything else is
fp32 (products of E4M3 values are exact in fp32), so the difference from the
exact result over the dequantized inputs is the rounding of P, bounded
element by element:

  |O_gpu − O_ref|_ic ≤ Σ_j e_ij |v_jc| + 2⁻⁸ |O_ref,ic| + 1e-4,
  e_ij = max(2⁻⁴ P_ij, 2⁻¹⁰ / (448 L_i))  for visible keys j,

with P_ij = exp(s_ij − M_i) / L_i the exact probabilities: E4M3 keeps 3
mantissa bits (round to nearest even: relative error ≤ 2⁻⁴ for 448 p ≥ 2⁻⁶)
and spaces its subnormals 2⁻⁹ apart (absolute error ≤ 2⁻¹⁰ below that); 2⁻⁸
covers the bf16 rounding of O.  The row sums use the unrounded p, so LSE keeps
the bf16 path's bar, |ΔLSE| ≤ 1e-3.  A further check keeps the mean error well
below the mean bound (rounding errors of both signs).
"""

import numpy as np
import pytest
import torch

import oracle
from exact_attention_63_gb300 import attn, inputs
from gpu_common import need_gpu

LSE_ATOL = 1e-3


def _bound(q, k, v, scale, causal, O_ref, rows):
    """Per-element bound of the E4M3 rounding of P for query rows ``rows`` of
    one head: q [Sq, d], k, v [Sk, d] (float64, dequantized)."""
    s = oracle.head_scores(q[rows], k, scale)
    mask = oracle.visible_mask(rows, k.shape[0], causal)
    P, M, L = oracle.head_probabilities(s, mask)
    e = np.where(mask, np.maximum(2.0 ** -4 * P, 2.0 ** -10 / (448.0 * L[:, None])), 0.0)
    return e @ np.abs(v) + 2.0 ** -8 * np.abs(O_ref) + 1e-4


def _check(w, o, lse, q8, k8, v8, dq, dk, dv, row_ranges=None):
    """Every element of O and LSE (of the given query-row ranges, default all)."""
    q = oracle.e4m3_to_f64(q8) * dq
    k = oracle.e4m3_to_f64(k8) * dk
    v = oracle.e4m3_to_f64(v8) * dv
    og = o.float().cpu().numpy().astype(np.float64)
    lg = lse.cpu().numpy().astype(np.float64)
    ranges = row_ranges or [(0, w.Sq)]
    err_sum = bnd_sum = 0.0
    for b in range(w.B):
        for h in range(w.H):
            for r0, r1 in ranges:
                for c0 in range(r0, r1, 1024):
                    rows = np.arange(c0, min(r1, c0 + 1024))
                    O_ref, L_ref = oracle.attention_head(q[b, :, h], k[b, :, h], v[b, :, h], w.scale, w.causal,
                                                         rows=rows)
                    bound = _bound(q[b, :, h], k[b, :, h], v[b, :, h], w.scale, w.causal, O_ref, rows)
                    got = og[b, rows, h]
                    assert np.all(np.isfinite(got))
                    err = np.abs(got - O_ref)
                    bad = err > bound
                    assert not bad.any(), f"{w.name} b{b} h{h}: {int(bad.sum())} elements beyond the E4M3 " \
                                          f"bound (worst excess {np.max(err - bound):.3e})"
                    dl = np.abs(lg[b, h, rows] - L_ref)
                    assert dl.max() <= LSE_ATOL, f"{w.name} b{b} h{h}: max |dLSE| {dl.max():.3e}"
                    err_sum += err.sum()
                    bnd_sum += bound.sum()
    assert err_sum <= 0.5 * bnd_sum, f"{w.name}: mean error {err_sum / bnd_sum:.2f} of the mean bound"


SMALL = [
    inputs.custom(1, 2, 300, 300, 128, False, seed=81),
    inputs.custom(1, 2, 300, 300, 128, True, seed=82),
    inputs.custom(2, 3, 129, 257, 128, False, seed=83),
    inputs.custom(2, 3, 257, 129, 128, True, seed=84),
    inputs.custom(1, 1, 1, 1, 128, False, seed=85),
    inputs.custom(1, 1, 1, 1, 128, True, seed=86),
    inputs.custom(1, 2, 128, 128, 128, True, seed=87),
    inputs.custom(1, 2, 1000, 1000, 128, False, sigma_qk=3.0, seed=88),
    inputs.custom(1, 2, 1000, 1000, 128, True, sigma_qk=3.0, seed=89),
]


@pytest.mark.gpu
@pytest.mark.parametrize("w", SMALL, ids=lambda w: w.name)
def test_fp8_small_all_elements(w):
    need_gpu()
    q8, k8, v8, dq, dk, dv = inputs.make_fp8_inputs(w)
    o, lse = attn.attn_fwd_fp8(q8.cuda(), k8.cuda(), v8.cuda(), dq, dk, dv, causal=w.causal, scale=w.scale)
    torch.cuda.synchronize()
    assert attn.get_status() == 0
    _check(w, o, lse, q8, k8, v8, dq, dk, dv)


@pytest.mark.gpu
@pytest.mark.parametrize("w", SMALL, ids=lambda w: w.name)
def test_fp8_fallback_kernel_small_all_elements(w):
    """The one-CTA FP8 kernel, which serves when the full-row kernel is not
    compiled to its register split (ATTN_TEST_FALLBACK_KERNEL): the same bound."""
    need_gpu()
    q8, k8, v8, dq, dk, dv = inputs.make_fp8_inputs(w)
    opts = attn.make_options(test_flags=attn.TEST_FALLBACK_KERNEL)
    o, lse = attn.attn_fwd_fp8(q8.cuda(), k8.cuda(), v8.cuda(), dq, dk, dv, causal=w.causal, scale=w.scale,
                               options=opts)
    torch.cuda.synchronize()
    assert attn.get_status() == 0
    _check(w, o, lse, q8, k8, v8, dq, dk, dv)


@pytest.mark.gpu
@pytest.mark.parametrize("idx,heads,row_ranges", [
    (2, [(0, 0), (3, 15), (1, 7)], None),
    (3, [(0, 0), (1, 15)], None),
    (5, [(0, 0), (0, 9)], [(0, 1024), (16320, 16448), (31744, 32768)]),
])
def test_fp8_full_size_sampled_heads(idx, heads, row_ranges):
    """The bench's FP8 workloads at full size: every element of sampled heads
    (of sampled row ranges on the 32768-row workload: the first and last
    tiles and one in the middle)."""
    need_gpu()
    w = inputs.WORKLOADS[idx]
    q8, k8, v8, dq, dk, dv = inputs.make_fp8_inputs(w)
    o, lse = attn.attn_fwd_fp8(q8.cuda(), k8.cuda(), v8.cuda(), dq, dk, dv, causal=w.causal, scale=w.scale)
    torch.cuda.synchronize()
    assert attn.get_status() == 0
    for b, h in heads:
        sel = lambda t: t[b:b + 1, :, h:h + 1]
        ws = inputs.custom(1, 1, w.Sq, w.Sk, w.d, w.causal, seed=w.seed, name=f"{w.name}[b{b},h{h}]")
        _check(ws, sel(o), lse[b:b + 1, h:h + 1], sel(q8), sel(k8), sel(v8), dq, dk, dv, row_ranges)


@pytest.mark.gpu
def test_fp8_deterministic_and_rejects_bad_arguments():
    need_gpu()
    w = inputs.custom(1, 2, 500, 500, 128, True, seed=90)
    q8, k8, v8, dq, dk, dv = (t.cuda() if torch.is_tensor(t) else t for t in inputs.make_fp8_inputs(w))
    o1, l1 = attn.attn_fwd_fp8(q8, k8, v8, dq, dk, dv, causal=True)
    o2, l2 = attn.attn_fwd_fp8(q8, k8, v8, dq, dk, dv, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    with pytest.raises(attn.AttnError):
        attn.attn_fwd_fp8(q8, k8, v8, 0.0, dk, dv)
    q64 = torch.zeros((1, 8, 1, 64), dtype=torch.float8_e4m3fn, device="cuda")
    with pytest.raises(attn.AttnError):
        attn.attn_fwd_fp8(q64, q64, q64, 1.0, 1.0, 1.0)
