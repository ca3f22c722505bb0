"""Grouped-query heads, bottom-right causal alignment and strided layouts
(attn_fwd_layout), GPU path vs the CPU oracle element by element."""

from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from exact_attention_63_gb300 import attn, inputs
from gpu_common import assert_close, f64, need_gpu, sample_rows

pytestmark = pytest.mark.gpu

C = inputs.custom
CASES = [
    # grouped-query attention, multi-query attention
    C(2, 8, 300, 300, 128, False, seed=61, H_kv=2),
    C(2, 8, 300, 300, 128, True, seed=62, H_kv=2),
    C(1, 4, 257, 383, 64, False, seed=63, H_kv=1),
    C(1, 6, 130, 130, 64, True, seed=64, H_kv=3),
    # bottom-right alignment: Sq < Sk, Sq > Sk (rows without keys), one query row
    C(1, 2, 200, 520, 128, True, seed=65, causal_align="bottom-right"),
    C(1, 2, 520, 200, 64, True, seed=66, causal_align="bottom-right"),
    C(2, 2, 129, 1000, 64, True, seed=67, causal_align="bottom-right"),
    C(1, 3, 1000, 129, 128, True, seed=68, causal_align="bottom-right"),
    C(2, 2, 1, 300, 128, True, seed=69, causal_align="bottom-right"),
    C(1, 2, 300, 1, 64, True, seed=70, causal_align="bottom-right"),
    C(1, 2, 300, 300, 64, True, seed=71, causal_align="bottom-right"),
    # both
    C(2, 8, 700, 333, 128, True, seed=72, H_kv=2, causal_align="bottom-right"),
    C(1, 4, 64, 1100, 64, True, seed=73, H_kv=1, causal_align="bottom-right"),
]


def reference(w, q, k, v, rows=None, b=0, h=0):
    off = (w.Sk - w.Sq) if (w.causal and w.causal_align == "bottom-right") else 0
    if rows is None:
        return oracle.attention_forward(q, k, v, w.scale, w.causal, causal_offset=off)
    return oracle.attention_rows(q, k, v, w.scale, w.causal, b, h, rows, causal_offset=off)


def check(o, lse, O_ref, L_ref, what):
    """Rows that see no key must be exactly O = 0, LSE = −inf; the rest within
    the parity bar."""
    o64, l64 = f64(o), f64(lse)
    unseen = ~np.isfinite(L_ref)                                   # [B, H, Sq]
    assert np.array_equal(unseen, np.isneginf(l64)), f"{what}: LSE −inf pattern differs"
    if unseen.any():
        o_unseen = np.transpose(o64, (0, 2, 1, 3))[unseen]        # [n, d]
        assert np.all(o_unseen == 0.0), f"{what}: rows without keys are not zero"
    seen = ~unseen
    assert_close(np.transpose(o64, (0, 2, 1, 3))[seen], l64[seen], np.transpose(O_ref, (0, 2, 1, 3))[seen],
                 L_ref[seen], what)


def run(w, q, k, v, **kw):
    o, lse = attn.attn_fwd(q, k, v, causal=w.causal, scale=w.scale, causal_align=w.causal_align, **kw)
    torch.cuda.synchronize()
    assert attn.get_status() == 0
    return o, lse


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_layout_cases_all_elements(w):
    need_gpu()
    q, k, v = inputs.make_inputs(w)
    o, lse = run(w, q.cuda(), k.cuda(), v.cuda())
    O_ref, L_ref = reference(w, q, k, v)
    check(o, lse, O_ref, L_ref, w.name)


def test_packed_qkv_and_strided_output():
    """q, k, v as views of one packed [B, S, 3, H, d] tensor; O written into
    a view of a wider buffer (head stride 2d)."""
    need_gpu()
    w = C(2, 4, 333, 333, 128, True, seed=74)
    q, k, v = inputs.make_inputs(w)
    packed = torch.stack([q, k, v], dim=2).cuda()                  # [B, S, 3, H, d]
    qv, kv_, vv = packed[:, :, 0], packed[:, :, 1], packed[:, :, 2]
    assert not qv.is_contiguous()
    wide = torch.full((w.B, w.Sq, w.H, 2 * w.d), 7.0, dtype=torch.bfloat16, device="cuda")
    out = wide[..., :w.d]
    o, lse = run(w, qv, kv_, vv, out=out)
    O_ref, L_ref = reference(w, q, k, v)
    check(o, lse, O_ref, L_ref, "packed qkv")
    assert torch.all(wide[..., w.d:] == 7.0), "the strided output wrote outside its view"


def test_head_major_inputs():
    """q, k, v stored (batch, heads, seq, d) and passed as permuted views."""
    need_gpu()
    w = C(2, 4, 300, 450, 64, True, seed=75, H_kv=2, causal_align="bottom-right")
    q, k, v = inputs.make_inputs(w)
    qh, kh, vh = (t.permute(0, 2, 1, 3).contiguous().cuda() for t in (q, k, v))
    o, lse = run(w, qh.permute(0, 2, 1, 3), kh.permute(0, 2, 1, 3), vh.permute(0, 2, 1, 3))
    O_ref, L_ref = reference(w, q, k, v)
    check(o, lse, O_ref, L_ref, "head-major")


def test_grouped_full_size_sampled_rows():
    """A grouped-query workload at measurement size (B=2, H=32, H_kv=8,
    S=4096, d=128, causal), checked on sampled rows."""
    need_gpu()
    w = C(2, 32, 4096, 4096, 128, True, seed=76, H_kv=8)
    q, k, v = inputs.make_inputs(w)
    o, lse = run(w, q.cuda(), k.cuda(), v.cuda())
    assert bool(torch.isfinite(o).all()) and bool(torch.isfinite(lse).all())
    o_c, l_c = o.cpu(), lse.cpu()
    for b, h, rows in sample_rows(w, seed=76):
        O_ref, L_ref = reference(w, q, k, v, rows=rows, b=b, h=h)
        assert_close(f64(o_c[b, rows, h, :]), f64(l_c[b, h, rows]), O_ref, L_ref, f"{w.name} b{b} h{h}")


def test_grouped_equals_repeated_heads():
    """The grouped kernel matches the kernel run on K/V with repeated heads
    (every element: both runs use the same arithmetic per head)."""
    need_gpu()
    w = C(1, 8, 520, 520, 128, False, seed=77, H_kv=2)
    q, k, v = (t.cuda() for t in inputs.make_inputs(w))
    o1, l1 = run(w, q, k, v)
    rep = w.H // w.kv_heads
    o2, l2 = run(w, q, k.repeat_interleave(rep, dim=2), v.repeat_interleave(rep, dim=2))
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_grouped_bench_variant_full_size_all_elements():
    """The bench's grouped-query variant (`--kv-heads 4`: B4 H16 H_kv 4 S2048
    d128) at full size, every element."""
    need_gpu()
    w = C(4, 16, 2048, 2048, 128, False, seed=2, H_kv=4)
    q, k, v = inputs.make_inputs(w)
    o, lse = run(w, q.cuda(), k.cuda(), v.cuda())
    O_ref, L_ref = reference(w, q, k, v)
    check(o, lse, O_ref, L_ref, w.name)
