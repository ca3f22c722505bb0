"""Repeated launches of every kernel variant: the outputs stay bit-identical
from launch to launch and the device status stays clean.  A race between the
pipeline's roles (a barrier phase taken for another, a buffer reused too
early) shows up here as an output that changes between launches or a wait
that runs out."""

import pytest
import torch

from exact_attention_63_gb300 import attn, inputs
from gpu_common import need_gpu

pytestmark = pytest.mark.gpu
FALLBACK = attn.make_options(test_flags=attn.TEST_FALLBACK_KERNEL)


def _repeat(fn, n, same=None):
    """`same[i](a, b)` compares output i of two launches (default: bit equality)."""
    ref = [t.clone() for t in fn()]
    for i in range(n):
        out = fn()
        if i % 25 == 24 or i == n - 1:
            torch.cuda.synchronize()
            assert attn.get_status() == 0, f"status flagged by launch {i}"
            for j, (a, b) in enumerate(zip(ref, out)):
                eq = torch.equal if same is None else same[j]
                assert eq(a, b), f"output {j} differs at launch {i}"


def _close_runs(a, b):
    # the one-pass backward's dQ: fp32 additions in a varying order
    a, b = a.float(), b.float()
    return bool(((a - b).abs() <= 2.0 ** -7 * a.abs() + 1e-3 * a.abs().max()).all())


def _dense(B, H, S, d, causal, hkv=0, align="top-left", sigma=1.0, seed=1):
    w = inputs.custom(B, H, S, S, d, causal, sigma_qk=sigma, seed=seed, H_kv=hkv, causal_align=align)
    return (w, *(t.cuda() for t in inputs.make_inputs(w)))


@pytest.mark.parametrize("d,causal,hkv,align,fallback", [
    (64, False, 0, "top-left", False), (64, False, 0, "top-left", True),
    (64, True, 2, "bottom-right", False), (128, False, 0, "top-left", False), (128, True, 4, "top-left", False),
])
def test_forward_repeats(d, causal, hkv, align, fallback):
    need_gpu()
    w, q, k, v = _dense(2, 8, 2048, d, causal, hkv=hkv, align=align, sigma=3.0 if d == 64 else 1.0)
    opts = FALLBACK if fallback else None
    _repeat(lambda: attn.attn_fwd(q, k, v, causal=causal, scale=w.scale, causal_align=align, options=opts), 150)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_varlen_repeats(d, causal):
    need_gpu()
    lens = inputs.varlen_lengths(24, 2048, seed=5)
    q, k, v, cq, ck = (t.cuda() for t in inputs.make_varlen_inputs(lens, lens, 8, 4, d, 9))
    _repeat(lambda: attn.attn_fwd_varlen(q, k, v, cq, ck, max(lens), causal=causal), 100)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("fallback", [False, True])
def test_fp8_repeats(causal, fallback):
    need_gpu()
    w = inputs.custom(2, 8, 2048, 2048, 128, causal, seed=3)
    q8, k8, v8, dq, dk, dv = inputs.make_fp8_inputs(w)
    q8, k8, v8 = q8.cuda(), k8.cuda(), v8.cuda()
    opts = FALLBACK if fallback else None
    _repeat(lambda: attn.attn_fwd_fp8(q8, k8, v8, dq, dk, dv, causal=causal, options=opts), 150)


@pytest.mark.parametrize("deterministic", [False, True])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_backward_repeats(d, causal, deterministic):
    """The two-pass schedule bit for bit; the one-pass one bit for bit in dK,
    dV and up to the order of its fp32 additions in dQ."""
    need_gpu()
    w, q, k, v = _dense(2, 8, 2048, d, causal, hkv=4)
    o, lse = attn.attn_fwd(q, k, v, causal=causal, scale=w.scale)
    g = torch.randn(q.shape, generator=torch.Generator().manual_seed(7)).to(torch.bfloat16).cuda()
    same = None if deterministic else [_close_runs, torch.equal, torch.equal]
    _repeat(lambda: attn.attn_bwd(q, k, v, o, lse, g, causal=causal, scale=w.scale, deterministic=deterministic),
            100, same)
