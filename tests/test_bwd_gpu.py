"""Backward pass (attn_bwd): GPU gradients vs the CPU oracle's, element by
element, for both schedules: the default (at d = 64 the one-pass kernel, dQ
added up across key tiles in fp32; at d = 128 the two passes) and the
deterministic one (two passes at every head dim)."""

from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import oracle_pool
from exact_attention_63_gb300 import attn, inputs
from gpu_common import f64, need_gpu

pytestmark = pytest.mark.gpu

# Gradient tolerance (the parity bar of the forward covers O and LSE only):
# every element within 1e-2 of the tensor's largest |value| plus 1e-2 of its
# own |value|.  Sources of error: P and dS rounded to bf16 before their
# products (2^-9 relative per term), D from the bf16 O, outputs rounded once
# to bf16 (2^-9 relative).
G_ATOL, G_RTOL = 1e-2, 1e-2

C = inputs.custom
CASES = [
    C(1, 2, 256, 256, 64, False, seed=101),
    C(1, 2, 300, 300, 128, True, seed=102),
    C(2, 3, 129, 200, 64, False, seed=103),
    C(1, 2, 64, 500, 128, True, seed=104),
    C(1, 2, 500, 64, 64, True, seed=105),
    C(1, 1, 1000, 1000, 128, True, seed=106),
    C(1, 2, 640, 640, 64, False, sigma_qk=3.0, seed=107),
    # grouped key/value heads, bottom-right alignment (Sq < Sk and Sq > Sk)
    C(2, 8, 300, 300, 128, True, seed=110, H_kv=2),
    C(1, 4, 257, 383, 64, False, seed=111, H_kv=1),
    C(1, 2, 200, 520, 128, True, seed=112, causal_align="bottom-right"),
    C(1, 2, 520, 200, 64, True, seed=113, causal_align="bottom-right"),
    C(1, 6, 700, 333, 128, True, seed=114, H_kv=3, causal_align="bottom-right"),
    # more tiles than SMs (several waves of CTAs): short tiles (two blocks),
    # causal with grouped heads, and tiles whose rows see no key between
    # tiles that do
    C(1, 160, 256, 256, 64, False, seed=115),
    C(1, 80, 384, 384, 128, True, seed=116, H_kv=16),
    C(1, 64, 520, 200, 64, True, seed=117, causal_align="bottom-right"),
]


SCHEDULES = {"default": False, "deterministic": True}


def grads(w, q, k, v, dout, deterministic: bool = False):
    dev = torch.device("cuda:0")
    qd, kd, vd, gd = (t.to(dev) for t in (q, k, v, dout))
    o, lse = attn.attn_fwd(qd, kd, vd, causal=w.causal, scale=w.scale, causal_align=w.causal_align)
    dq, dk, dv = attn.attn_bwd(qd, kd, vd, o, lse, gd, causal=w.causal, scale=w.scale, causal_align=w.causal_align,
                               deterministic=deterministic)
    torch.cuda.synchronize()
    assert attn.get_status() == 0
    return dq, dk, dv


def check(name, got, ref, what):
    g = f64(got)
    assert np.all(np.isfinite(g)), f"{what} {name}: non-finite"
    bound = G_ATOL * np.abs(ref).max() + G_RTOL * np.abs(ref)
    excess = np.abs(g - ref) - bound
    assert (excess <= 0).all(), (f"{what} {name}: {(excess > 0).sum()} elements out of tolerance, "
                                 f"max |err| {np.abs(g - ref).max():.3e} (max |ref| {np.abs(ref).max():.3e})")


@pytest.mark.parametrize("schedule", SCHEDULES)
@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_backward_matches_oracle(w, schedule):
    need_gpu()
    q, k, v = inputs.make_inputs(w)
    g = torch.Generator().manual_seed(w.seed + 1000)
    dout = torch.randn(q.shape, generator=g).to(torch.bfloat16)
    dq, dk, dv = grads(w, q, k, v, dout, SCHEDULES[schedule])
    off = (w.Sk - w.Sq) if (w.causal and w.causal_align == "bottom-right") else 0
    rq, rk, rv = oracle.attention_backward(q, k, v, dout, w.scale, w.causal, causal_offset=off)
    check("dq", dq, rq, w.name)
    check("dk", dk, rk, w.name)
    check("dv", dv, rv, w.name)


def test_backward_padded_keys_with_very_negative_scores():
    """Every score of every query far below zero (LSE < −88, where exp(−LSE)
    overflows fp32) and Sk not a multiple of the 128-key tile: the tile's
    padding rows (zero K and V, score 0) must not reach the gradients.

    Scores that low need keys sharing a large component c·u against the
    queries.  Each query's dS sums to zero over the keys, so that component
    cancels out of dQ = scale·dS·K exactly, but not after dS is rounded to
    bf16 (in any schedule): dQ's error lies along u.  dQ is therefore
    checked with its u component removed (and for finiteness); dK and dV as
    everywhere."""
    need_gpu()
    w = C(1, 2, 200, 300, 64, False, seed=118)
    q, k, v = inputs.make_inputs(w)
    base = torch.randn(64, generator=torch.Generator().manual_seed(3)).double()
    u = base / base.norm()
    # q·k ≈ −40·24 = −960 (noise ±40 from the unit-variance parts): scores ≈ −120 ± 5
    q = (40.0 * u.expand(1, w.Sq, w.H, 64) + q.double()).to(torch.bfloat16)
    k = (-24.0 * u.expand(1, w.Sk, w.H, 64) + k.double()).to(torch.bfloat16)
    g = torch.Generator().manual_seed(w.seed + 1000)
    dout = torch.randn(q.shape, generator=g).to(torch.bfloat16)
    dev = torch.device("cuda:0")
    o, lse = attn.attn_fwd(q.to(dev), k.to(dev), v.to(dev), scale=w.scale)
    assert float(lse.max()) < -88.0
    rq, rk, rv = oracle.attention_backward(q, k, v, dout, w.scale, False)
    un = u.numpy()
    perp = lambda x: x - (x @ un)[..., None] * un
    for schedule, det in SCHEDULES.items():
        dq, dk, dv = grads(w, q, k, v, dout, det)
        assert np.all(np.isfinite(f64(dq))), f"{schedule}: dq non-finite"
        check("dq ⟂ u", torch.from_numpy(perp(f64(dq))), perp(rq), f"{w.name} {schedule}")
        check("dk", dk, rk, f"{w.name} {schedule}")
        check("dv", dv, rv, f"{w.name} {schedule}")


@pytest.mark.parametrize("idx", [2, 3, 4])
def test_backward_full_size_all_elements(idx):
    """The bench's backward workloads at full size (B4 H16 S2048 d128; B2 H16
    S8192 d128 causal; B8 H32 S4096 d64, σ_QK = 3), every element of dQ, dK,
    dV against the oracle (one head per process).  (Workload 5's oracle would
    hold 32768² float64 matrices per head.)"""
    need_gpu()
    w = inputs.WORKLOADS[idx]
    q, k, v = inputs.make_inputs(w)
    g = torch.Generator().manual_seed(w.seed + 2000)
    dout = torch.randn(q.shape, generator=g).to(torch.bfloat16)
    rq, rk, rv = oracle_pool.attention_backward_pool(q, k, v, dout, w.scale, w.causal)
    for schedule, det in SCHEDULES.items():
        dq, dk, dv = grads(w, q, k, v, dout, det)
        check("dq", dq, rq, f"{w.name} {schedule}")
        check("dk", dk, rk, f"{w.name} {schedule}")
        check("dv", dv, rv, f"{w.name} {schedule}")


def close_runs(a, b):
    """Two runs of the one-pass (d = 64) dQ: the same up to the order of its fp32
    additions (a bf16 rounding may flip: 2^-7 relative, plus 1e-3 of the
    tensor's largest |value| for sums that cancel)."""
    a, b = a.float(), b.float()
    return bool(((a - b).abs() <= 2.0 ** -7 * a.abs() + 1e-3 * a.abs().max()).all())


@pytest.mark.parametrize("d", [64, 128])
def test_backward_deterministic(d):
    """The two-pass schedule is reproducible bit for bit; the default one (the
    one-pass kernel at d = 64) in dK and dV (accumulated in tensor memory in a
    fixed order), and in dQ up to the order of the fp32 additions."""
    need_gpu()
    w = C(2, 4, 520, 520, d, True, seed=108)
    q, k, v = (t.cuda() for t in inputs.make_inputs(w))
    dout = torch.randn(q.shape, generator=torch.Generator().manual_seed(5)).to(torch.bfloat16).cuda()
    o, lse = attn.attn_fwd(q, k, v, causal=True)
    a = attn.attn_bwd(q, k, v, o, lse, dout, causal=True, deterministic=True)
    b_ = attn.attn_bwd(q, k, v, o, lse, dout, causal=True, deterministic=True)
    c = attn.attn_bwd(q, k, v, o, lse, dout, causal=True)
    e = attn.attn_bwd(q, k, v, o, lse, dout, causal=True)
    torch.cuda.synchronize()
    assert attn.get_status() == 0
    assert all(torch.equal(x, y) for x, y in zip(a, b_))
    assert torch.equal(c[1], e[1]) and torch.equal(c[2], e[2])
    assert close_runs(c[0], e[0])


def test_backward_longest_workload_sampled_rows():
    """Workload 5's backward at full size (B1 H16 S32768 d128 causal): dQ rows
    and dK, dV rows sampled across the sequence (the first and last tiles,
    tile edges, the middle, random rows) in two heads, against the oracle's
    per-row gradients (its whole-head matrices would be 32768² float64).  The
    tolerance's scale is the largest |value| among the sampled rows."""
    need_gpu()
    w = inputs.WORKLOADS[5]
    q, k, v = inputs.make_inputs(w)
    g = torch.Generator().manual_seed(w.seed + 2000)
    dout = torch.randn(q.shape, generator=g).to(torch.bfloat16)
    dq, dk, dv = grads(w, q, k, v, dout)
    rng = np.random.default_rng(5)
    fixed = [0, 1, 127, 128, 255, 256, 16383, 16384, w.Sq - 129, w.Sq - 128, w.Sq - 1]
    rows = np.array(sorted(set(fixed) | set(int(x) for x in rng.integers(0, w.Sq, 20))))
    for h in (0, w.H - 1):
        sel = lambda t: oracle.to_f64(t[0, :, h, :])
        rq, rk, rv = oracle.attention_backward_rows(sel(q), sel(k), sel(v), sel(dout), w.scale, w.causal, rows, rows)
        check("dq", dq[0, rows, h], rq, f"{w.name} head {h}")
        check("dk", dk[0, rows, h], rk, f"{w.name} head {h}")
        check("dv", dv[0, rows, h], rv, f"{w.name} head {h}")


def test_backward_long_d64_one_pass_sampled_rows():
    """The one-pass kernel at 32768 keys (B1 H2 S32768 d64 causal): every dQ
    row gathers reduce-adds from up to 256 key tiles.  dQ rows and dK, dV rows
    sampled across the sequence in both heads, against the oracle's per-row
    gradients; the tolerance's scale is the largest |value| among them."""
    need_gpu()
    w = C(1, 2, 32768, 32768, 64, True, seed=119)
    q, k, v = inputs.make_inputs(w)
    g = torch.Generator().manual_seed(w.seed + 2000)
    dout = torch.randn(q.shape, generator=g).to(torch.bfloat16)
    dq, dk, dv = grads(w, q, k, v, dout)
    rng = np.random.default_rng(6)
    fixed = [0, 1, 127, 128, 255, 256, 16383, 16384, w.Sq - 129, w.Sq - 128, w.Sq - 1]
    rows = np.array(sorted(set(fixed) | set(int(x) for x in rng.integers(0, w.Sq, 20))))
    for h in range(w.H):
        sel = lambda t: oracle.to_f64(t[0, :, h, :])
        rq, rk, rv = oracle.attention_backward_rows(sel(q), sel(k), sel(v), sel(dout), w.scale, w.causal, rows, rows)
        check("dq", dq[0, rows, h], rq, f"{w.name} head {h}")
        check("dk", dk[0, rows, h], rk, f"{w.name} head {h}")
        check("dv", dv[0, rows, h], rv, f"{w.name} head {h}")


@pytest.mark.parametrize("d", [64, 128])
def test_autograd_attention(d):
    """attn.attention through torch.autograd: o.backward(dO) leaves the
    oracle's gradients in q.grad, k.grad, v.grad (grouped heads, causal)."""
    need_gpu()
    w = C(2, 4, 333, 333, d, True, seed=120 + d, H_kv=2)
    q, k, v = inputs.make_inputs(w)
    g = torch.Generator().manual_seed(w.seed + 1000)
    dout = torch.randn(q.shape, generator=g).to(torch.bfloat16)
    qd, kd, vd = (t.cuda().requires_grad_() for t in (q, k, v))
    o, lse = attn.attention(qd, kd, vd, causal=True, scale=w.scale)
    o.backward(dout.cuda())
    torch.cuda.synchronize()
    assert attn.get_status() == 0
    rq, rk, rv = oracle.attention_backward(q, k, v, dout, w.scale, True)
    check("dq", qd.grad, rq, w.name)
    check("dk", kd.grad, rk, w.name)
    check("dv", vd.grad, rv, w.name)


@pytest.mark.parametrize("schedule", SCHEDULES)
@pytest.mark.parametrize("d,causal,hkv", [(64, False, 0), (128, True, 0), (64, True, 2), (128, False, 2)])
def test_backward_strided_inputs(d, causal, hkv, schedule):
    """q, k, v as slices of a packed QKV tensor (or q and a packed KV tensor
    with grouped heads), o written by the forward into a slice of a wider
    buffer: the gradients equal the oracle's on the dense tensors."""
    need_gpu()
    w = C(2, 4, 300, 300, d, causal, seed=130 + d + hkv, H_kv=hkv)
    q, k, v = inputs.make_inputs(w)
    if not w.H_kv:
        qkv = torch.stack([q, k, v], dim=2).cuda()  # [B, S, 3, H, d]
        qd, kd, vd = qkv[:, :, 0], qkv[:, :, 1], qkv[:, :, 2]
    else:
        qd = q.cuda()
        kv = torch.stack([k, v], dim=2).cuda()  # [B, S, 2, H_kv, d]
        kd, vd = kv[:, :, 0], kv[:, :, 1]
    assert not qd.is_contiguous() or not kd.is_contiguous()
    obuf = torch.empty((w.B, w.Sq, 2, w.H, d), dtype=torch.bfloat16, device="cuda")
    o = obuf[:, :, 1]
    o, lse = attn.attn_fwd(qd, kd, vd, causal=causal, scale=w.scale, out=o)
    g = torch.Generator().manual_seed(w.seed + 1000)
    dout = torch.randn(q.shape, generator=g).to(torch.bfloat16)
    dq, dk, dv = attn.attn_bwd(qd, kd, vd, o, lse, dout.cuda(), causal=causal, scale=w.scale,
                               deterministic=SCHEDULES[schedule])
    torch.cuda.synchronize()
    assert attn.get_status() == 0
    rq, rk, rv = oracle.attention_backward(q, k, v, dout, w.scale, causal)
    check("dq", dq, rq, w.name)
    check("dk", dk, rk, w.name)
    check("dv", dv, rv, w.name)
