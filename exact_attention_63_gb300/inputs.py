"""Seeded synthetic inputs for the attention forward workloads.

This module only draws random numbers and names shapes: it holds none of the
attention arithmetic, and both the CUDA path's tests/bench and the CPU oracle
read the tensors it returns.

Recipe (the pages name no dataset; the workloads are synthetic):
  * a CPU ``torch.Generator`` seeded with the workload's seed;
  * three fp32 ``randn`` draws in the order Q, K, V, each shaped
    (batch, seq, heads, head_dim) — the layout of the pages' Python API call
    ("FlashAttention-3: Pipeline Assíncrono …", section "Implementando
    FlashAttention-3 em produção");
  * each multiplied by its standard deviation, then rounded to bf16 (RNE).
Both sides read exactly these bf16 values.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, asdict

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    Sq: int
    Sk: int
    d: int
    causal: bool
    sigma_qk: float = 1.0
    sigma_v: float = 1.0
    seed: int = 0
    H_kv: int = 0                  # key/value heads (grouped-query attention); 0 = H
    causal_align: str = "top-left"  # or "bottom-right" (key j visible to row i iff j <= i + Sk - Sq)

    @property
    def kv_heads(self) -> int:
        return self.H_kv or self.H

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    @property
    def flops(self) -> float:
        """Counted FLOPs: 4·B·H·Sq·Sk·d, halved when causal."""
        f = 4.0 * self.B * self.H * self.Sq * self.Sk * self.d
        return f / 2 if self.causal else f

    @property
    def io_bytes(self) -> int:
        """Algorithmic HBM bytes: Q, K, V read once, O written once (bf16), LSE (fp32)."""
        return 2 * self.d * self.B * (2 * self.H * self.Sq + 2 * self.kv_heads * self.Sk) + 4 * self.B * self.H * self.Sq

    def as_dict(self):
        d = asdict(self)
        d["scale"] = self.scale
        return d


# The five attention-forward workloads (B, H, Sq=Sk, head_dim, causal, σ).
WORKLOADS = {
    1: Workload("attn_fwd_b1_h2_s256_d64", 1, 2, 256, 256, 64, False, seed=1),
    2: Workload("attn_fwd_b4_h16_s2048_d128", 4, 16, 2048, 2048, 128, False, seed=2),
    3: Workload("attn_fwd_b2_h16_s8192_d128_causal", 2, 16, 8192, 8192, 128, True, seed=3),
    # Q and K drawn with standard deviation 3 ("peaky" logits), V with 1.
    4: Workload("attn_fwd_b8_h32_s4096_d64_peaky", 8, 32, 4096, 4096, 64, False, sigma_qk=3.0, seed=4),
    5: Workload("attn_fwd_b1_h16_s32768_d128_causal", 1, 16, 32768, 32768, 128, True, seed=5),
}


def make_inputs(w: Workload, seed: int | None = None, device=None):
    """Return bf16 (q, k, v) for workload ``w`` (CPU unless ``device`` given)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(w.seed if seed is None else seed)
    q = torch.randn((w.B, w.Sq, w.H, w.d), generator=g, dtype=torch.float32)
    k = torch.randn((w.B, w.Sk, w.kv_heads, w.d), generator=g, dtype=torch.float32)
    v = torch.randn((w.B, w.Sk, w.kv_heads, w.d), generator=g, dtype=torch.float32)
    if w.sigma_qk != 1.0:
        q.mul_(w.sigma_qk)
        k.mul_(w.sigma_qk)
    if w.sigma_v != 1.0:
        v.mul_(w.sigma_v)
    out = tuple(t.to(torch.bfloat16) for t in (q, k, v))
    if device is not None:
        out = tuple(t.to(device) for t in out)
    return out


def custom(B, H, Sq, Sk, d, causal, sigma_qk=1.0, sigma_v=1.0, seed=0, name=None, H_kv=0,
           causal_align="top-left") -> Workload:
    """A workload with explicit sizes (tests: ragged tails, edge cases)."""
    tag = (f"_hkv{H_kv}" if H_kv else "") + ("_causal" if causal else "") + \
        ("_br" if causal and causal_align == "bottom-right" else "")
    return Workload(name or f"attn_b{B}_h{H}_sq{Sq}_sk{Sk}_d{d}{tag}",
                    B, H, Sq, Sk, d, causal, sigma_qk, sigma_v, seed, H_kv, causal_align)


# ------------------------------------------------------- packed sequences
def varlen_lengths(n: int, max_len: int, seed: int) -> list[int]:
    """A seeded mix of n sequence lengths in [0, max_len]: mostly uniform,
    with the edge lengths of a 128-row tile mixed in (1, 127, 128, 129) and the
    longest one present."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    lens = torch.randint(1, max_len + 1, (n,), generator=g).tolist()
    edges = [1, 127, 128, 129, max_len]
    for i, e in enumerate(edges):
        if i < n and e <= max_len:
            lens[(i * 7) % n] = e
    return lens


def make_varlen_inputs(lens_q, lens_k, H: int, H_kv: int, d: int, seed: int, sigma_qk: float = 1.0, device=None):
    """bf16 q [total_q, H, d], k, v [total_k, H_kv, d] and int32 offset tables
    cu_q, cu_k ([n + 1], starting at 0) for sequences of the given lengths."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    tq, tk = int(sum(lens_q)), int(sum(lens_k))
    q = torch.randn((tq, H, d), generator=g, dtype=torch.float32) * sigma_qk
    k = torch.randn((tk, H_kv, d), generator=g, dtype=torch.float32) * sigma_qk
    v = torch.randn((tk, H_kv, d), generator=g, dtype=torch.float32)
    cu_q = torch.tensor([0] + list(torch.cumsum(torch.tensor(lens_q), 0).tolist()), dtype=torch.int32)
    cu_k = torch.tensor([0] + list(torch.cumsum(torch.tensor(lens_k), 0).tolist()), dtype=torch.int32)
    out = tuple(t.to(torch.bfloat16) for t in (q, k, v)) + (cu_q, cu_k)
    if device is not None:
        out = tuple(t.to(device) for t in out)
    return out


# ------------------------------------------------------------------- FP8
E4M3_MAX = 448.0  # largest finite FP8 E4M3 value


def make_fp8_inputs(w: Workload, seed: int | None = None, device=None):
    """FP8 (E4M3) q, k, v for workload ``w`` and their per-tensor scale factors.

    The same fp32 draws as ``make_inputs`` (seed, order Q, K, V, the
    workload's standard deviations), each tensor divided by its scale factor
    descale = max|x| / 448 and rounded to E4M3 (round to nearest even), so its
    largest magnitude lands on 448.  Returns (q8, k8, v8, descale_q, descale_k,
    descale_v) with the tensors as torch.float8_e4m3fn, shaped like the bf16
    inputs; the values they stand for are descale · x8.
    """
    g = torch.Generator(device="cpu")
    g.manual_seed(w.seed if seed is None else seed)
    q = torch.randn((w.B, w.Sq, w.H, w.d), generator=g, dtype=torch.float32)
    k = torch.randn((w.B, w.Sk, w.kv_heads, w.d), generator=g, dtype=torch.float32)
    v = torch.randn((w.B, w.Sk, w.kv_heads, w.d), generator=g, dtype=torch.float32)
    if w.sigma_qk != 1.0:
        q.mul_(w.sigma_qk)
        k.mul_(w.sigma_qk)
    if w.sigma_v != 1.0:
        v.mul_(w.sigma_v)
    out, scales = [], []
    for t in (q, k, v):
        descale = float(t.abs().max()) / E4M3_MAX
        out.append((t / descale).to(torch.float8_e4m3fn))
        scales.append(descale)
    if device is not None:
        out = [t.to(device) for t in out]
    return (*out, *scales)
