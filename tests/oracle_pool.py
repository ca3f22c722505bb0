"""The oracle's per-head attention over a pool of spawned CPU processes, so
that full-size workloads can be checked on every element in seconds.

Test infrastructure: the workers import numpy and the oracle only, and are
started with `spawn` (a pool forked after CUDA has been used can hang)."""

from __future__ import annotations

import multiprocessing as mp
import os

import numpy as np

from oracle import attention as A


def _head(job):
    q, k, v, scale, causal = job
    return A.attention_head(q.astype(np.float64), k.astype(np.float64), v.astype(np.float64), scale, causal)


def attention_forward_pool(q, k, v, scale: float, causal: bool, workers: int | None = None):
    """q, k, v: CPU bf16 tensors [B, S, H, d] with one K/V head per query head.
    Returns O [B, Sq, H, d] and LSE [B, H, Sq] in float64 (the oracle's
    attention_head for every (b, h); bf16 → float32 is exact)."""
    qf, kf, vf = (t.float().numpy() for t in (q, k, v))
    B, Sq, H, d = qf.shape
    jobs = [(np.ascontiguousarray(qf[b, :, h]), np.ascontiguousarray(kf[b, :, h]), np.ascontiguousarray(vf[b, :, h]),
             scale, causal) for b in range(B) for h in range(H)]
    n = workers or min(16, os.cpu_count() or 1)
    with mp.get_context("spawn").Pool(n) as pool:
        res = pool.map(_head, jobs, chunksize=1)
    O = np.empty((B, Sq, H, d))
    L = np.empty((B, H, Sq))
    for i, (o, lse) in enumerate(res):
        b, h = divmod(i, H)
        O[b, :, h] = o
        L[b, h] = lse
    return O, L


def _bwd_head(job):
    q, k, v, g, scale, causal = job
    dq, dk, dv, _ = A.attention_backward_head(q, k, v, g, scale, causal)
    return dq, dk, dv


def attention_backward_pool(q, k, v, dout, scale: float, causal: bool, workers: int | None = None):
    """The oracle's gradients (attention_backward_head) for every (b, h), one
    per process; q, k, v, dout: CPU bf16 tensors [B, S, H, d] with one K/V
    head per query head.  Returns dQ, dK, dV in float64."""
    qf, kf, vf, gf = (t.float().numpy() for t in (q, k, v, dout))
    B, Sq, H, d = qf.shape
    jobs = [tuple(np.ascontiguousarray(x[b, :, h]) for x in (qf, kf, vf, gf)) + (scale, causal)
            for b in range(B) for h in range(H)]
    n = workers or min(16, os.cpu_count() or 1)
    with mp.get_context("spawn").Pool(n) as pool:
        res = pool.map(_bwd_head, jobs, chunksize=1)
    dQ, dK, dV = np.empty(qf.shape), np.empty(kf.shape), np.empty(vf.shape)
    for i, (dq, dk, dv) in enumerate(res):
        b, h = divmod(i, H)
        dQ[b, :, h], dK[b, :, h], dV[b, :, h] = dq, dk, dv
    return dQ, dK, dV
