"""Exact attention forward for GB300 (sm_103a).

O = softmax(Q Kᵀ · scale) V, optionally causal, computed tile by tile with an
online softmax so the S×S score matrix never reaches HBM; emits O (bf16) and
the per-row log-sum-exp (fp32).  The work runs in hand-written CUDA kernels
behind a C ABI (``include/attn_gb300.h``); ``attn.py`` is a thin ctypes
binding that passes device pointers and the current CUDA stream.

Importing this package loads nothing native; the shared library is loaded on
first use and a missing library raises immediately (there is no fallback).
"""

__all__ = ["attn", "inputs"]
