"""Plain, slow, obviously-correct exact attention forward in float64.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``): the product path never
imports this module.

What is computed (the definition, not the tiled algorithm):
  "FlashAttention-4 no Blackwell B200 …", section "Por que o Blackwell exige
  mais do que multiplicações rápidas": scaled attention is
  softmax(Q Kᵀ / √d) V.  The tiled/online method reaches exactly this result up
  to rounding ("FlashAttention-4 em Blackwell B200 …", FAQ question 2: the
  softmax is identical to the original attention), so the oracle is the
  definition written out, two-pass and non-online:

  for each batch b, head h and query row i
    s_ij   = scale · Σ_c q_ic k_jc                   (float64, over the exact
                                                      bf16 input values)
    V_i    = { j : 0 ≤ j < Sk and (not causal or j ≤ i) }
    M_i    = max_{j∈V_i} s_ij
    L_i    = Σ_{j∈V_i} exp(s_ij − M_i)
    P_ij   = exp(s_ij − M_i) / L_i  for j ∈ V_i, else 0
    O_i    = Σ_j P_ij v_j
    LSE_i  = M_i + ln L_i        (natural log-sum-exp of the scaled logits)

Readings where the pages are silent (each also listed in the design notes):
  * layout: Q, K, V, O are (batch, seq, heads, head_dim), the only layout the
    pages show ("FlashAttention-3: Pipeline Assíncrono …", section
    "Implementando FlashAttention-3 em produção"); LSE is (batch, heads, Sq).
  * causal: key j is visible to query i iff j ≤ i (top-left alignment).  The
    pages give no rule for Sq ≠ Sk; the other common one, bottom-right
    alignment (j ≤ i + Sk − Sq: the last query row sees every key), is the
    ``causal_offset = Sk − Sq`` case below.
  * grouped-query attention: "FlashAttention 4: Atenção Mais Rápida …",
    section "Compatibilidade e status atual", describes GQA as several query
    heads sharing one key/value projection.  With H query heads and H_kv key/
    value heads (H a multiple of H_kv), query head h reads key/value head
    h // (H / H_kv): consecutive query heads share one, H_kv = 1 being MQA.
  * a row with no visible key has O = 0 and LSE = −inf.
  * the scale is an argument; the pages pass 1/√head_dim.

Library primitives used as steps: numpy matmul (dgemm), exp, log, max, sum.
"""

from __future__ import annotations

import numpy as np

# Rows of Q processed per matmul, to bound memory (a chunk of scores is
# ROW_CHUNK × Sk float64 values).
ROW_CHUNK = 1024


def to_f64(x) -> np.ndarray:
    """Exact float64 copy of a bf16/fp32 torch tensor or array-like.

    bf16 → fp32 → fp64 is exact, so the oracle sees the same values as the GPU.
    """
    try:
        import torch  # local import: the oracle itself needs only numpy

        if isinstance(x, torch.Tensor):
            return x.detach().to("cpu", torch.float32).numpy().astype(np.float64)
    except ImportError:  # pragma: no cover
        pass
    return np.asarray(x, dtype=np.float64)


def visible_mask(rows: np.ndarray, Sk: int, causal: bool, causal_offset: int = 0) -> np.ndarray:
    """Boolean [len(rows), Sk]: True where key j is visible to query row i.

    Visible set: 0 ≤ j < Sk, and j ≤ i + causal_offset when causal (offset 0 =
    top-left alignment, Sk − Sq = bottom-right).
    """
    rows = np.asarray(rows, dtype=np.int64)
    keys = np.arange(Sk, dtype=np.int64)
    if not causal:
        return np.ones((rows.shape[0], Sk), dtype=bool)
    return keys[None, :] <= rows[:, None] + causal_offset


def head_scores(q: np.ndarray, k: np.ndarray, scale: float) -> np.ndarray:
    """s = scale · q kᵀ for one head. q: [n, d], k: [Sk, d], float64."""
    return scale * (q @ k.T)


def head_probabilities(s: np.ndarray, mask: np.ndarray):
    """Two-pass softmax of each row over its visible keys.

    Returns (P, M, L): P [n, Sk] with zeros outside the visible set,
    M [n] the row maximum over visible keys (−inf if none),
    L [n] = Σ_visible exp(s − M) (0 if none).
    """
    masked = np.where(mask, s, -np.inf)
    M = masked.max(axis=1)
    finite = np.isfinite(M)
    shift = np.where(finite, M, 0.0)
    E = np.where(mask, np.exp(masked - shift[:, None]), 0.0)
    L = E.sum(axis=1)
    with np.errstate(invalid="ignore", divide="ignore"):
        P = np.where(finite[:, None], E / np.where(finite, L, 1.0)[:, None], 0.0)
    return P, M, L


def attention_head(q, k, v, scale: float, causal: bool, rows=None, causal_offset: int = 0):
    """Exact attention for one head, float64.

    q: [Sq, d], k: [Sk, d], v: [Sk, d].  ``rows`` selects query rows (default
    all); causal masks see keys j ≤ i + causal_offset.  Returns (O [n, d],
    LSE [n]) for the selected rows.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    Sk = k.shape[0]
    rows = np.arange(q.shape[0]) if rows is None else np.asarray(rows, dtype=np.int64)
    O = np.zeros((rows.shape[0], v.shape[1]), dtype=np.float64)
    LSE = np.full((rows.shape[0],), -np.inf, dtype=np.float64)
    for c0 in range(0, rows.shape[0], ROW_CHUNK):
        r = rows[c0:c0 + ROW_CHUNK]
        # Causal rows never see keys beyond their own index (+ offset): only
        # the needed key prefix is multiplied (same result, less work).
        kmax = Sk if not causal else int(min(Sk, r.max() + 1 + causal_offset))
        if kmax <= 0:
            continue  # no row of the chunk sees a key: O = 0, LSE = −inf
        s = head_scores(q[r], k[:kmax], scale)
        P, M, L = head_probabilities(s, visible_mask(r, kmax, causal, causal_offset))
        O[c0:c0 + r.shape[0]] = P @ v[:kmax]
        with np.errstate(divide="ignore"):
            LSE[c0:c0 + r.shape[0]] = np.where(np.isfinite(M), M + np.log(np.where(L > 0, L, 1.0)), -np.inf)
    return O, LSE


def kv_head(h: int, H: int, H_kv: int) -> int:
    """Key/value head read by query head h (grouped-query attention)."""
    if H_kv < 1 or H % H_kv != 0:
        raise ValueError(f"H = {H} is not a multiple of H_kv = {H_kv}")
    return h // (H // H_kv)


def attention_forward(q, k, v, scale: float, causal: bool, causal_offset: int = 0):
    """Exact attention over all batches and heads.

    q: [B, Sq, H, d]; k, v: [B, Sk, H_kv, d] (torch tensors or arrays), H a
    multiple of H_kv.  Causal masks see keys j ≤ i + causal_offset.
    Returns O [B, Sq, H, d] float64 and LSE [B, H, Sq] float64.
    """
    q, k, v = to_f64(q), to_f64(k), to_f64(v)
    B, Sq, H, d = q.shape
    H_kv = k.shape[2]
    O = np.zeros((B, Sq, H, v.shape[3]), dtype=np.float64)
    LSE = np.zeros((B, H, Sq), dtype=np.float64)
    for b in range(B):
        for h in range(H):
            g = kv_head(h, H, H_kv)
            O[b, :, h, :], LSE[b, h, :] = attention_head(q[b, :, h, :], k[b, :, g, :], v[b, :, g, :], scale, causal,
                                                         causal_offset=causal_offset)
    return O, LSE


def attention_rows(q, k, v, scale: float, causal: bool, b: int, h: int, rows, causal_offset: int = 0):
    """Exact attention for selected query rows of one (batch, head).

    Used to check full-size GPU outputs on a sample of rows; K/V may have fewer
    heads than Q (grouped-query attention).  Returns (O [n, d], LSE [n]) float64.
    """
    g = kv_head(h, q.shape[2], k.shape[2])
    qh = to_f64(q[b, :, h, :]) if not isinstance(q, np.ndarray) else q[b, :, h, :]
    kh = to_f64(k[b, :, g, :]) if not isinstance(k, np.ndarray) else k[b, :, g, :]
    vh = to_f64(v[b, :, g, :]) if not isinstance(v, np.ndarray) else v[b, :, g, :]
    return attention_head(qh, kh, vh, scale, causal, rows=rows, causal_offset=causal_offset)


def attention_varlen(q, k, v, cu_q, cu_k, scale: float, causal: bool, bottom_right: bool = False):
    """Exact attention over a batch of sequences of different lengths packed
    along the row dimension (the "varlen" layout).

    q: [total_q, H, d]; k, v: [total_k, H_kv, d]; cu_q, cu_k: [n + 1]
    ascending row offsets (cu[0] = 0): sequence s owns query rows
    [cu_q[s], cu_q[s+1]) and key rows [cu_k[s], cu_k[s+1]), and attends only to
    its own keys.  Causal masks align per sequence: top-left (j ≤ i) or, with
    ``bottom_right``, j ≤ i + len_k − len_q.  Rows that see no key get O = 0,
    LSE = −inf.  Returns O [total_q, H, d] and LSE [H, total_q] (float64).
    """
    q, k, v = to_f64(q), to_f64(k), to_f64(v)
    cu_q = [int(x) for x in np.asarray(cu_q)]
    cu_k = [int(x) for x in np.asarray(cu_k)]
    total_q, H, d = q.shape
    H_kv = k.shape[1]
    O = np.zeros((total_q, H, v.shape[2]), dtype=np.float64)
    LSE = np.full((H, total_q), -np.inf, dtype=np.float64)
    for s in range(len(cu_q) - 1):
        q0, q1, k0, k1 = cu_q[s], cu_q[s + 1], cu_k[s], cu_k[s + 1]
        if q1 <= q0:
            continue
        off = (k1 - k0) - (q1 - q0) if (causal and bottom_right) else 0
        for h in range(H):
            g = kv_head(h, H, H_kv)
            if k1 <= k0:
                continue  # no keys: O = 0, LSE = −inf
            O[q0:q1, h, :], LSE[h, q0:q1] = attention_head(q[q0:q1, h, :], k[k0:k1, g, :], v[k0:k1, g, :], scale,
                                                           causal, causal_offset=off)
    return O, LSE


def attention_backward_head(q, k, v, dO, scale: float, causal: bool, causal_offset: int = 0):
    """Gradients of one head's attention output with respect to q, k and v.

    The pages give no backward formulas ("FlashAttention-4 no Blackwell B200
    …", section "Redução de tráfego no backward", only says where FA4 keeps its
    intermediates), so this is the derivative of the definition above, written
    out in float64 for a loss whose gradient with respect to O is dO (the LSE
    output is not differentiated):
      P = softmax over visible keys of s,  dV = Pᵀ dO,  dP = dO Vᵀ,
      D_i = Σ_c dO_ic O_ic = Σ_j P_ij dP_ij,  dS = P ∘ (dP − D),
      dQ = scale · dS K,  dK = scale · dSᵀ Q.
    Rows without visible keys contribute nothing.  q, dO: [Sq, d]; k, v:
    [Sk, d].  Returns (dQ [Sq, d], dK [Sk, d], dV [Sk, d], D [Sq]).
    """
    q, k, v, dO = (np.asarray(x, dtype=np.float64) for x in (q, k, v, dO))
    s = head_scores(q, k, scale)
    P, M, L = head_probabilities(s, visible_mask(np.arange(q.shape[0]), k.shape[0], causal, causal_offset))
    O = P @ v
    dV = P.T @ dO
    dP = dO @ v.T
    D = (dO * O).sum(axis=1)
    dS = P * (dP - D[:, None])
    return scale * (dS @ k), scale * (dS.T @ q), dV, D


def attention_backward_rows(q, k, v, dO, scale: float, causal: bool, qrows, krows, causal_offset: int = 0):
    """Selected rows of one head's gradients, without the whole Sq×Sk matrices.

    The same formulas as attention_backward_head, evaluated for query rows
    ``qrows`` (rows of dQ) and key rows ``krows`` (rows of dK and dV): a query
    row's dQ needs only its own scores, P_ij = exp(s_ij − LSE_i),
    dP_ij = dO_i · v_j and D_i = dO_i · O_i; a key row's dK and dV sum over
    every query row, taken in chunks of ROW_CHUNK rows.  O and LSE come from
    attention_head.  Returns (dQ [len(qrows), d], dK [len(krows), d],
    dV [len(krows), d]).
    """
    q, k, v, dO = (np.asarray(x, dtype=np.float64) for x in (q, k, v, dO))
    qrows = np.asarray(qrows, dtype=np.int64)
    krows = np.asarray(krows, dtype=np.int64)
    Sq, Sk = q.shape[0], k.shape[0]
    O, LSE = attention_head(q, k, v, scale, causal, causal_offset=causal_offset)
    D = (dO * O).sum(axis=1)

    def probs(rows, keys):
        s = head_scores(q[rows], k[keys], scale)
        mask = visible_mask(rows, Sk, causal, causal_offset)[:, keys]
        finite = np.isfinite(LSE[rows])
        with np.errstate(invalid="ignore"):
            P = np.where(mask & finite[:, None], np.exp(s - np.where(finite, LSE[rows], 0.0)[:, None]), 0.0)
        return P

    P = probs(qrows, np.arange(Sk))
    dS = P * (dO[qrows] @ v.T - D[qrows][:, None])
    dQ = scale * (dS @ k)
    dK = np.zeros((krows.shape[0], k.shape[1]))
    dV = np.zeros((krows.shape[0], v.shape[1]))
    for c0 in range(0, Sq, ROW_CHUNK):
        rows = np.arange(c0, min(Sq, c0 + ROW_CHUNK))
        P = probs(rows, krows)
        dS = P * (dO[rows] @ v[krows].T - D[rows][:, None])
        dV += P.T @ dO[rows]
        dK += scale * (dS.T @ q[rows])
    return dQ, dK, dV


def attention_backward(q, k, v, dO, scale: float, causal: bool, causal_offset: int = 0):
    """Gradients over all batches and heads: q, dO [B, Sq, H, d], k, v
    [B, Sk, H_kv, d] (torch tensors or arrays; H a multiple of H_kv).  A
    key/value head shared by a group of query heads gets the sum of their
    gradients.  Returns dQ, dK, dV (float64, the shapes of q, k, v)."""
    q, k, v, dO = to_f64(q), to_f64(k), to_f64(v), to_f64(dO)
    B, Sq, H, d = q.shape
    H_kv = k.shape[2]
    dQ, dK, dV = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    for b in range(B):
        for h in range(H):
            g = kv_head(h, H, H_kv)
            dq, dk, dv, _ = attention_backward_head(q[b, :, h], k[b, :, g], v[b, :, g], dO[b, :, h], scale, causal,
                                                    causal_offset)
            dQ[b, :, h] = dq
            dK[b, :, g] += dk
            dV[b, :, g] += dv
    return dQ, dK, dV


def combine_partials(O_parts, LSE_parts):
    """Merge attention results computed over disjoint key ranges.

    Each part r holds (O_r, LSE_r) of the same query rows over its own key
    subset.  Since exp(LSE_r) is that subset's share of the softmax
    denominator, the full result is LSE = ln Σ_r exp(LSE_r) and
    O = Σ_r exp(LSE_r − LSE) · O_r.  Parts with LSE_r = −inf (no visible key)
    contribute nothing.  Inputs: lists of arrays [..., n, d] and [..., n].
    """
    L = np.stack([np.asarray(x, dtype=np.float64) for x in LSE_parts])
    Os = np.stack([np.asarray(x, dtype=np.float64) for x in O_parts])
    M = L.max(axis=0)
    finite = np.isfinite(M)
    shift = np.where(finite, M, 0.0)
    W = np.where(np.isfinite(L), np.exp(L - shift[None]), 0.0)
    tot = W.sum(axis=0)
    with np.errstate(divide="ignore", invalid="ignore"):
        LSE = np.where(finite, shift + np.log(np.where(tot > 0, tot, 1.0)), -np.inf)
        w = np.where(finite[None], W / np.where(tot > 0, tot, 1.0)[None], 0.0)
    O = (w[..., None] * Os).sum(axis=0)
    return O, LSE


def e4m3_to_f64(x8) -> np.ndarray:
    """Exact float64 values of FP8 E4M3 data (a torch float8_e4m3fn tensor, or
    its raw bytes as uint8)."""
    import torch  # local import, as in to_f64

    if isinstance(x8, torch.Tensor) and x8.dtype == torch.uint8:
        x8 = x8.view(torch.float8_e4m3fn)
    return x8.detach().to("cpu", torch.float32).numpy().astype(np.float64)


def attention_forward_fp8(q8, k8, v8, descale_q: float, descale_k: float, descale_v: float, scale: float,
                          causal: bool, causal_offset: int = 0):
    """Exact attention over FP8 (E4M3) inputs with per-tensor scale factors.

    "FlashAttention-3: Pipeline Assíncrono …", section "Estabilidade em FP8":
    the FP8 forward keeps Q, K and V in E4M3 (1 sign, 4 exponent, 3 mantissa
    bits, range ±448), accumulates the products in fp32 and applies static
    scale factors.  The values these tensors stand for are x = descale_x · x8
    (one factor per tensor, the reading adopted for "static scale factors"),
    so the exact result is the plain definition over the dequantized values:
      s_ij = scale · Σ_c (descale_q q8_ic)(descale_k k8_jc),
      O_i  = Σ_j softmax_j(s_ij) · descale_v v8_j,  LSE_i = ln Σ_j exp(s_ij).
    The two passes of the method (exact row maximum, then exponentials and
    P·V with P in FP8) are how a kernel reaches this result; the rounding of
    P to E4M3 is the kernel's error, bounded by the tests.
    """
    q = e4m3_to_f64(q8) * float(descale_q)
    k = e4m3_to_f64(k8) * float(descale_k)
    v = e4m3_to_f64(v8) * float(descale_v)
    return attention_forward(q, k, v, scale, causal, causal_offset)
