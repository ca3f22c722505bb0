"""Fit the cubic used by the kernels' FMA-pipe exp2.

The softmax computes 2^x for x ≤ τ.  Writing x = j + f with j = ⌊x⌋ and
f ∈ [0, 1), 2^x = 2^j · 2^f; 2^j is added straight into the float's exponent
field and 2^f is approximated by a cubic p(f) = 1 + c1 f + c2 f² + c3 f³
("FlashAttention 4: Atenção Mais Rápida …", section "Exponenciais de Software
via Núcleos CUDA": a cubic polynomial evaluated on the FMA units instead of
the special-function units; the pages give no coefficients, so they are
fitted here).

The constant term is pinned to exactly 1 so that p(0) = 1: then an input
clamped at −127 produces the bit pattern of +0.0 exactly, and p(f) ≥ 1 on
[0, 1) keeps the exponent field from underflowing into the sign bit.

The remaining coefficients minimise the maximum relative error
max_f |p(f) / 2^f − 1| over a dense grid — a linear program (minimax fit),
solved with scipy's HiGHS.  The coefficients are then rounded to float32 and
the error of float32 Horner evaluation is reported.  Run:

    python fit_exp2_poly.py

and copy the printed constants into attn_device.cuh (kPolyC1..kPolyC3).
"""

import numpy as np
from scipy.optimize import linprog


def fit(n=4097):
    f = np.linspace(0.0, 1.0, n)
    t = np.exp2(f)
    # variables: c1, c2, c3, e ; minimise e
    # |(1 + c1 f + c2 f^2 + c3 f^3) / t - 1| <= e
    A = np.stack([f / t, f**2 / t, f**3 / t], axis=1)
    b = 1.0 - 1.0 / t
    ones = np.ones((n, 1))
    A_ub = np.vstack([np.hstack([A, -ones]), np.hstack([-A, -ones])])
    b_ub = np.concatenate([b, -b])
    res = linprog(c=[0, 0, 0, 1], A_ub=A_ub, b_ub=b_ub, bounds=[(None, None)] * 4, method="highs")
    assert res.success, res.message
    return res.x[:3], res.x[3]


def horner_f32(c, f):
    f = f.astype(np.float32)
    c1, c2, c3 = (np.float32(x) for x in c)
    p = np.float32(c3) * f + c2
    p = p * f + c1
    p = p * f + np.float32(1.0)
    return p


if __name__ == "__main__":
    c, e = fit()
    c32 = [np.float32(x) for x in c]
    f = np.linspace(0.0, 1.0, 1 << 20, endpoint=False)
    rel = np.abs(horner_f32(c32, f).astype(np.float64) / np.exp2(f) - 1.0)
    print(f"fp64 minimax max rel err: {e:.3e}")
    print(f"fp32 Horner max rel err:  {rel.max():.3e}")
    print(f"p(1-) = {horner_f32(c32, np.array([np.nextafter(1, 0)]))[0]!r}")
    for i, x in enumerate(c32, 1):
        print(f"kPolyC{i} = {float(x)!r}f  // 0x{np.array(x).view(np.uint32):08x}")
