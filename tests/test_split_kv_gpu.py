"""Split-KV on the kernel's own outputs: one problem's keys cut into ranges,
each range computed by the attention kernel, the partial (O_r, LSE_r) merged
by the library's host merge (the exchange step of the multi-GPU split-KV
plan), and the result compared with the unsplit oracle on every element.

This checks on one GPU what the multi-GPU split needs from the kernel: that
its LSE is the natural-log sum over exactly the visible keys of its range
(−inf for rows that see none), so that LSE = ln Σ_r exp(LSE_r) and
O = Σ_r exp(LSE_r − LSE)·O_r reproduce the whole problem.  Causal masks are
cut as the ranks would cut them: the first key range keeps top-left
alignment, a range ending at the last key is bottom-right aligned, and a
range that every row sees in full is not masked at all.
"""

import numpy as np
import pytest
import torch

import oracle
from exact_attention_63_gb300 import attn
from exact_attention_63_gb300 import dist as adist
from exact_attention_63_gb300 import inputs
from gpu_common import assert_close, need_gpu


def _partials(q, k, v, ranges, scale, mask_of):
    """Kernel outputs per key range: ranges [(a, b)], mask_of(i) -> (causal, align)."""
    os_, ls_ = [], []
    for i, (a, b) in enumerate(ranges):
        causal, align = mask_of(i)
        o, lse = attn.attn_fwd(q, k[:, a:b], v[:, a:b], causal=causal, scale=scale, causal_align=align)
        os_.append(o.float())
        ls_.append(lse)
    torch.cuda.synchronize()
    assert attn.get_status() == 0
    # merge per (b, h): O [R, B, Sq, H, d] -> [R, B, H, Sq, d] to line up with LSE [R, B, H, Sq]
    O = torch.stack(os_).permute(0, 1, 3, 2, 4).double()
    L = torch.stack(ls_).double()
    o_m, l_m = adist.merge_partials(O, L)
    return o_m.permute(0, 2, 1, 3).cpu().numpy(), l_m.cpu().numpy()


@pytest.mark.gpu
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("world", [2, 3])
def test_split_kv_non_causal(d, world):
    need_gpu()
    w = inputs.custom(2, 3, 700, 1000, d, False, sigma_qk=2.0, seed=90 + d + world)
    q, k, v = (t.cuda() for t in inputs.make_inputs(w))
    ranges = [adist.split_keys(w.Sk, world, r) for r in range(world)]
    assert ranges[0][0] == 0 and ranges[-1][1] == w.Sk
    o, lse = _partials(q, k, v, ranges, w.scale, lambda i: (False, "top-left"))
    O_ref, L_ref = oracle.attention_forward(*(t.cpu() for t in (q, k, v)), w.scale, False)
    assert_close(o, lse, O_ref, L_ref, f"split-KV x{world} d={d}")


@pytest.mark.gpu
@pytest.mark.parametrize("d", [64, 128])
def test_split_kv_causal_square(d):
    """Sq = Sk: keys [0, c) top-left causal (rows < c see a prefix, later rows
    all of it), keys [c, S) bottom-right (rows < c see none)."""
    need_gpu()
    w = inputs.custom(1, 4, 900, 900, d, True, seed=95 + d)
    q, k, v = (t.cuda() for t in inputs.make_inputs(w))
    ranges = [adist.split_keys(w.Sk, 2, r) for r in range(2)]
    o, lse = _partials(q, k, v, ranges, w.scale, lambda i: (True, "top-left" if i == 0 else "bottom-right"))
    O_ref, L_ref = oracle.attention_forward(*(t.cpu() for t in (q, k, v)), w.scale, True)
    assert_close(o, lse, O_ref, L_ref, f"split-KV causal d={d}")
    # rows before the second range's first key saw nothing there: the merge kept range 0 alone
    c = ranges[1][0]
    assert np.allclose(lse[:, :, :c], L_ref[:, :, :c], atol=1e-3)


@pytest.mark.gpu
def test_split_kv_causal_bottom_right_short_queries():
    """Sq < Sk, bottom-right (the last query row sees every key): the first
    half of the keys is visible to every row (no mask), the second half is
    bottom-right causal."""
    need_gpu()
    w = inputs.custom(2, 2, 300, 1000, 128, True, seed=97, causal_align="bottom-right")
    q, k, v = (t.cuda() for t in inputs.make_inputs(w))
    ranges = [(0, 512), (512, 1000)]
    assert ranges[0][1] - 1 <= 0 + w.Sk - w.Sq  # row 0 sees every key of range 0
    o, lse = _partials(q, k, v, ranges, w.scale,
                       lambda i: (False, "top-left") if i == 0 else (True, "bottom-right"))
    O_ref, L_ref = oracle.attention_forward(*(t.cpu() for t in (q, k, v)), w.scale, True,
                                            causal_offset=w.Sk - w.Sq)
    assert_close(o, lse, O_ref, L_ref, "split-KV bottom-right Sq<Sk")
