"""Device status word: a pipeline wait that runs out reports ATTN_ERR_TIMEOUT
without faulting, and the context stays usable afterwards."""

import numpy as np
import pytest
import torch

import oracle
from exact_attention_63_gb300 import attn, inputs
from gpu_common import assert_close, need_gpu

pytestmark = pytest.mark.gpu


def test_wait_limit_reports_timeout_and_context_survives():
    need_gpu()
    w = inputs.custom(1, 2, 256, 256, 64, False, seed=51)
    q, k, v = (t.cuda() for t in inputs.make_inputs(w))
    assert attn.get_status() == 0
    opts = attn.make_options(timeout_ms=50, test_flags=attn.TEST_WITHHOLD_KV)
    attn.attn_fwd(q, k, v, causal=False, scale=w.scale, options=opts)
    assert attn.get_status() == -8          # ATTN_ERR_TIMEOUT, read and cleared
    assert attn.get_status() == 0           # cleared
    o, lse = attn.attn_fwd(q, k, v, causal=False, scale=w.scale)
    torch.cuda.synchronize()
    assert attn.get_status() == 0
    O_ref, L_ref = oracle.attention_forward(q.cpu(), k.cpu(), v.cpu(), w.scale, False)
    assert_close(o, lse, O_ref, L_ref, "after timeout")


@pytest.mark.parametrize("flags", [0, attn.TEST_FALLBACK_KERNEL], ids=["full_row", "fallback"])
def test_fp8_wait_limit_reports_timeout_and_context_survives(flags):
    """Both FP8 kernels: a wait that runs out sets ATTN_ERR_TIMEOUT without a
    fault, and the next call computes correctly."""
    need_gpu()
    w = inputs.custom(1, 2, 300, 300, 128, True, seed=52)
    q8, k8, v8, dq, dk, dv = inputs.make_fp8_inputs(w)
    q8, k8, v8 = q8.cuda(), k8.cuda(), v8.cuda()
    assert attn.get_status() == 0
    opts = attn.make_options(timeout_ms=50, test_flags=attn.TEST_WITHHOLD_KV | flags)
    attn.attn_fwd_fp8(q8, k8, v8, dq, dk, dv, causal=True, scale=w.scale, options=opts)
    assert attn.get_status() == -8
    assert attn.get_status() == 0
    o, lse = attn.attn_fwd_fp8(q8, k8, v8, dq, dk, dv, causal=True, scale=w.scale,
                               options=attn.make_options(test_flags=flags))
    torch.cuda.synchronize()
    assert attn.get_status() == 0
    O_ref, L_ref = oracle.attention_forward_fp8(q8.cpu(), k8.cpu(), v8.cpu(), dq, dk, dv, w.scale, True)
    assert np.abs(lse.cpu().numpy().astype(np.float64) - L_ref).max() <= 1e-3
