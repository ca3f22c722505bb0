"""Device status word: a pipeline wait that runs out reports ATTN_ERR_TIMEOUT
without faulting, and the context stays usable afterwards."""

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
