"""attn_fwd_host_static: the host-buffer call for callers that cannot allocate
device memory (for example a plugin whose framework owns all device memory
through its own allocator, or a code path where allocating after start-up is
forbidden because cudaMalloc may synchronise the device).  The library stages
the data in its own fixed 32 MiB device array instead of a caller workspace.

Both entry points run the same copies and the same kernel, so its results
must equal the existing host-buffer entry point's (which uses a
caller-allocated workspace) bit for bit, call after call, whether this file
runs alone in a fresh process or after the other tests; and once the first
call on the device has reserved the array, further calls must not change the
device's free memory or the allocator's counts.  This file is named so that
pytest collects it last.
"""

import ctypes

import pytest
import torch

from exact_attention_63_gb300 import attn, inputs
import oracle
from gpu_common import assert_close, need_gpu


def _host(w):
    q, k, v = inputs.make_inputs(w)
    qh, kh, vh = (t.pin_memory() for t in (q, k, v))
    oh = torch.empty_like(qh).pin_memory()
    lh = torch.empty((w.B, w.H, w.Sq), dtype=torch.float32).pin_memory()
    return qh, kh, vh, oh, lh


def _call_static(w, qh, kh, vh, oh, lh):
    # Straight through the C ABI with ctypes (no Python-side wrapper).
    L = attn.lib()
    return L.attn_fwd_host_static(qh.data_ptr(), kh.data_ptr(), vh.data_ptr(), oh.data_ptr(), lh.data_ptr(),
                                  w.B, w.H, w.Sq, w.Sk, w.d, ctypes.c_float(w.scale), int(w.causal),
                                  ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


@pytest.mark.gpu
def test_static_entry_matches_workspace_entry_on_consecutive_calls():
    need_gpu()
    cases = [inputs.custom(2, 3, 700, 650, 128, True, seed=71),
             inputs.custom(1, 4, 1000, 1000, 64, False, sigma_qk=3.0, seed=72),
             inputs.custom(2, 3, 700, 650, 128, True, seed=73)]
    for w in cases:  # consecutive calls share (and overwrite) the static array
        assert attn.workspace_size(w.B, w.H, w.Sq, w.Sk, w.d) <= attn.STATIC_WORKSPACE_BYTES
        qh, kh, vh, oh, lh = _host(w)
        assert _call_static(w, qh, kh, vh, oh, lh) == 0
        torch.cuda.current_stream().synchronize()
        assert attn.get_status() == 0

        o_ref = torch.empty_like(oh).pin_memory()
        l_ref = torch.empty_like(lh).pin_memory()
        ws = torch.empty(attn.workspace_size(w.B, w.H, w.Sq, w.Sk, w.d), dtype=torch.uint8, device="cuda")
        attn.attn_fwd_host(qh, kh, vh, o_ref, l_ref, w.causal, w.scale, ws)
        torch.cuda.current_stream().synchronize()
        assert torch.equal(oh, o_ref), f"static vs workspace {w.name}: O differs"
        assert torch.equal(lh, l_ref), f"static vs workspace {w.name}: LSE differs"
        # and both within the parity bar of the oracle
        O_ref, L_ref = oracle.attention_forward(qh, kh, vh, w.scale, w.causal)
        assert_close(oh, lh, O_ref, L_ref, f"static {w.name}")


@pytest.mark.gpu
def test_static_entry_allocates_nothing_after_its_first_call():
    need_gpu()
    w = inputs.custom(1, 4, 1000, 1000, 64, False, sigma_qk=3.0, seed=74)
    qh, kh, vh, oh, lh = _host(w)
    assert _call_static(w, qh, kh, vh, oh, lh) == 0  # the first call may load the module (reserves the array)
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    stats0 = torch.cuda.memory_stats()
    for _ in range(5):
        assert _call_static(w, qh, kh, vh, oh, lh) == 0
    torch.cuda.synchronize()
    assert attn.get_status() == 0
    free1, _ = torch.cuda.mem_get_info()
    stats1 = torch.cuda.memory_stats()
    assert free1 == free0, f"device free memory moved by {free0 - free1} bytes"
    for key in ("allocation.all.allocated", "segment.all.allocated"):
        assert stats1.get(key, 0) == stats0.get(key, 0), key


@pytest.mark.gpu
def test_static_entry_rejects_problems_above_its_limit():
    need_gpu()
    w = inputs.custom(1, 16, 4096, 4096, 128, False)  # needs ~64 MiB > 32 MiB
    assert attn.workspace_size(w.B, w.H, w.Sq, w.Sk, w.d) > attn.STATIC_WORKSPACE_BYTES
    t = torch.zeros(16, dtype=torch.bfloat16).pin_memory()  # never touched: rejected first
    L = attn.lib()
    rc = L.attn_fwd_host_static(t.data_ptr(), t.data_ptr(), t.data_ptr(), t.data_ptr(), t.data_ptr(),
                                w.B, w.H, w.Sq, w.Sk, w.d, ctypes.c_float(w.scale), 0, None)
    assert rc == -11
