"""Sequences of different lengths packed along the rows (attn_fwd_varlen),
GPU path vs the CPU oracle element by element."""

from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from exact_attention_63_gb300 import attn, inputs
from gpu_common import assert_close, f64, need_gpu

pytestmark = pytest.mark.gpu

# (name, lens_q, lens_k, H, H_kv, d, causal, causal_align, seed)
CASES = [
    ("equal_d128", [1, 127, 128, 129, 300, 64, 1000], None, 4, 2, 128, False, "top-left", 81),
    ("equal_causal_d128", [1, 127, 128, 129, 300, 64, 1000], None, 4, 2, 128, True, "top-left", 82),
    ("equal_causal_d64_mqa", [200, 5, 513, 256, 33], None, 4, 1, 64, True, "top-left", 83),
    ("unequal_d64", [5, 200, 130, 64, 0, 300], [300, 100, 130, 0, 50, 700], 2, 2, 64, False, "top-left", 84),
    ("unequal_causal_tl", [5, 200, 130, 64, 0, 300], [300, 100, 130, 0, 50, 700], 2, 2, 128, True, "top-left", 85),
    ("unequal_causal_br", [5, 200, 130, 64, 0, 300], [300, 100, 130, 0, 50, 700], 4, 2, 64, True, "bottom-right",
     86),
    ("one_sequence", [777], [777], 2, 2, 128, True, "top-left", 87),
    ("mix_d128", inputs.varlen_lengths(12, 700, 88), None, 8, 2, 128, True, "bottom-right", 88),
    # non-causal, many sequences: the compacted tile order (300 sequences,
    # several tiles per CTA) and, past its table's capacity of 4095
    # sequences, the padded order
    ("many_d64", [(i * 37) % 401 for i in range(300)], None, 2, 1, 64, False, "top-left", 92),
    ("beyond_table_d64", [(i * 7) % 13 for i in range(4100)], None, 2, 2, 64, False, "top-left", 93),
]


def run_case(lens_q, lens_k, H, H_kv, d, causal, align, seed, sigma=1.0, options=None):
    lens_k = lens_q if lens_k is None else lens_k
    q, k, v, cu_q, cu_k = inputs.make_varlen_inputs(lens_q, lens_k, H, H_kv, d, seed, sigma_qk=sigma)
    dev = torch.device("cuda:0")
    o, lse = attn.attn_fwd_varlen(q.to(dev), k.to(dev), v.to(dev), cu_q.to(dev), cu_k.to(dev),
                                  max(max(lens_q), 1), causal=causal, causal_align=align, options=options)
    torch.cuda.synchronize()
    assert attn.get_status() == 0
    O_ref, L_ref = oracle.attention_varlen(q, k, v, cu_q.numpy(), cu_k.numpy(), 1.0 / np.sqrt(d), causal,
                                           bottom_right=(align == "bottom-right"))
    return o, lse, O_ref, L_ref


def check(o, lse, O_ref, L_ref, what):
    """Rows without keys: exactly O = 0 and LSE = −inf; the rest within the bar."""
    o64, l64 = f64(o), f64(lse)                     # [T, H, d], [H, T]
    unseen = ~np.isfinite(L_ref)                   # [H, T]
    assert np.array_equal(unseen, np.isneginf(l64)), f"{what}: LSE −inf pattern differs"
    ot = np.transpose(o64, (1, 0, 2))              # [H, T, d]
    if unseen.any():
        assert np.all(ot[unseen] == 0.0), f"{what}: rows without keys are not zero"
    seen = ~unseen
    assert_close(ot[seen], l64[seen], np.transpose(O_ref, (1, 0, 2))[seen], L_ref[seen], what)


@pytest.mark.parametrize("case", CASES, ids=lambda c: c[0])
def test_varlen_cases(case):
    need_gpu()
    name, lens_q, lens_k, H, H_kv, d, causal, align, seed = case
    o, lse, O_ref, L_ref = run_case(lens_q, lens_k, H, H_kv, d, causal, align, seed)
    check(o, lse, O_ref, L_ref, name)


@pytest.mark.parametrize("case", [c for c in CASES if c[5] == 64 and len(c[1]) <= 300], ids=lambda c: c[0])
def test_varlen_d64_fallback_kernel(case):
    """Packed sequences at d = 64 through the full-row kernel's fallback
    (ATTN_TEST_FALLBACK_KERNEL): the same results."""
    need_gpu()
    name, lens_q, lens_k, H, H_kv, d, causal, align, seed = case
    opts = attn.make_options(test_flags=attn.TEST_FALLBACK_KERNEL)
    o, lse, O_ref, L_ref = run_case(lens_q, lens_k, H, H_kv, d, causal, align, seed, options=opts)
    check(o, lse, O_ref, L_ref, name + " (fallback kernel)")


def test_varlen_peaky_logits():
    """Q, K with standard deviation 3: rescaling inside packed sequences."""
    need_gpu()
    o, lse, O_ref, L_ref = run_case([640, 129, 1000], None, 2, 2, 64, False, "top-left", 89, sigma=3.0)
    check(o, lse, O_ref, L_ref, "peaky")


def test_varlen_matches_batched_call():
    """Equal lengths: the packed call returns what the batched call returns,
    bit for bit (same tiles, same arithmetic)."""
    need_gpu()
    B, S, H, d = 3, 700, 4, 128
    q, k, v, cu_q, cu_k = inputs.make_varlen_inputs([S] * B, [S] * B, H, H, d, 90, device="cuda")
    o1, l1 = attn.attn_fwd_varlen(q, k, v, cu_q, cu_k, S, causal=True)
    o2, l2 = attn.attn_fwd(q.view(B, S, H, d), k.view(B, S, H, d), v.view(B, S, H, d), causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o1.view(B, S, H, d), o2)
    assert torch.equal(l1, l2.permute(1, 0, 2).reshape(H, B * S))


def test_varlen_writes_only_its_rows():
    """Guard regions around O and LSE keep their sentinel values."""
    need_gpu()
    lens = [3, 130, 1, 257]
    H, d = 2, 64
    q, k, v, cu_q, cu_k = inputs.make_varlen_inputs(lens, lens, H, H, d, 91, device="cuda")
    T, G = q.shape[0], 4096
    o_buf = torch.full((T * H * d + 2 * G,), float("nan"), dtype=torch.bfloat16, device="cuda")
    l_buf = torch.full((H * T + 2 * G,), 12345.0, dtype=torch.float32, device="cuda")
    o = o_buf[G:G + T * H * d].view(T, H, d)
    lse = l_buf[G:G + H * T].view(H, T)
    attn.attn_fwd_varlen(q, k, v, cu_q, cu_k, max(lens), causal=True, out=o, lse=lse)
    torch.cuda.synchronize()
    assert torch.isnan(o_buf[:G]).all() and torch.isnan(o_buf[G + T * H * d:]).all()
    assert (l_buf[:G] == 12345.0).all() and (l_buf[G + H * T:] == 12345.0).all()
    assert bool(torch.isfinite(o).all()) and bool(torch.isfinite(lse).all())


@pytest.mark.parametrize("causal", [False, True])
def test_varlen_rows_beyond_max_seqlen_not_written(causal):
    """max_seqlen_q shorter than a sequence: that sequence's rows from
    max_seqlen_q on are left untouched (both tile orders), the rest is exact."""
    need_gpu()
    lens = [300, 700, 90]
    H, d, m = 2, 64, 384  # 384 = three q tiles; the 700-row sequence is cut there
    q, k, v, cu_q, cu_k = inputs.make_varlen_inputs(lens, lens, H, H, d, 94)
    dev = torch.device("cuda:0")
    o = torch.full(q.shape, float("nan"), dtype=torch.bfloat16, device=dev)
    lse = torch.full((H, q.shape[0]), 777.0, dtype=torch.float32, device=dev)
    attn.attn_fwd_varlen(q.to(dev), k.to(dev), v.to(dev), cu_q.to(dev), cu_k.to(dev), m, causal=causal,
                         out=o, lse=lse)
    torch.cuda.synchronize()
    O_ref, L_ref = oracle.attention_varlen(q, k, v, cu_q.numpy(), cu_k.numpy(), 1.0 / np.sqrt(d), causal)
    start = int(cu_q[1])
    cut = np.zeros(q.shape[0], dtype=bool)
    cut[start + m:start + lens[1]] = True
    o_c, l_c = o.cpu(), lse.cpu()
    assert torch.isnan(o_c[torch.from_numpy(cut)]).all()
    assert (l_c[:, torch.from_numpy(cut)] == 777.0).all()
    keep = ~cut
    check(o_c[torch.from_numpy(keep)], l_c[:, torch.from_numpy(keep)], O_ref[keep], L_ref[:, keep], "cut")


def test_varlen_bench_mix_full_size_all_elements():
    """The bench's packed workload `--config 2 --varlen 32` (32 sequences of up
    to 2048 rows, H16, d128) at full size, every element."""
    need_gpu()
    lens = inputs.varlen_lengths(32, 2048, inputs.WORKLOADS[2].seed)
    o, lse, O_ref, L_ref = run_case(lens, None, 16, 16, 128, False, "top-left", inputs.WORKLOADS[2].seed)
    check(o, lse, O_ref, L_ref, "bench mix")
