"""C-ABI library: it loads, exports every declared symbol, and rejects bad
arguments before touching the GPU (no GPU needed for any of this)."""

import ctypes
import os
import re

import pytest

from exact_attention_63_gb300 import attn

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "attn_gb300.h")


@pytest.fixture(scope="module")
def L():
    if not os.path.exists(attn._LIB_PATH):
        from exact_attention_63_gb300 import build

        build.build()
    return attn.lib()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[a-z_]+\**\s+\**(attn_[a-z0-9_]+)\s*\(", src, flags=re.M)))


def test_header_declares_expected_api():
    assert declared_functions() == sorted(attn.EXPORTS)


def test_library_exports_every_declared_symbol(L):
    for name in declared_functions():
        assert hasattr(L, name), name


def test_version_and_strerror(L):
    assert L.attn_version() >= 100
    for code in [0, *attn.ERRORS]:
        assert L.attn_strerror(code)
    assert L.attn_strerror(12345) == b"unknown status"


A = 0x10000  # a fake, 16-byte aligned "device" address: never dereferenced


@pytest.mark.parametrize("args,expect", [
    ((0, A, A, A, A, 1, 1, 8, 8, 64, 0.125, 0), -1),
    ((A, A, A, A, 0, 1, 1, 8, 8, 64, 0.125, 0), -1),
    ((A, A, A, A, A, 0, 1, 8, 8, 64, 0.125, 0), -2),
    ((A, A, A, A, A, 1, -1, 8, 8, 64, 0.125, 0), -2),
    ((A, A, A, A, A, 1, 1, 0, 8, 64, 0.125, 0), -2),
    ((A, A, A, A, A, 1, 1, 8, 0, 64, 0.125, 0), -2),
    ((A, A, A, A, A, 65536, 65536, 4096, 8, 64, 0.125, 0), -2),
    ((A, A, A, A, A, 1, 1, 8, 8, 96, 0.125, 0), -3),
    ((A, A, A, A, A, 1, 1, 8, 8, 256, 0.125, 0), -3),
    ((A, A, A, A, A, 1, 1, 8, 8, 64, float("nan"), 0), -4),
    ((A, A, A, A, A, 1, 1, 8, 8, 64, float("inf"), 0), -4),
    ((A, A, A, A, A, 1, 1, 8, 8, 64, 0.0, 0), -4),
    ((A, A, A, A, A, 1, 1, 8, 8, 64, -1.0, 0), -4),
    ((A + 8, A, A, A, A, 1, 1, 8, 8, 64, 0.125, 0), -5),
    ((A, A, A, A, A + 4, 1, 1, 8, 8, 64, 0.125, 0), -5),
])
def test_rejected_before_launch(L, args, expect):
    assert attn.raw_fwd(*args) == expect


def test_bad_options_rejected(L):
    o = attn.make_options(rescale_threshold=float("nan"))
    rc = L.attn_fwd_ex(A, A, A, A, A, 1, 1, 8, 8, 64, 0.125, 0, ctypes.byref(o), None)
    assert rc == -9
    o = attn.make_options(rescale_threshold=70.0)
    assert L.attn_fwd_ex(A, A, A, A, A, 1, 1, 8, 8, 64, 0.125, 0, ctypes.byref(o), None) == -9
    for bad_mask in (0x200, 0x0F, 0x03, 0x101):
        o = attn.make_options(poly_exp2_mask=bad_mask)
        assert L.attn_fwd_ex(A, A, A, A, A, 1, 1, 8, 8, 64, 0.125, 0, ctypes.byref(o), None) == -9
    o = attn.make_options()
    o.struct_size = 4
    assert L.attn_fwd_ex(A, A, A, A, A, 1, 1, 8, 8, 64, 0.125, 0, ctypes.byref(o), None) == -9


def test_workspace_size_and_checks(L):
    n = attn.workspace_size(2, 3, 100, 50, 64)
    up = lambda x: (x + 255) // 256 * 256  # noqa: E731
    assert n == 2 * up(2 * 100 * 3 * 64 * 2) + 2 * up(2 * 50 * 3 * 64 * 2) + up(2 * 3 * 100 * 4)
    assert attn.workspace_size(1, 1, 1, 1, 96) == 0
    rc = L.attn_fwd_host(A, A, A, A, A, 2, 3, 100, 50, 64, 0.125, 0, A, n - 1, None)
    assert rc == -10
    rc = L.attn_fwd_host(A, A, A, A, A, 2, 3, 100, 50, 64, 0.125, 0, A + 16, n, None)
    assert rc == -10
    rc = L.attn_fwd_host(0, A, A, A, A, 2, 3, 100, 50, 64, 0.125, 0, A, n, None)
    assert rc == -1


def test_no_gpu_reports_arch_error(L):
    import torch

    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert attn.raw_fwd(A, A, A, A, A, 1, 1, 8, 8, 64, 0.125, 0) == -6


def test_python_binding_rejects_cpu_tensors():
    import torch

    q = torch.zeros(1, 8, 1, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        attn.attn_fwd(q, q, q)


@pytest.mark.parametrize("lay,expect", [
    (dict(num_kv_heads=3), -12),                       # H = 4 is not a multiple of 3
    (dict(num_kv_heads=-1), -12),
    (dict(num_kv_heads=8), -12),                       # more K/V heads than query heads
    (dict(causal_align=2), -12),
    (dict(q_strides=(4096, 512, 60)), -12),            # not a multiple of 8 elements
    (dict(k_strides=(4096, 0, 64)), -12),              # zero mixed with non-zero strides
    (dict(v_strides=(-4096, 512, 64)), -12),
    (dict(o_strides=(1 << 38, 512, 64)), -12),         # beyond the TMA stride range
])
def test_bad_layout_rejected(L, lay, expect):
    layout = attn.make_layout(**lay)
    assert attn.raw_fwd_layout(A, A, A, A, A, 2, 4, 8, 8, 64, 0.125, 1, layout) == expect


def test_layout_struct_size_checked(L):
    layout = attn.make_layout()
    layout.struct_size = 8
    assert attn.raw_fwd_layout(A, A, A, A, A, 1, 1, 8, 8, 64, 0.125, 0, layout) == -12


def test_layout_argument_checks_come_first(L):
    # Plain argument errors are reported as by attn_fwd, layout or not.
    layout = attn.make_layout(num_kv_heads=3)
    assert attn.raw_fwd_layout(A, A, A, A, A, 1, 4, 8, 8, 96, 0.125, 0, layout) == -3
    assert attn.raw_fwd_layout(0, A, A, A, A, 1, 4, 8, 8, 64, 0.125, 0, None) == -1


@pytest.mark.parametrize("args,expect", [
    ((0, A, A, A, A, A, A, 2, 100, 100, 64, 4, 2, 64, 0.125, 1), -1),
    ((A, A, A, A, A, 0, A, 2, 100, 100, 64, 4, 2, 64, 0.125, 1), -1),
    ((A, A, A, A, A, A, A, 0, 100, 100, 64, 4, 2, 64, 0.125, 1), -2),   # no sequences
    ((A, A, A, A, A, A, A, 2, 0, 100, 64, 4, 2, 64, 0.125, 1), -2),
    ((A, A, A, A, A, A, A, 2, 100, 0, 64, 4, 2, 64, 0.125, 1), -2),
    ((A, A, A, A, A, A, A, 2, 100, 100, 0, 4, 2, 64, 0.125, 1), -2),   # max_seqlen_q
    ((A, A, A, A, A, A, A, 2, 100, 100, 64, 4, 2, 80, 0.125, 1), -3),
    ((A, A, A, A, A, A, A, 2, 100, 100, 64, 4, 2, 64, 0.0, 1), -4),
    ((A, A, A, A, A, A + 2, A, 2, 100, 100, 64, 4, 2, 64, 0.125, 1), -5),  # table not 4-byte aligned
    ((A + 8, A, A, A, A, A, A, 2, 100, 100, 64, 4, 2, 64, 0.125, 1), -5),
    ((A, A, A, A, A, A, A, 2, 100, 100, 64, 4, 3, 64, 0.125, 1), -12),  # H not a multiple of H_kv
    ((A, A, A, A, A, A, A, 2, 100, 100, 64, 4, 0, 64, 0.125, 1), -12),
])
def test_varlen_rejected_before_launch(L, args, expect):
    assert attn.raw_fwd_varlen(*args) == expect


def test_varlen_bad_alignment_rejected(L):
    assert attn.raw_fwd_varlen(A, A, A, A, A, A, A, 2, 100, 100, 64, 4, 2, 64, 0.125, 1, causal_align=5) == -12


def test_backward_layout_checks(L):
    bad = attn.make_layout(num_kv_heads=3)
    assert L.attn_bwd_layout(A, A, A, A, A, A, A, A, A, 1, 4, 8, 8, 64, 0.125, 1, ctypes.byref(bad), A, 1 << 20,
                             None) == -12
    # strides as for the forward: positive multiples of 8 elements (q, k, v, o may be strided)
    bad_strides = attn.make_layout(q_strides=(4096, 516, 64))
    assert L.attn_bwd_layout(A, A, A, A, A, A, A, A, A, 1, 4, 8, 8, 64, 0.125, 1, ctypes.byref(bad_strides), A,
                             1 << 20, None) == -12
    bad_o = attn.make_layout(o_strides=(4096, 512, 0))
    assert L.attn_bwd_layout(A, A, A, A, A, A, A, A, A, 1, 4, 8, 8, 64, 0.125, 1, ctypes.byref(bad_o), A,
                             1 << 20, None) == -12
    assert L.attn_bwd(A, A, A, A, A, A, A, A, A, 1, 4, 8, 8, 64, 0.125, 1, A, 16, None) == -10  # workspace too small
    assert L.attn_bwd(A, A, A, A, A, 0, A, A, A, 1, 4, 8, 8, 64, 0.125, 1, A, 1 << 20, None) == -1
    assert L.attn_bwd_ex(A, A, A, A, A, A, A, A, A, 1, 4, 8, 8, 64, 0.125, 1, None, 2, A, 1 << 20, None) == -9
    # workspace: −LSE·log2 e and D ([B·H, pitch] fp32 each, rounded up to 256
    # bytes), then the one-pass (d = 64) schedule's fp32 dQ accumulator
    # [B·H, pitch, 64]
    assert L.attn_bwd_workspace_size(1, 4, 8) == 2 * 4 * 128 * 4 + 4 * 128 * 64 * 4
    assert L.attn_bwd_workspace_size(2, 3, 129) == 2 * 6 * 256 * 4 + 6 * 256 * 64 * 4
    assert L.attn_bwd(A, A, A, A, A, A, A, A, A, 1, 4, 8, 8, 64, 0.125, 1, A,
                      L.attn_bwd_workspace_size(1, 4, 8) - 1, None) == -10


def test_static_workspace_size_matches_header():
    """The binding's copy of ATTN_STATIC_WORKSPACE_BYTES (used by the GPU test's
    limit checks) equals the header's definition."""
    src = open(HEADER).read()
    m = re.search(r"#define\s+ATTN_STATIC_WORKSPACE_BYTES\s+\((\d+)u\s*<<\s*(\d+)\)", src)
    assert m, "ATTN_STATIC_WORKSPACE_BYTES not found in the header"
    assert int(m.group(1)) << int(m.group(2)) == attn.STATIC_WORKSPACE_BYTES


@pytest.mark.parametrize("args,expect", [
    ((0, A, A, A, A, 1, 1, 8, 8, 128, 0.1, 1.0, 1.0, 1.0, 0), -1),
    ((A, A, A, A, A, 0, 1, 8, 8, 128, 0.1, 1.0, 1.0, 1.0, 0), -2),
    ((A, A, A, A, A, 1, 1, 8, 8, 64, 0.1, 1.0, 1.0, 1.0, 0), -3),
    ((A, A, A, A, A, 1, 1, 8, 8, 128, 0.0, 1.0, 1.0, 1.0, 0), -4),
    ((A, A, A, A, A, 1, 1, 8, 8, 128, 0.1, 0.0, 1.0, 1.0, 0), -4),
    ((A, A, A, A, A, 1, 1, 8, 8, 128, 0.1, 1.0, float("inf"), 1.0, 0), -4),
    ((A, A, A, A, A, 1, 1, 8, 8, 128, 0.1, 1.0, 1.0, -1.0, 0), -4),
    ((A + 1, A, A, A, A, 1, 1, 8, 8, 128, 0.1, 1.0, 1.0, 1.0, 0), -5),
])
def test_fp8_rejects_bad_arguments_before_launch(L, args, expect):
    assert L.attn_fwd_fp8(*args, None) == expect


def test_fp8_ex_rejects_options_that_do_not_apply(L):
    """attn_fwd_fp8_ex takes timeout_ms and test_flags only; everything else,
    and unknown test flags, are ATTN_ERR_OPTION before any device call."""
    args = (A, A, A, A, A, 1, 1, 8, 8, 128, 0.1, 1.0, 1.0, 1.0, 0)
    for kw in ({"rescale_threshold": 8.0}, {"poly_exp2_mask": 0x11}, {"test_flags": 4}):
        opts = attn.make_options(**kw)
        assert L.attn_fwd_fp8_ex(*args, ctypes.byref(opts), None) == -9, kw
    assert attn.TEST_FALLBACK_KERNEL == 2
