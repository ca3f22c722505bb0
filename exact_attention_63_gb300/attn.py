"""Thin ctypes binding over the C ABI in ``include/attn_gb300.h``.

Argument marshalling only: shape/dtype checks, device pointers, the current
CUDA stream.  All of the computation runs in the library's CUDA kernels; if
the shared library is missing or cannot be loaded, every call raises — there
is no fallback path.
"""

from __future__ import annotations

import ctypes
import math
import os

import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libattn_gb300.so")
_lib = None

ATTN_OK = 0
ERRORS = {
    -1: "ATTN_ERR_NULL", -2: "ATTN_ERR_SHAPE", -3: "ATTN_ERR_HEAD_DIM", -4: "ATTN_ERR_SCALE",
    -5: "ATTN_ERR_ALIGN", -6: "ATTN_ERR_ARCH", -7: "ATTN_ERR_LAUNCH", -8: "ATTN_ERR_TIMEOUT",
    -9: "ATTN_ERR_OPTION", -10: "ATTN_ERR_WORKSPACE", -11: "ATTN_ERR_STATIC_LIMIT", -12: "ATTN_ERR_LAYOUT",
}

# Every symbol the header declares (checked by the CPU test-suite).
EXPORTS = ["attn_fwd", "attn_fwd_ex", "attn_fwd_host", "attn_fwd_host_workspace_size", "attn_get_status",
           "attn_strerror", "attn_last_cuda_error", "attn_version", "attn_fwd_host_static", "attn_fwd_layout",
           "attn_fwd_varlen", "attn_bwd", "attn_bwd_workspace_size", "attn_bwd_layout", "attn_bwd_ex",
           "attn_fwd_fp8", "attn_fwd_fp8_ex"]

CAUSAL_ALIGN = {"top-left": 0, "bottom-right": 1}

# Size of the library's fixed device staging area used by attn_fwd_host_static.
STATIC_WORKSPACE_BYTES = 32 << 20


class AttnError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{ERRORS.get(code, code)}: {msg}")
        self.code = code


class Options(ctypes.Structure):
    """Mirror of ``attn_options``."""
    _fields_ = [("struct_size", ctypes.c_size_t), ("rescale_threshold", ctypes.c_float),
                ("poly_exp2_mask", ctypes.c_uint), ("counters", ctypes.c_void_p), ("timeout_ms", ctypes.c_uint),
                ("test_flags", ctypes.c_uint)]


class Layout(ctypes.Structure):
    """Mirror of ``attn_layout``."""
    _fields_ = [("struct_size", ctypes.c_size_t), ("num_kv_heads", ctypes.c_int), ("causal_align", ctypes.c_int),
                ("q_strides", ctypes.c_longlong * 3), ("k_strides", ctypes.c_longlong * 3),
                ("v_strides", ctypes.c_longlong * 3), ("o_strides", ctypes.c_longlong * 3)]


def make_layout(num_kv_heads: int = 0, causal_align: int = 0, q_strides=(0, 0, 0), k_strides=(0, 0, 0),
                v_strides=(0, 0, 0), o_strides=(0, 0, 0)) -> Layout:
    lay = Layout()
    lay.struct_size = ctypes.sizeof(Layout)
    lay.num_kv_heads = num_kv_heads
    lay.causal_align = causal_align
    for name, st in (("q_strides", q_strides), ("k_strides", k_strides), ("v_strides", v_strides),
                     ("o_strides", o_strides)):
        getattr(lay, name)[:] = [int(x) for x in st]
    return lay


def lib():
    """Load the shared library (raises if it is missing)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_LIB_PATH):
        raise RuntimeError(f"{_LIB_PATH} is missing: build it with `python -m exact_attention_63_gb300.build`")
    L = ctypes.CDLL(_LIB_PATH)
    vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    L.attn_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp]
    L.attn_fwd.restype = i
    L.attn_fwd_ex.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, i, ctypes.POINTER(Options), vp]
    L.attn_fwd_ex.restype = i
    L.attn_fwd_layout.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, i, ctypes.POINTER(Layout),
                                  ctypes.POINTER(Options), vp]
    L.attn_fwd_layout.restype = i
    L.attn_fwd_varlen.argtypes = [vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, f, i, i, ctypes.POINTER(Options),
                                  vp]
    L.attn_fwd_varlen.restype = i
    L.attn_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp, sz, vp]
    L.attn_bwd.restype = i
    L.attn_bwd_layout.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, i, ctypes.POINTER(Layout), vp,
                                  sz, vp]
    L.attn_bwd_layout.restype = i
    L.attn_bwd_ex.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, i, ctypes.POINTER(Layout),
                              ctypes.c_uint, vp, sz, vp]
    L.attn_bwd_ex.restype = i
    L.attn_bwd_workspace_size.argtypes = [i, i, i]
    L.attn_bwd_workspace_size.restype = sz
    L.attn_fwd_host.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp, sz, vp]
    L.attn_fwd_host.restype = i
    L.attn_fwd_host_workspace_size.argtypes = [i, i, i, i, i]
    L.attn_fwd_host_workspace_size.restype = sz
    L.attn_fwd_host_static.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp]
    L.attn_fwd_host_static.restype = i
    L.attn_fwd_fp8.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, f, f, f, i, vp]
    L.attn_fwd_fp8.restype = i
    L.attn_fwd_fp8_ex.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, f, f, f, i, ctypes.POINTER(Options), vp]
    L.attn_fwd_fp8_ex.restype = i
    L.attn_get_status.argtypes = [vp]
    L.attn_get_status.restype = i
    L.attn_strerror.argtypes = [i]
    L.attn_strerror.restype = ctypes.c_char_p
    L.attn_last_cuda_error.argtypes = []
    L.attn_last_cuda_error.restype = ctypes.c_char_p
    L.attn_version.argtypes = []
    L.attn_version.restype = i
    _lib = L
    return L


def _check(rc: int):
    if rc != ATTN_OK:
        L = lib()
        msg = L.attn_strerror(rc).decode()
        extra = L.attn_last_cuda_error().decode()
        raise AttnError(rc, msg + (f" ({extra})" if extra and rc == -7 else ""))


def _stream_handle(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check_tensor(name, t):
    if t.dtype != torch.bfloat16 or not t.is_cuda or t.dim() != 4 or t.stride(3) != 1:
        raise ValueError(f"{name} must be a 4-D bf16 CUDA tensor (batch, seq, heads, head_dim) "
                         "with a contiguous head_dim")


def _check_inputs(q, k, v):
    for name, t in (("q", q), ("k", k), ("v", v)):
        _check_tensor(name, t)
    B, Sq, H, d = q.shape
    if k.shape != v.shape or k.shape[0] != B or k.shape[3] != d or k.shape[2] < 1 or H % k.shape[2] != 0:
        raise ValueError(f"shape mismatch: q {tuple(q.shape)}, k {tuple(k.shape)}, v {tuple(v.shape)} "
                         "(k and v: (batch, Sk, H_kv, head_dim) with H a multiple of H_kv)")
    return B, H, Sq, k.shape[1], d


def _strides(t):
    return (t.stride(0), t.stride(1), t.stride(2))


def attn_fwd(q, k, v, causal: bool = False, scale: float | None = None, out=None, lse=None, stream=None,
             options: Options | None = None, causal_align: str = "top-left"):
    """Exact attention forward.  Returns (o [B,Sq,H,d] bf16, lse [B,H,Sq] fp32).

    k and v may have fewer heads than q (grouped-query attention: query head h
    reads key/value head h // (H / H_kv)); q, k, v and out may be strided views
    whose head_dim is contiguous (strides are passed to the library, which
    needs them to be multiples of 8 elements).  ``causal_align`` is
    "top-left" (key j visible to row i iff j <= i) or "bottom-right"
    (iff j <= i + Sk - Sq).
    """
    B, H, Sq, Sk, d = _check_inputs(q, k, v)
    if causal_align not in CAUSAL_ALIGN:
        raise ValueError(f"causal_align must be one of {sorted(CAUSAL_ALIGN)}")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty((B, Sq, H, d), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((B, H, Sq), dtype=torch.float32, device=q.device)
    _check_tensor("out", out)
    if tuple(out.shape) != (B, Sq, H, d):
        raise ValueError("out must be shaped like q")
    if lse.shape != (B, H, Sq) or lse.dtype != torch.float32 or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous fp32 tensor of shape (B, H, Sq)")
    dense = all(t.is_contiguous() for t in (q, k, v, out))
    plain = dense and k.shape[2] == H and (not causal or causal_align == "top-left")
    L = lib()
    with torch.cuda.device(q.device):
        s = _stream_handle(stream)
        if options is not None:
            options.struct_size = ctypes.sizeof(Options)
        if plain and options is None:
            rc = L.attn_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                            B, H, Sq, Sk, d, float(scale), int(bool(causal)), s)
        elif plain:
            rc = L.attn_fwd_ex(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                               B, H, Sq, Sk, d, float(scale), int(bool(causal)), ctypes.byref(options), s)
        else:
            lay = make_layout(k.shape[2], CAUSAL_ALIGN[causal_align], _strides(q), _strides(k), _strides(v),
                              _strides(out))
            rc = L.attn_fwd_layout(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                                   B, H, Sq, Sk, d, float(scale), int(bool(causal)), ctypes.byref(lay),
                                   ctypes.byref(options) if options is not None else None, s)
    _check(rc)
    return out, lse


def attn_fwd_varlen(q, k, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q: int, causal: bool = False,
                    scale: float | None = None, out=None, lse=None, stream=None, options: Options | None = None,
                    causal_align: str = "top-left"):
    """Exact attention over sequences of different lengths packed along the rows.

    q [total_q, H, d], k and v [total_k, H_kv, d] (dense bf16, H a multiple of
    H_kv); cu_seqlens_q / cu_seqlens_k: int32 CUDA tensors of n + 1 ascending
    row offsets starting at 0 (sequence s owns rows [cu[s], cu[s+1]));
    max_seqlen_q >= every query length.  Returns (o [total_q, H, d] bf16,
    lse [H, total_q] fp32).  Causal masks align per sequence.
    """
    for name, t in (("q", q), ("k", k), ("v", v)):
        if t.dtype != torch.bfloat16 or not t.is_cuda or t.dim() != 3 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous 3-D bf16 CUDA tensor (rows, heads, head_dim)")
    total_q, H, d = q.shape
    total_k, H_kv = k.shape[0], k.shape[1]
    if k.shape != v.shape or k.shape[2] != d or H % H_kv != 0:
        raise ValueError(f"shape mismatch: q {tuple(q.shape)}, k {tuple(k.shape)}, v {tuple(v.shape)}")
    for name, t in (("cu_seqlens_q", cu_seqlens_q), ("cu_seqlens_k", cu_seqlens_k)):
        if t.dtype != torch.int32 or not t.is_cuda or t.dim() != 1 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous 1-D int32 CUDA tensor")
    n_seq = cu_seqlens_q.numel() - 1
    if cu_seqlens_k.numel() != n_seq + 1:
        raise ValueError("cu_seqlens_q and cu_seqlens_k must have the same length")
    if causal_align not in CAUSAL_ALIGN:
        raise ValueError(f"causal_align must be one of {sorted(CAUSAL_ALIGN)}")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((H, total_q), dtype=torch.float32, device=q.device)
    if out.shape != q.shape or out.dtype != torch.bfloat16 or not out.is_contiguous():
        raise ValueError("out must be a contiguous bf16 tensor shaped like q")
    if lse.shape != (H, total_q) or lse.dtype != torch.float32 or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous fp32 tensor of shape (H, total_q)")
    if options is not None:
        options.struct_size = ctypes.sizeof(Options)
    with torch.cuda.device(q.device):
        rc = lib().attn_fwd_varlen(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                                   cu_seqlens_q.data_ptr(), cu_seqlens_k.data_ptr(), n_seq, total_q, total_k,
                                   int(max_seqlen_q), H, H_kv, d, float(scale), int(bool(causal)),
                                   CAUSAL_ALIGN[causal_align], ctypes.byref(options) if options is not None else None,
                                   _stream_handle(stream))
    _check(rc)
    return out, lse


BWD_DETERMINISTIC = 1


def attn_bwd(q, k, v, o, lse, dout, causal: bool = False, scale: float | None = None, dq=None, dk=None, dv=None,
             workspace=None, stream=None, causal_align: str = "top-left", deterministic: bool = False):
    """Gradients of attn_fwd's output: returns (dq, dk, dv), bf16, shaped
    like q, k, v (dense).  o and lse are what attn_fwd returned for the same
    inputs; dout is the gradient of the loss with respect to o.
    (batch, seq, heads, head_dim) tensors; q, k, v and o may be strided views
    whose head_dim is contiguous (e.g. slices of a packed QKV tensor); dout is
    made dense if it is not; k and v may have fewer heads than q (grouped
    query heads; a shared head's gradient sums its group's).  At head dim 64
    one pass computes all three by default (dq's fp32 sums run in a varying
    order, so its last bits may change between runs); at 128, or with
    deterministic=True, two passes, reproducible bit for bit."""
    B, H, Sq, Sk, d = _check_inputs(q, k, v)
    H_kv = k.shape[2]
    for name, t in (("o", o), ("dout", dout)):
        _check_tensor(name, t)
        if t.shape != q.shape:
            raise ValueError(f"{name} must be shaped like q")
    dout = dout.contiguous()
    if causal_align not in CAUSAL_ALIGN:
        raise ValueError(f"causal_align must be one of {sorted(CAUSAL_ALIGN)}")
    if lse.shape != (B, H, Sq) or lse.dtype != torch.float32 or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous fp32 tensor of shape (B, H, Sq)")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dq = torch.empty(q.shape, dtype=torch.bfloat16, device=q.device) if dq is None else dq
    dk = torch.empty(k.shape, dtype=torch.bfloat16, device=k.device) if dk is None else dk
    dv = torch.empty(v.shape, dtype=torch.bfloat16, device=v.device) if dv is None else dv
    for name, t, ref in (("dq", dq, q), ("dk", dk, k), ("dv", dv, v)):
        if t.shape != ref.shape or t.dtype != torch.bfloat16 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous bf16 tensor shaped like its input")
    L = lib()
    need = int(L.attn_bwd_workspace_size(B, H, Sq))
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    lay = make_layout(H_kv, CAUSAL_ALIGN[causal_align], _strides(q), _strides(k), _strides(v), _strides(o))
    with torch.cuda.device(q.device):
        rc = L.attn_bwd_ex(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                           dout.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, Sq, Sk, d,
                           float(scale), int(bool(causal)), ctypes.byref(lay),
                           BWD_DETERMINISTIC if deterministic else 0, workspace.data_ptr(),
                           workspace.numel() * workspace.element_size(), _stream_handle(stream))
    _check(rc)
    return dq, dk, dv


class _Attention(torch.autograd.Function):
    """attn_fwd as an autograd function: the forward keeps O and LSE, the
    backward hands them with dO to attn_bwd (the LSE output itself is not
    differentiated)."""

    @staticmethod
    def forward(ctx, q, k, v, causal, scale, causal_align, deterministic):
        o, lse = attn_fwd(q, k, v, causal=causal, scale=scale, causal_align=causal_align)
        ctx.save_for_backward(q, k, v, o, lse)
        ctx.cfg = (causal, scale, causal_align, deterministic)
        ctx.mark_non_differentiable(lse)
        return o, lse

    @staticmethod
    def backward(ctx, do, _dlse):
        q, k, v, o, lse = ctx.saved_tensors
        causal, scale, causal_align, deterministic = ctx.cfg
        dq, dk, dv = attn_bwd(q, k, v, o, lse, do.contiguous(), causal=causal, scale=scale,
                              causal_align=causal_align, deterministic=deterministic)
        return dq, dk, dv, None, None, None, None


def attention(q, k, v, causal: bool = False, scale: float | None = None, causal_align: str = "top-left",
              deterministic: bool = False):
    """Exact attention with gradients: returns (o, lse) like attn_fwd, and
    o's gradient flows back to q, k and v through attn_bwd.  (batch, seq,
    heads, head_dim) bf16 CUDA tensors, strided views allowed as for
    attn_fwd; k and v may have fewer heads than q.  ``deterministic`` selects attn_bwd's bit-reproducible
    schedule."""
    return _Attention.apply(q, k, v, causal, scale, causal_align, deterministic)


TEST_WITHHOLD_KV = 1
TEST_FALLBACK_KERNEL = 2


def make_options(rescale_threshold: float = 0.0, poly_exp2_mask: int = 0, counters=None, timeout_ms: int = 0,
                 test_flags: int = 0):
    o = Options()
    o.struct_size = ctypes.sizeof(Options)
    o.rescale_threshold = rescale_threshold
    o.poly_exp2_mask = poly_exp2_mask
    o.counters = None if counters is None else counters.data_ptr()
    o.timeout_ms = timeout_ms
    o.test_flags = test_flags
    return o


def workspace_size(B, H, Sq, Sk, d) -> int:
    return int(lib().attn_fwd_host_workspace_size(B, H, Sq, Sk, d))


def attn_fwd_host(q_h, k_h, v_h, o_h, lse_h, causal: bool, scale: float, workspace, stream=None):
    """End-to-end call on host tensors (pinned CPU bf16 q/k/v/o, fp32 lse).

    ``workspace`` is a CUDA uint8 tensor of at least ``workspace_size(...)``
    bytes.  Enqueues copies + kernel on the stream; does not synchronise.
    """
    B, Sq, H, d = q_h.shape
    Sk = k_h.shape[1]
    L = lib()
    with torch.cuda.device(workspace.device):
        rc = L.attn_fwd_host(q_h.data_ptr(), k_h.data_ptr(), v_h.data_ptr(), o_h.data_ptr(), lse_h.data_ptr(),
                             B, H, Sq, Sk, d, float(scale), int(bool(causal)), workspace.data_ptr(),
                             workspace.numel() * workspace.element_size(), _stream_handle(stream))
    _check(rc)


def attn_fwd_host_static(q_h, k_h, v_h, o_h, lse_h, causal: bool, scale: float, stream=None):
    """End-to-end call on host tensors with no device workspace from the
    caller: the library stages the data in its own fixed 32 MiB device array
    (for callers that cannot allocate device memory).  Does not synchronise."""
    B, Sq, H, d = q_h.shape
    Sk = k_h.shape[1]
    rc = lib().attn_fwd_host_static(q_h.data_ptr(), k_h.data_ptr(), v_h.data_ptr(), o_h.data_ptr(),
                                    lse_h.data_ptr(), B, H, Sq, Sk, d, float(scale), int(bool(causal)),
                                    _stream_handle(stream))
    _check(rc)


def attn_fwd_fp8(q8, k8, v8, descale_q: float, descale_k: float, descale_v: float, causal: bool = False,
                 scale: float | None = None, out=None, lse=None, stream=None, options=None):
    """Exact attention forward on FP8 (E4M3) inputs: q8 [B,Sq,H,128], k8, v8
    [B,Sk,H,128] as torch.float8_e4m3fn (or their raw bytes as uint8), standing
    for descale_x · x8.  Returns (o [B,Sq,H,128] bf16, lse [B,H,Sq] fp32).
    ``options`` (from make_options; timeout_ms and test_flags only) selects
    attn_fwd_fp8_ex."""
    for name, t in (("q8", q8), ("k8", k8), ("v8", v8)):
        if t.dtype not in (torch.float8_e4m3fn, torch.uint8) or not t.is_cuda or t.dim() != 4 or \
                not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous 4-D E4M3 CUDA tensor (batch, seq, heads, head_dim)")
    B, Sq, H, d = q8.shape
    if k8.shape != v8.shape or k8.shape[0] != B or k8.shape[2] != H or k8.shape[3] != d:
        raise ValueError(f"shape mismatch: q8 {tuple(q8.shape)}, k8 {tuple(k8.shape)}, v8 {tuple(v8.shape)}")
    Sk = k8.shape[1]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty((B, Sq, H, d), dtype=torch.bfloat16, device=q8.device)
    if lse is None:
        lse = torch.empty((B, H, Sq), dtype=torch.float32, device=q8.device)
    if out.dtype != torch.bfloat16 or tuple(out.shape) != (B, Sq, H, d) or not out.is_contiguous():
        raise ValueError("out must be a contiguous bf16 tensor shaped like q8")
    if lse.shape != (B, H, Sq) or lse.dtype != torch.float32 or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous fp32 tensor of shape (B, H, Sq)")
    with torch.cuda.device(q8.device):
        args = (q8.data_ptr(), k8.data_ptr(), v8.data_ptr(), out.data_ptr(), lse.data_ptr(), B, H, Sq, Sk, d,
                float(scale), float(descale_q), float(descale_k), float(descale_v), int(bool(causal)))
        if options is None:
            rc = lib().attn_fwd_fp8(*args, _stream_handle(stream))
        else:
            rc = lib().attn_fwd_fp8_ex(*args, ctypes.byref(options), _stream_handle(stream))
    _check(rc)
    return out, lse


def get_status(stream=None) -> int:
    """Synchronise the stream and return/clear the device status (0 = ok)."""
    return int(lib().attn_get_status(_stream_handle(stream)))


def raw_fwd_varlen(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, cu_q_ptr, cu_k_ptr, n_seq, total_q, total_k, max_q, H, H_kv,
                   d, scale, causal, causal_align=0, stream_ptr=0) -> int:
    """Direct attn_fwd_varlen call with integer pointers; returns the status code (tests)."""
    return int(lib().attn_fwd_varlen(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, cu_q_ptr, cu_k_ptr, n_seq, total_q, total_k,
                                     max_q, H, H_kv, d, float(scale), int(causal), causal_align, None,
                                     ctypes.c_void_p(stream_ptr)))


def raw_fwd_layout(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, B, H, Sq, Sk, d, scale, causal, layout, stream_ptr=0) -> int:
    """Direct attn_fwd_layout call with integer pointers; returns the status code (tests)."""
    return int(lib().attn_fwd_layout(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, B, H, Sq, Sk, d, float(scale), int(causal),
                                     None if layout is None else ctypes.byref(layout), None,
                                     ctypes.c_void_p(stream_ptr)))


def raw_fwd(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, B, H, Sq, Sk, d, scale, causal, stream_ptr=0) -> int:
    """Direct C-ABI call with integer pointers; returns the status code (tests)."""
    return int(lib().attn_fwd(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, B, H, Sq, Sk, d, float(scale), int(causal),
                              ctypes.c_void_p(stream_ptr)))
