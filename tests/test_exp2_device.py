"""The softmax's FMA-pipe exp2 (attn::ex2_poly2) evaluated on the GPU and
pinned to the closed form 2^x in float64 on a dense grid.

The kernels compute 2^x either on the MUFU unit or, for a compile-time share
of the exponentials, with a cubic on the FMA pipes ("FlashAttention 4: Atenção
Mais Rápida …", section "Exponenciais de Software via Núcleos CUDA").  The
cubic's fit (exact constant term, minimax relative error 8.6e-5 on [0, 1)) is
checked here on the device code itself, built from the library's header by
this test: relative error ≤ 1e-4 wherever 2^x is a normal float, exactly +0.0
at and below the lower clamp (−127), exact powers of two at integers, and
2^127 at and above the upper clamp.
"""

import ctypes
import os
import subprocess
import tempfile

import numpy as np
import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "exact_attention_63_gb300", "csrc")


@pytest.fixture(scope="module")
def probe():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from exact_attention_63_gb300 import build

    nvcc = build.nvcc_path()
    out = os.path.join(tempfile.mkdtemp(prefix="ex2probe_"), "libex2probe.so")
    cmd = [nvcc, *build.ARCH, "-O3", "-std=c++17", "-shared", "-Xcompiler", "-fPIC", "-cudart", "shared",
           "-I" + CSRC, os.path.join(ROOT, "tests", "ex2_poly_probe.cu"), "-o", out]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    L = ctypes.CDLL(out)
    L.ex2_poly_eval_launch.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p]
    L.ex2_poly_eval_launch.restype = ctypes.c_int
    return L


def _eval(L, x: np.ndarray) -> np.ndarray:
    xs = np.asarray(x, dtype=np.float32)
    if xs.size % 2:
        xs = np.append(xs, np.float32(0))
    xd = torch.from_numpy(xs).cuda()
    yd = torch.empty_like(xd)
    rc = L.ex2_poly_eval_launch(xd.data_ptr(), yd.data_ptr(), xd.numel(),
                                ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0
    torch.cuda.synchronize()
    return yd.cpu().numpy()[: np.asarray(x).size]


@pytest.mark.gpu
def test_poly_exp2_relative_error_on_dense_grid(probe):
    # The softmax feeds it x = s·scale·log2(e) − m ≤ τ (at most 64); cover to 127.
    x = np.linspace(-126.0, 127.0, (1 << 22) + 2, dtype=np.float64).astype(np.float32)
    y = _eval(probe, x).astype(np.float64)
    ref = np.exp2(x.astype(np.float64))
    rel = np.abs(y / ref - 1.0)
    assert rel.max() <= 1e-4, f"max relative error {rel.max():.3e} at x = {x[rel.argmax()]}"
    # a finer grid over one period shows the fit's own error (8.6e-5)
    f = np.linspace(0.0, 1.0, 1 << 16, endpoint=False, dtype=np.float32)
    rel_f = np.abs(_eval(probe, f).astype(np.float64) / np.exp2(f.astype(np.float64)) - 1.0)
    assert 5e-5 < rel_f.max() <= 1e-4


@pytest.mark.gpu
def test_poly_exp2_integers_are_exact_powers_of_two(probe):
    j = np.arange(-126, 128, dtype=np.float32)
    y = _eval(probe, j).astype(np.float64)
    assert np.array_equal(y, np.exp2(j.astype(np.float64)))


@pytest.mark.gpu
def test_poly_exp2_clamps(probe):
    lo = np.array([-np.inf, -1e30, -1000.0, -200.0, -127.5, -127.0], dtype=np.float32)
    y = _eval(probe, lo)
    assert np.all(y == 0.0) and not np.any(np.signbit(y)), y
    # between the clamp and the smallest normal: a value in [0, 2^-126]
    mid = np.linspace(-126.999, -126.001, 64, dtype=np.float32)
    ym = _eval(probe, mid).astype(np.float64)
    assert np.all(ym >= 0.0) and np.all(ym <= 2.0 ** -126)
    hi = np.array([127.0, 127.5, 128.0, 300.0, 1e30, np.inf], dtype=np.float32)
    yh = _eval(probe, hi).astype(np.float64)
    assert np.all(yh == 2.0 ** 127), yh
