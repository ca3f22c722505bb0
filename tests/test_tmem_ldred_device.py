"""The reducing TMEM load the FP8 kernel's first pass uses for unmasked key
blocks (tcgen05.ld.red …max.f32), pinned on the device: every thread gets its
row's 32 values unchanged and, in the extra register, exactly their maximum
(rows with −inf, −0/+0, huge and tiny magnitudes, all −inf)."""

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
    out = os.path.join(tempfile.mkdtemp(prefix="ldredprobe_"), "libldredprobe.so")
    cmd = [nvcc, *build.ARCH, "-O3", "-std=c++17", "-shared", "-Xcompiler", "-fPIC", "-cudart", "shared",
           "-I" + CSRC, os.path.join(ROOT, "tests", "tmem_ldred_probe.cu"), "-o", out]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    L = ctypes.CDLL(out)
    L.ldred_probe_launch.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    L.ldred_probe_launch.restype = ctypes.c_int
    return L


def _rows():
    rng = np.random.default_rng(7)
    x = rng.standard_normal((128, 32)).astype(np.float32) * 30.0
    x[1] = -np.inf                                  # a fully masked row
    x[2, ::3] = -np.inf                             # partly masked
    x[3] = -rng.random(32).astype(np.float32)       # all negative
    x[4] = 0.0
    x[4, 5] = -0.0                                  # zeros of both signs
    x[5] = rng.standard_normal(32).astype(np.float32) * 1e30
    x[6] = rng.standard_normal(32).astype(np.float32) * 1e-30
    x[7, :] = 3.0
    x[8] = np.arange(32, dtype=np.float32)          # maximum in the last column
    x[9] = np.arange(32, dtype=np.float32)[::-1]    # ... in the first
    return x


@pytest.mark.gpu
def test_reducing_tmem_load_returns_row_maximum(probe):
    x = _rows()
    xin = torch.from_numpy(x).cuda()
    vals = torch.empty_like(xin)
    maxes = torch.empty(128, dtype=torch.float32, device="cuda")
    rc = probe.ldred_probe_launch(xin.data_ptr(), vals.data_ptr(), maxes.data_ptr(),
                                  ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0
    torch.cuda.synchronize()
    v, m = vals.cpu().numpy(), maxes.cpu().numpy()
    assert np.array_equal(v.view(np.uint32), x.view(np.uint32)), "loaded values differ from the stored ones"
    want = x.max(axis=1)
    assert np.array_equal(m, want), f"rows {np.nonzero(m != want)[0][:8]}: {m[m != want][:4]} vs {want[m != want][:4]}"
