"""Error bounds of the approximate math in the shape-specialised kernels,
evaluated on the GPU through the library's probe entry point and compared
with float64 (numpy) on the same FP32 inputs, and with CUDA's accurate
sinf / cosf / expf.

Bounds (stated here, asserted below), over the ranges the kernels see and
beyond them:
  sin / cos   |x| <= 2e4 (rotary angles)         absolute error <= 2e-6
  exp         -60 <= x <= 0 (exp(segsum) below   relative error <= 5e-6
              the diagonal: segsum <= 0)
  sigmoid     |x| <= 40 (gate pre-activations)   relative error <= 3e-6
(The larger exp / sigmoid errors at the ends of these ranges come from
rounding x log2 e to FP32 before ex2.approx: half an ulp of 86 is 2^-18.)
"""

import ctypes

import numpy as np
import pytest
import torch

import mamba_mimo_chunked_gb300 as mm

pytestmark = pytest.mark.gpu


def probe(which, x):
    lib = mm.load_library()
    lib.mamba_mimo_probe_fast_math.restype = ctypes.c_int
    xd = torch.as_tensor(x, dtype=torch.float32).cuda()
    out = torch.empty(4 * xd.numel(), dtype=torch.float32, device="cuda")
    st = lib.mamba_mimo_probe_fast_math(which, ctypes.c_void_p(xd.data_ptr()), ctypes.c_void_p(out.data_ptr()),
                                        xd.numel(), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, lib.mamba_mimo_last_error().decode()
    torch.cuda.synchronize()
    return xd.cpu().numpy().astype(np.float64), out.cpu().numpy().astype(np.float64).reshape(-1, 4)


def grid(lo, hi, n, seed):
    rng = np.random.default_rng(seed)
    edges = np.array([lo, hi, 0.0, -0.0, np.pi, -np.pi, 2 * np.pi, 1e-30, -1e-30], dtype=np.float64)
    edges = edges[(edges >= lo) & (edges <= hi)]
    return np.concatenate([rng.uniform(lo, hi, n), np.linspace(lo, hi, n), edges]).astype(np.float32)


def test_sincos_absolute_error():
    for lo, hi in ((-np.pi, np.pi), (-2e4, 2e4)):
        x, out = probe(0, grid(lo, hi, 1 << 18, 1))
        s, c = np.sin(x), np.cos(x)
        assert np.max(np.abs(out[:, 0] - s)) <= 2e-6
        assert np.max(np.abs(out[:, 1] - c)) <= 2e-6
        # CUDA's accurate sinf / cosf agree with float64 far closer
        assert np.max(np.abs(out[:, 2] - s)) <= 2e-7 and np.max(np.abs(out[:, 3] - c)) <= 2e-7


def test_exp_relative_error():
    x, out = probe(1, grid(-60.0, 0.0, 1 << 18, 2))
    ref = np.exp(x)
    assert np.max(np.abs(out[:, 0] - ref) / ref) <= 5e-6
    assert np.max(np.abs(out[:, 2] - ref) / ref) <= 5e-7


def test_sigmoid_relative_error():
    x, out = probe(2, grid(-40.0, 40.0, 1 << 18, 3))
    ref = 1.0 / (1.0 + np.exp(-x))
    assert np.max(np.abs(out[:, 0] - ref) / ref) <= 3e-6
    assert np.max(np.abs(out[:, 2] - ref) / ref) <= 5e-7


def test_probe_rejects_bad_arguments():
    lib = mm.load_library()
    assert lib.mamba_mimo_probe_fast_math(3, None, None, 0, None) != 0
    assert lib.mamba_mimo_probe_fast_math(0, None, None, -1, None) != 0
