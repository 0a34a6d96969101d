"""The allocation-free entry point, mamba_mimo_bwd_fwd_fixed_scratch.

It serves callers that cannot allocate device memory themselves (a host
framework that owns all device memory through its own pool, code that must
not call cudaMalloc because it can synchronise the device) and therefore
cannot hand the library a workspace: its workspace is a built-in device
array.  These tests call it through the C ABI and check that two calls in a
row give the same results as the entry point with a caller workspace, and
that a problem too large for the built-in area is refused.  This file is
collected last on purpose: it must pass alone and after the other tests.
"""

import ctypes

import numpy as np
import pytest
import torch

import mamba_mimo_chunked_gb300 as mm
import oracle
import synthetic_inputs as si

pytestmark = pytest.mark.gpu
TOL = 1e-3
FIXED_SCRATCH_BYTES = 32 << 20


def _entry(lib):
    fn = lib.mamba_mimo_bwd_fwd_fixed_scratch
    fn.restype = ctypes.c_int
    fn.argtypes = ([ctypes.POINTER(mm._Dims)] + [ctypes.c_void_p] * 17 + [ctypes.c_int64] * 2
                   + [ctypes.c_void_p] * 6)
    return fn


def _rel_rms(a, b):
    a, b = a.double(), b.double()
    den = torch.sqrt(torch.mean(b * b))
    num = torch.sqrt(torch.mean((a - b) ** 2))
    return float(num / den) if den > 0 else float(num)


def _call_fixed(fn, inp, like):
    out = [None if t is None else torch.full_like(t, float("nan")) for t in like]
    q, v = inp["q"], inp["v"]
    B, S, R, G, N = q.shape
    H, P = v.shape[2:]
    ptr = mm._ptr
    st = fn(ctypes.byref(mm._Dims(B, S, H, G, R, N, P)), *[ptr(inp[n]) for n in si.ARG_NAMES],
            inp["chunk_size"], inp["rotary_dim_divisor"], *[ptr(t) for t in out],
            ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return st, out


@pytest.mark.parametrize("index", [2, 1])   # the timed shape (specialised kernels), tail+GQA (generic)
def test_fixed_scratch_matches_caller_workspace_twice(cuda_lib, index):
    lib = mm.load_library()
    fn = _entry(lib)
    inp = si.make_inputs(**si.WORKLOADS[index].shape_kwargs(), seed=si.WORKLOAD_SEED_BASE + index,
                         device="cuda")
    want = mm.mamba_mimo_bwd_fwd(*si.args_of(inp))
    torch.cuda.synchronize()
    for _ in range(2):
        st, got = _call_fixed(fn, inp, want)
        assert st == 0, lib.mamba_mimo_last_error().decode()
        torch.cuda.synchronize()
        for g, w in zip(got, want):
            if w is None:
                continue
            assert torch.isfinite(g.float()).all()
            assert _rel_rms(g.float(), w.float()) < TOL


def test_fixed_scratch_refuses_problems_larger_than_its_area(cuda_lib):
    lib = mm.load_library()
    fn = _entry(lib)
    wl = si.WORKLOADS[4]  # throughput shape: needs more workspace than the built-in area
    need = mm.workspace_size(wl.B, wl.S, wl.H, wl.G, wl.R, wl.N, wl.P, wl.C, wl.div, wl.reduced,
                             wl.has_z)
    assert need > FIXED_SCRATCH_BYTES
    # Every tensor pointer is NULL: the size check refuses the problem first;
    # were that check ever to come later, the NULL inputs would be refused as
    # invalid arguments (a different status) -- no kernel can be launched.
    st = fn(ctypes.byref(mm._Dims(wl.B, wl.S, wl.H, wl.G, wl.R, wl.N, wl.P)), *([None] * 17),
            wl.C, wl.div, *([None] * 5), None)
    assert st == 5
    assert "built-in scratch area" in lib.mamba_mimo_last_error().decode()


def test_fixed_scratch_matches_the_oracle(cuda_lib):
    # the tail+GQA workload (ragged last chunk, grouped heads, per-rank dout)
    # through the allocation-free entry point, element by element against the
    # CPU oracle
    lib = mm.load_library()
    fn = _entry(lib)
    inp = si.workload_inputs(1)
    dev = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    like = mm.mamba_mimo_bwd_fwd(*si.args_of(dev))
    torch.cuda.synchronize()
    st, got = _call_fixed(fn, dev, like)
    assert st == 0, lib.mamba_mimo_last_error().decode()
    torch.cuda.synchronize()
    want = oracle.bwd_fwd(*si.args_of(inp))
    for name, g in zip(oracle.OUTPUT_NAMES, got):
        w = want[name]
        assert (g is None) == (w is None), name
        if g is None:
            continue
        gn = g.float().cpu().numpy().astype(np.float64)
        assert np.all(np.isfinite(gn)), name
        err = np.sqrt(np.mean((gn - w) ** 2)) / max(np.sqrt(np.mean(w ** 2)), 1e-30)
        assert err < TOL, (name, err)
