"""Failure detection on the GPU without a fault: every barrier wait and the
look-back spin inside the kernels are bounded.  Test hooks make each CTA's
first barrier expect bytes that never arrive, or keep a segment from
publishing its sum; the waits run out, the kernels record a tagged error word
and return, the host reads MMBF_ERR_DEVICE_TIMEOUT, and the context stays
usable for the next call."""

import numpy as np
import pytest
import torch

import mamba_mimo_chunked_gb300 as mm
import oracle
import synthetic_inputs as si

pytestmark = pytest.mark.gpu


def tma_shape_inputs(seed):
    # N = P = 64: the kernels that load by TMA; two heads, a ragged tail
    return si.make_inputs(B=1, S=70, H=2, G=1, R=4, N=64, P=64, C=16, div=4, reduced=True,
                          has_z=True, has_d=True, seed=seed, recipe="workload")


def dev(inp):
    return [a.to("cuda") if isinstance(a, torch.Tensor) else a for a in si.args_of(inp)]


def rel_rms(a, b):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    return float(np.sqrt(np.mean((a - b) ** 2)) / np.sqrt(np.mean(b ** 2)))


@pytest.mark.parametrize("form", [0, 2])  # the single-kernel form, the two-kernel form
def test_bounded_wait_reports_timeout_and_context_recovers(cuda_lib, form):
    lib = mm.load_library()
    inp = tma_shape_inputs(5)
    lib.mamba_mimo_set_test_hooks(1 | form)
    try:
        mm.mamba_mimo_bwd_fwd(*dev(inp))
        assert mm.last_kernel_variant() == 3
        assert mm.last_plan()["single_kernel"] == (0 if form else 1)
        with pytest.raises(TimeoutError, match="bounded wait ran out .code [0-9]+: a shared-memory barrier"):
            mm.device_status()
    finally:
        lib.mamba_mimo_set_test_hooks(0)
    # the next call runs normally and is correct
    got = mm.mamba_mimo_bwd_fwd(*dev(inp))
    mm.device_status()
    want = oracle.bwd_fwd(*si.args_of(inp))
    for name in oracle.OUTPUT_NAMES:
        g = getattr(got, name)
        assert rel_rms(g.float().cpu().numpy(), want[name]) < 1e-3, name


def test_look_back_wait_reports_timeout_and_context_recovers(cuda_lib):
    # Several segments per head in the single-kernel form (B1 S2005 H16:
    # 14-chunk segments).  With hook bit 2 the first segment of every head
    # never publishes its sum: the later segments' look-back spin runs out.
    lib = mm.load_library()
    inp = si.make_inputs(B=1, S=2005, H=16, G=1, R=4, N=64, P=64, C=16, div=4, reduced=True,
                         has_z=True, has_d=True, seed=6, recipe="workload")
    lib.mamba_mimo_set_test_hooks(4)
    try:
        mm.mamba_mimo_bwd_fwd(*dev(inp))
        assert mm.last_kernel_variant() == 3
        assert mm.last_plan()["single_kernel"] == 1 and mm.last_plan()["segments"] > 1
        with pytest.raises(TimeoutError, match="bounded wait ran out .code 5: the look-back"):
            mm.device_status()
    finally:
        lib.mamba_mimo_set_test_hooks(0)
    got = mm.mamba_mimo_bwd_fwd(*dev(inp))
    mm.device_status()
    want = oracle.bwd_fwd(*si.args_of(inp))
    for name in oracle.OUTPUT_NAMES:
        g = getattr(got, name)
        assert rel_rms(g.float().cpu().numpy(), want[name]) < 1e-3, name
