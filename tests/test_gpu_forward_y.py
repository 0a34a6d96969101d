"""The layer's forward output y (mamba_mimo_bwd_fwd_y) against the oracle's
forward_y, on every kernel family: rel-RMS < 1e-3 like the op's outputs, and
the op's own outputs equal to those of the plain call."""

import numpy as np
import pytest
import torch

import mamba_mimo_chunked_gb300 as mm
import oracle
import synthetic_inputs as si

pytestmark = pytest.mark.gpu
TOL = 1e-3


def rel_rms(a, b):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    den = np.sqrt(np.mean(b ** 2))
    return float(np.sqrt(np.mean((a - b) ** 2)) / den) if den > 0 else float(np.sqrt(np.mean((a - b) ** 2)))


def dev_args(inp):
    return [a.to("cuda") if isinstance(a, torch.Tensor) else a for a in si.args_of(inp)]


def check(inp, tag):
    got, y = mm.mamba_mimo_bwd_fwd_with_y(*dev_args(inp))
    plain = mm.mamba_mimo_bwd_fwd(*dev_args(inp))
    torch.cuda.synchronize()
    mm.device_status()
    want = oracle.bwd_fwd(*si.args_of(inp), want_y=True)
    yg = y.float().cpu().numpy()
    assert yg.shape == want["y"].shape, tag
    assert np.all(np.isfinite(yg)), tag
    err = rel_rms(yg, want["y"])
    assert err < TOL, f"{tag}: y rel-RMS {err}"
    for a, b, name in zip(got, plain, oracle.OUTPUT_NAMES):
        if a is not None:
            assert torch.allclose(a.float(), b.float(), rtol=2e-2, atol=1e-6), (tag, name)
            assert rel_rms(a.float().cpu().numpy(), b.float().cpu().numpy()) < 1e-5, (tag, name)
    return err


def unit(**kw):
    base = dict(B=1, S=48, H=2, G=1, R=4, N=64, P=64, C=16, div=4, reduced=True, has_z=True,
                has_d=True, seed=21, recipe="workload")
    base.update(kw)
    return si.make_inputs(**base)


@pytest.fixture(autouse=True)
def _lib(cuda_lib):
    return cuda_lib


@pytest.mark.parametrize("reduced,has_z,has_d", [(True, True, True), (True, False, True),
                                                 (False, True, False), (False, False, False),
                                                 (True, True, False)])
@pytest.mark.parametrize("shape", [dict(), dict(R=8), dict(N=32, P=32), dict(R=3, N=12, P=5, C=6, div=2),
                                   dict(N=128, C=32, div=2, S=80)])
def test_forward_y_branches_and_families(reduced, has_z, has_d, shape):
    check(unit(reduced=reduced, has_z=has_z, has_d=has_d, **shape), f"{shape} {reduced}{has_z}{has_d}")


@pytest.mark.parametrize("kw", [dict(S=70), dict(S=20, B=2, H=4, G=2), dict(S=35, H=3, G=1, R=2, C=8),
                                dict(S=77, R=8, C=16, H=2, reduced=False)])
def test_forward_y_tails_batches_groups(kw):
    check(unit(**kw), str(kw))


def test_forward_y_timed_workload_sampled_heads():
    wl = si.WORKLOADS[2]
    inp = si.make_inputs(**wl.shape_kwargs(), seed=si.WORKLOAD_SEED_BASE + 2, device="cuda")
    _, y = mm.mamba_mimo_bwd_fwd_with_y(*si.args_of(inp))
    torch.cuda.synchronize()
    for (b, h) in [(0, 0), (0, 9)]:
        sl = {k: (v.cpu() if isinstance(v, torch.Tensor) else v) for k, v in si.head_slice(inp, b, h).items()}
        want = oracle.bwd_fwd(*si.args_of(sl), want_y=True)["y"]   # [1,S,1,P]
        got = y[b:b + 1, :, h:h + 1].float().cpu().numpy()
        assert rel_rms(got, want) < TOL, (b, h)
    del inp, y
    torch.cuda.empty_cache()


def test_forward_y_rejects_a_missing_buffer():
    lib = mm.load_library()
    inp = unit()
    args = dev_args(inp)
    with pytest.raises(ValueError):
        mm.mamba_mimo_bwd_fwd_with_y(*args, y=torch.empty(1, dtype=torch.bfloat16, device="cuda"))
