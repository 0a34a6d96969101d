"""GPU parity of the second backward stage (mamba_mimo_bwd_bwd) against the
float64 oracle (oracle/bwd_bwd.py), through the C ABI and its binding.

Both sides read the same inputs (BF16 q/k/v/dout/trap and caches, FP32 the
rest).  The oracle computes in float64, the kernels in FP32 (products of at
most 64 terms, a reverse scan over chunks with decays below one), so every
output is held to a relative RMS error below 1e-4; DDA and DANGLES, whose
entries can sit near zero, also to a max-abs error below 1e-3 of their
largest entry (the pages' global relative criterion for those two).  Those
checks take DQ, DK and DV in FP32 (output_dtype=torch.float32); with the
default outputs (the inputs' dtype) the three must equal the FP32 results
rounded to nearest even.  FP16 and FP32 activations (dout, q, k, v, the
caches, trap) are checked the same way: both sides read the same values.
"""

import numpy as np
import pytest
import torch

import mamba_mimo_chunked_gb300 as mm
import synthetic_inputs as si
from oracle import bwd_bwd as bb

pytestmark = pytest.mark.gpu

KEYS = ("dout", "q", "k", "v", "q_bias", "k_bias", "mimo_v", "mimo_o", "d", "da_cs", "da_cs_rev", "dt",
        "trap", "segsum", "angles")


ACT = ("dout", "q", "k", "v", "trap")  # with the two caches: the activation-dtype inputs


def _problem(B, S, H, G, R, N, P, C, div=4, reduced=True, has_d=True, seed=0, caches="forward",
             act=torch.bfloat16):
    inp = si.make_inputs(B=B, S=S, H=H, G=G, R=R, N=N, P=P, C=C, div=div, reduced=reduced, has_z=False,
                         has_d=has_d, seed=seed, recipe="workload")
    for name in ACT:  # BF16 values, stored in the requested dtype (exact for FP32)
        inp[name] = inp[name].to(act)
    if caches == "forward":  # the caches a forward pass leaves (float64, stored as BF16)
        a = {k: bb._f64(inp[k]) for k in KEYS}
        nc = (S + C - 1) // C
        st = np.zeros((B, H, nc, N, P))
        qk = np.zeros((B, H, S, R, R))
        for b in range(B):
            for h in range(H):
                _, s_, q_, _ = bb.forward(a, b, h, C, div)
                st[b, h], qk[b, h] = s_, q_[:S]
        states = torch.from_numpy(st).to(act)
        qk_dot = torch.from_numpy(qk).to(act)
    else:
        states, qk_dot = si.make_stage1_caches(B=B, S=S, H=H, R=R, N=N, P=P, C=C, seed=seed + 1)
        states, qk_dot = states.to(act), qk_dot.to(act)
    args = (inp["dout"], inp["q"], inp["k"], inp["v"], inp["q_bias"], inp["k_bias"], inp["mimo_v"], states,
            qk_dot, inp["da_cs"], inp["da_cs_rev"], inp["dt"], inp["trap"], inp["segsum"], inp["angles"])
    kw = dict(mimo_o=inp["mimo_o"], d=inp["d"], chunk_size=C, rotary_dim_divisor=div)
    return args, kw


def _run_gpu(args, kw, output_dtype=torch.float32):
    dev = torch.device("cuda:0")
    g = mm.mamba_mimo_bwd_bwd(*[a.to(dev) for a in args], output_dtype=output_dtype,
                              **{k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in kw.items()})
    torch.cuda.synchronize(dev)
    return g


def _compare(got, want):
    for name in bb.OUTPUT_NAMES:
        w = want[name]
        if w is None:
            assert got[name] is None, name
            continue
        g = got[name].double().cpu().numpy()
        assert g.shape == w.shape, (name, g.shape, w.shape)
        assert np.all(np.isfinite(g)), name
        scale = np.sqrt(np.mean(w ** 2))
        err = np.sqrt(np.mean((g - w) ** 2)) / max(scale, 1e-30)
        assert err < 1e-4, f"{name}: relative RMS {err:.3e}"
        if name in ("DDA", "DANGLES"):
            m = np.max(np.abs(g - w)) / max(np.max(np.abs(w)), 1e-30)
            assert m < 1e-3, f"{name}: max-abs relative {m:.3e}"


CASES = [
    dict(B=1, S=40, H=2, G=1, R=4, N=64, P=64, C=16, div=4, reduced=True, has_d=True),    # the timed family, tail 8
    dict(B=2, S=33, H=2, G=2, R=2, N=32, P=32, C=16, div=2, reduced=False, has_d=False),  # per-rank dout, no D
    dict(B=1, S=100, H=1, G=1, R=1, N=16, P=16, C=64, div=4, reduced=True, has_d=True),   # R = 1, C*R = 64
    dict(B=1, S=20, H=2, G=1, R=8, N=32, P=16, C=8, div=4, reduced=True, has_d=True),     # R = 8
    dict(B=1, S=9, H=2, G=1, R=16, N=16, P=8, C=4, div=2, reduced=False, has_d=True),     # R = 16
    dict(B=1, S=48, H=4, G=2, R=4, N=32, P=32, C=16, div=4, reduced=True, has_d=True),    # GQA
    dict(B=1, S=1, H=1, G=1, R=4, N=64, P=64, C=16, div=4, reduced=True, has_d=True),     # one token
]

# Shapes past 64 in N, P or C*R (the persistent kernel with tiles in global
# scratch): the first stage's largest state, the op page's N = 256, C*R =
# 128 both ways, extents that are not multiples of 16, GQA.
WIDE = [
    dict(B=1, S=40, H=2, G=1, R=4, N=128, P=128, C=16, div=4, reduced=True, has_d=True),
    dict(B=1, S=70, H=1, G=1, R=2, N=256, P=64, C=32, div=2, reduced=True, has_d=True),
    dict(B=1, S=40, H=2, G=1, R=8, N=64, P=64, C=16, div=4, reduced=False, has_d=True),
    dict(B=1, S=300, H=1, G=1, R=1, N=16, P=128, C=128, div=4, reduced=True, has_d=False),
    dict(B=2, S=50, H=2, G=1, R=3, N=80, P=72, C=24, div=4, reduced=True, has_d=True),
    dict(B=1, S=33, H=4, G=2, R=4, N=128, P=96, C=16, div=2, reduced=True, has_d=True),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"S{c['S']}_R{c['R']}_N{c['N']}_C{c['C']}")
def test_parity_with_forward_caches(case):
    args, kw = _problem(**case, seed=21)
    want = bb.bwd_bwd(*args, **kw)
    _compare(_run_gpu(args, kw), want)


@pytest.mark.parametrize("act", [torch.float16, torch.float32], ids=["f16", "f32"])
@pytest.mark.parametrize("case", [CASES[0], CASES[1], CASES[5]], ids=["S40_R4", "S33_R2", "GQA"])
def test_parity_other_activation_dtypes(case, act):
    args, kw = _problem(**case, seed=29, act=act)
    want = bb.bwd_bwd(*args, **kw)
    _compare(_run_gpu(args, kw), want)


@pytest.mark.parametrize("act", [torch.float16, torch.float32], ids=["f16", "f32"])
@pytest.mark.parametrize("case", [WIDE[0], WIDE[4]], ids=["N128_P128", "N80_P72"])
def test_parity_wide_shapes_other_activation_dtypes(case, act):
    # the persistent kernel's FP16 / FP32 instantiations, with FP16 DQ / DK /
    # DV for FP16 activations (the default output dtype)
    args, kw = _problem(**case, seed=47, act=act)
    want = bb.bwd_bwd(*args, **kw)
    _compare(_run_gpu(args, kw), want)
    if act == torch.float16:
        g16 = _run_gpu(args, kw, output_dtype=None)
        for name in ("DQ", "DK", "DV"):
            assert g16[name].dtype == torch.float16
            w = want[name]
            err = np.sqrt(np.mean((g16[name].double().cpu().numpy() - w) ** 2)) / np.sqrt(np.mean(w ** 2))
            assert err < 2.0 ** -11, f"{name}: relative RMS {err:.3e}"


@pytest.mark.parametrize("case", WIDE, ids=lambda c: f"S{c['S']}_R{c['R']}_N{c['N']}_P{c['P']}_C{c['C']}")
def test_parity_wide_shapes(case):
    args, kw = _problem(**case, seed=31)
    want = bb.bwd_bwd(*args, **kw)
    _compare(_run_gpu(args, kw), want)


def test_wide_shape_more_items_than_persistent_ctas():
    # 2 x 8 heads x 24 chunks = 384 items on 152 CTAs: each CTA reuses its scratch
    args, kw = _problem(B=2, S=380, H=8, G=2, R=4, N=128, P=128, C=16, seed=37, caches="random")
    want = bb.bwd_bwd(*args, **kw)
    _compare(_run_gpu(args, kw), want)


def test_parity_timed_shape_all_heads():
    # B1 S8192 H16 R4 N=P=64 C16: given caches (seeded stand-ins); every head
    args, kw = _problem(B=1, S=8192, H=16, G=1, R=4, N=64, P=64, C=16, seed=5, caches="random")
    want = bb.bwd_bwd(*args, **kw)
    _compare(_run_gpu(args, kw), want)


def test_deterministic_and_four_launches():
    args, kw = _problem(B=1, S=200, H=2, G=1, R=4, N=64, P=64, C=16, seed=3, caches="random")
    g1 = _run_gpu(args, kw)
    assert mm.last_launch_count() == 4
    g2 = _run_gpu(args, kw)
    for name in bb.OUTPUT_NAMES:
        assert torch.equal(g1[name], g2[name]), name


@pytest.mark.parametrize("act,out", [(torch.bfloat16, None), (torch.float16, None), (torch.bfloat16, torch.float16),
                                     (torch.float32, torch.bfloat16)], ids=["bf16", "f16", "bf16_to_f16", "f32_to_bf16"])
@pytest.mark.parametrize("case", [CASES[0], CASES[1]], ids=["S40_R4", "S33_R2"])
def test_lower_precision_dq_dk_dv_are_the_rounded_fp32_results(case, act, out):
    args, kw = _problem(**case, seed=23, act=act)
    g32 = _run_gpu(args, kw)
    g16 = _run_gpu(args, kw, output_dtype=out)
    want_dt = act if out is None else out
    for name in bb.OUTPUT_NAMES:
        if g32[name] is None:
            assert g16[name] is None
        elif name in ("DQ", "DK", "DV"):
            assert g16[name].dtype == want_dt, name
            assert torch.equal(g16[name], g32[name].to(want_dt)), name
        else:
            assert g16[name].dtype == torch.float32 and torch.equal(g16[name], g32[name]), name
    # and against the oracle, within the output's rounding: at most 2^-8
    # relative per entry for BF16 (8 significant bits), 2^-11 for FP16 (11
    # bits, normal range; below it the absolute step is 2^-24)
    want = bb.bwd_bwd(*args, **kw)
    for name in ("DQ", "DK", "DV"):
        g = g16[name].double().cpu().numpy()
        err = np.sqrt(np.mean((g - want[name]) ** 2)) / np.sqrt(np.mean(want[name] ** 2))
        assert err < (2.0 ** -8 if want_dt == torch.bfloat16 else 2.0 ** -11), f"{name}: relative RMS {err:.3e}"


def test_explicit_workspace_reuse_and_non_contiguous_inputs():
    args, kw = _problem(B=1, S=40, H=2, G=1, R=4, N=64, P=64, C=16, seed=41, caches="random")
    dev = torch.device("cuda:0")
    base = _run_gpu(args, kw)
    B, S, R, G, N = args[1].shape
    H, P = args[3].shape[2], args[3].shape[3]
    nbytes = mm.bwd_bwd_workspace_size(B, S, H, G, R, N, P, 16, 4)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    dargs = [a.to(dev) for a in args]
    # the same values through non-contiguous views (the binding makes them dense)
    dargs[1] = dargs[1].transpose(1, 2).contiguous().transpose(1, 2)
    dargs[3] = dargs[3].transpose(1, 2).contiguous().transpose(1, 2)
    assert not dargs[1].is_contiguous() and not dargs[3].is_contiguous()
    dkw = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in kw.items()}
    for _ in range(2):  # one workspace, two calls
        g = mm.mamba_mimo_bwd_bwd(*dargs, output_dtype=torch.float32, workspace=ws, **dkw)
        torch.cuda.synchronize(dev)
        for name in bb.OUTPUT_NAMES:
            assert torch.equal(g[name], base[name]), name
    with pytest.raises(ValueError):
        mm.mamba_mimo_bwd_bwd(*dargs, output_dtype=torch.float32, workspace=ws[: nbytes - 256], **dkw)


def test_unaligned_activation_takes_the_element_wise_loads():
    # q 4-byte aligned but not 16-byte aligned (a valid ABI call): the
    # 16-byte vector loads of the timed-shape instantiation must not be used
    args, kw = _problem(B=1, S=40, H=2, G=1, R=4, N=64, P=64, C=16, seed=43)
    want = bb.bwd_bwd(*args, **kw)
    dev = torch.device("cuda:0")
    q = args[1].to(dev)
    buf = torch.empty(q.numel() + 2, dtype=q.dtype, device=dev)
    buf[2:].copy_(q.flatten())
    q_off = buf[2:].view(q.shape)
    assert q_off.data_ptr() % 16 == 4
    dargs = [a.to(dev) for a in args]
    dargs[1] = q_off
    g = mm.mamba_mimo_bwd_bwd(*dargs, output_dtype=torch.float32,
                              **{k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in kw.items()})
    torch.cuda.synchronize(dev)
    _compare(g, want)


def test_outside_the_envelope_raises():
    args, kw = _problem(B=1, S=16, H=1, G=1, R=2, N=512, P=16, C=16, seed=1, caches="random")
    with pytest.raises(NotImplementedError):
        _run_gpu(args, kw)
