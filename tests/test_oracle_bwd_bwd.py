"""Pins of the second-stage oracle (oracle/bwd_bwd.py) against things other
than itself:

  * its float64 forward reproduces the first-stage oracle in exact mode
    (states and the chunk output), which tests/test_oracle_pins.py pins to
    the token recurrence, closed forms and finite differences;
  * each of the 12 gradients equals a central finite difference of that
    forward's loss L = sum dPhiO * out, taken with respect to the input (or
    intermediate) the gradient names, with the states and qk_dot recomputed
    by the forward at every perturbed point;
  * structure the reading fixes: DSSDA's masked and padded entries are 0,
    DDA lives on each chunk's last valid token, GQA gradients are per head.

Sizes are tiny (a few chunks, a ragged tail) so the finite differences run
in seconds.
"""

import numpy as np
import pytest

import oracle
import synthetic_inputs as si
from oracle import bwd_bwd as bb

KEYS = ("dout", "q", "k", "v", "q_bias", "k_bias", "mimo_v", "mimo_o", "d", "da_cs", "da_cs_rev", "dt",
        "trap", "segsum", "angles")


def _case(B=1, S=6, H=2, G=2, R=2, N=8, P=4, C=4, div=4, reduced=True, has_d=True, seed=3):
    inp = si.make_inputs(B=B, S=S, H=H, G=G, R=R, N=N, P=P, C=C, div=div, reduced=reduced, has_z=False,
                         has_d=has_d, seed=seed, recipe="workload")
    a = {k: bb._f64(inp[k]) for k in KEYS}
    return inp, a, C, div


def _pairs(a):
    return [(b, h) for b in range(a["q"].shape[0]) for h in range(a["v"].shape[2])]


def _loss(a, C, div, over=None):
    over = over or {}
    return sum(bb.forward(a, b, h, C, div, **over.get((b, h), {}))[0] for b, h in _pairs(a))


def _grads(a, C, div):
    B, S, R, G, N = a["q"].shape
    H, P = a["v"].shape[2], a["v"].shape[3]
    nc = (S + C - 1) // C
    states = np.zeros((B, H, nc, N, P))
    qk = np.zeros((B, H, S, R, R))
    for b, h in _pairs(a):
        _, st, q_, _ = bb.forward(a, b, h, C, div)
        states[b, h] = st
        qk[b, h] = q_[:S]
    return bb.bwd_bwd(a["dout"], a["q"], a["k"], a["v"], a["q_bias"], a["k_bias"], a["mimo_v"], states, qk,
                      a["da_cs"], a["da_cs_rev"], a["dt"], a["trap"], a["segsum"], a["angles"],
                      mimo_o=a["mimo_o"], d=a["d"], chunk_size=C, rotary_dim_divisor=div)


def _fd_input(a, C, div, key, eps=1e-6):
    """Central differences of L over every entry of input ``key``."""
    base = a[key]
    g = np.zeros_like(base)
    for idx in np.ndindex(base.shape):
        vals = []
        for sgn in (1.0, -1.0):
            x = base.copy()
            x[idx] += sgn * eps
            vals.append(_loss(dict(a, **{key: x}), C, div))
        g[idx] = (vals[0] - vals[1]) / (2 * eps)
    return g


def _fd_pair(a, C, div, b, h, name, base, eps=1e-6):
    """Central differences of one pair's L over an intermediate passed to the
    forward by name (gamma, factor, the chunk decay's da_cs)."""
    g = np.zeros_like(base)
    for idx in np.ndindex(base.shape):
        vals = []
        for sgn in (1.0, -1.0):
            x = base.copy()
            x[idx] += sgn * eps
            vals.append(bb.forward(a, b, h, C, div, **{name: x})[0])
        g[idx] = (vals[0] - vals[1]) / (2 * eps)
    return g


def _close(an, fd, tol=2e-6):
    scale = max(np.max(np.abs(fd)), 1e-3)
    err = np.max(np.abs(an - fd)) / scale
    assert err < tol, f"max |analytic - finite difference| / max |fd| = {err:.3e}"


@pytest.mark.parametrize("reduced", [True, False])
def test_forward_matches_first_stage_oracle(reduced):
    inp, a, C, div = _case(B=2, S=11, H=2, G=1, R=2, N=16, P=8, C=4, reduced=reduced, seed=5)
    ref = oracle.bwd_fwd(*si.args_of(inp), round_bf16=False, want_out=True)
    for b, h in _pairs(a):
        _, st, _, out = bb.forward(a, b, h, C, div)
        np.testing.assert_allclose(st, ref["states"][b, h], rtol=1e-10, atol=1e-10)
        np.testing.assert_allclose(out, ref["out"][b, h], rtol=1e-10, atol=1e-10)


@pytest.mark.parametrize("reduced,has_d,div,R", [(True, True, 4, 2), (False, True, 2, 2), (True, False, 4, 1)])
def test_input_gradients_match_finite_differences(reduced, has_d, div, R):
    _, a, C, div = _case(R=R, reduced=reduced, has_d=has_d, div=div, seed=7)
    g = _grads(a, C, div)
    B, S, R_, G, N = a["q"].shape
    H = a["v"].shape[2]
    # G == H: each q/k group is read by one head, so the per-head DQ/DK are the whole gradient
    dq = g["DQ"].reshape(B, S, R_, H, N)
    dk = g["DK"].reshape(B, S, R_, H, N)
    _close(dq, _fd_input(a, C, div, "q"))
    _close(dk, _fd_input(a, C, div, "k"))
    _close(g["DV"], _fd_input(a, C, div, "v"))
    _close(g["DMIMO_V"].sum(axis=0), _fd_input(a, C, div, "mimo_v"))
    _close(g["DANGLES"], _fd_input(a, C, div, "angles"))
    _close(g["DDA_CS_REV"], _fd_input(a, C, div, "da_cs_rev"))
    _close(g["DSSDA"], _fd_input(a, C, div, "segsum"))
    if has_d:
        _close(g["DD"].sum(axis=0), _fd_input(a, C, div, "d"))
    else:
        assert g["DD"] is None


def test_token_and_decay_gradients_match_finite_differences():
    _, a, C, div = _case(S=10, C=4, seed=11)
    g = _grads(a, C, div)
    S = a["q"].shape[1]
    nc = (S + C - 1) // C
    for b, h in _pairs(a):
        gam, fac = bb.token_scalars(a["dt"][b, h], a["trap"][b, h], S, nc * C)
        dcs = np.zeros(nc * C)
        dcs[:S] = a["da_cs"][b, h]
        _close(g["DGAMMA"][b, h], _fd_pair(a, C, div, b, h, "gamma", gam)[:S])
        _close(g["DFACTOR"][b, h], _fd_pair(a, C, div, b, h, "factor", fac)[:S])
        _close(g["DDA"][b, h], _fd_pair(a, C, div, b, h, "da_cs_dec", dcs)[:S])
    # the inter use of da_cs alone: perturb da_cs with the chunk decay held
    dec = {(b, h): {"da_cs_dec": np.pad(a["da_cs"][b, h], (0, nc * C - S))} for b, h in _pairs(a)}
    fd = np.zeros_like(a["da_cs"])
    eps = 1e-6
    for idx in np.ndindex(fd.shape):
        vals = []
        for sgn in (1.0, -1.0):
            x = a["da_cs"].copy()
            x[idx] += sgn * eps
            vals.append(_loss(dict(a, da_cs=x), C, div, dec))
        fd[idx] = (vals[0] - vals[1]) / (2 * eps)
    _close(g["DDA_CS"], fd)


def test_gqa_gradients_are_per_head():
    _, a, C, div = _case(H=4, G=2, seed=13)
    g = _grads(a, C, div)
    B, S, R, G, N = a["q"].shape
    H = a["v"].shape[2]
    per = g["DQ"].reshape(B, S, R, H, N)
    summed = np.stack([per[..., gi * (H // G):(gi + 1) * (H // G), :].sum(axis=3) for gi in range(G)], axis=3)
    _close(summed, _fd_input(a, C, div, "q"))


def test_structure_of_segsum_and_decay_gradients():
    _, a, C, div = _case(S=10, C=4, seed=17)
    g = _grads(a, C, div)
    S = a["q"].shape[1]
    nc = (S + C - 1) // C
    upper = np.triu(np.ones((C, C), dtype=bool))
    assert np.all(g["DSSDA"][..., upper] == 0.0)
    tail = np.arange(nc * C).reshape(nc, C)[-1] >= S
    assert np.all(g["DSSDA"][:, :, -1][..., tail, :] == 0.0)
    assert np.all(g["DSSDA"][:, :, -1][..., :, tail] == 0.0)
    last = [min((c + 1) * C, S) - 1 for c in range(nc)]
    off = np.ones(S, dtype=bool)
    off[last] = False
    assert np.all(g["DDA"][..., off] == 0.0)
    assert np.all(g["DDA"][..., last[-1]] == 0.0)  # the state after the last chunk is never read
    assert np.all(g["DDA"][..., last[0]] == 0.0)  # the state entering chunk 0 is zero
    assert np.all(g["DDA"][..., last[1]] != 0.0)
