"""Pins of the CPU oracle to facts that do not come from the oracle itself.

Every test here runs on CPU.  Each one is chosen so that a plausible slip in
``oracle/mmbf_oracle.c`` (a dropped term, a wrong sign, a transposed operand,
an off-by-one chunk index, a missing or extra BF16 rounding point) fails:

* bf16 rounding primitive vs torch's float -> bfloat16 conversion, and ties;
* the chunked scan (exact mode) vs an independently written token-by-token
  recurrence, with rotary done as complex multiplication and the gate
  gradients taken by torch autograd of the forward y = gated projection
  (pins the state semantics, inter/intra/diag split, trapezoid factors,
  decay bookkeeping, tail padding, GQA and the dmimo_o/dz/dmimo_z formulas);
* chunk-size invariance, the zero-decay closed form (one masked matmul),
  tail == explicitly padded run, GQA == repeated heads, mimo_v == 0;
* hand-derived BF16 worked examples for the rounding points the pages name
  (bias, same-token QK, diagonal rank order, dz rank order, factor, the
  causal A matrix, PsiV), where exact arithmetic gives a different answer;
* the BF16-vs-exact gap stays small (gross error detector).
"""

import math

import numpy as np
import pytest
import torch

import oracle
import synthetic_inputs as si

pytestmark = pytest.mark.filterwarnings("ignore::DeprecationWarning")


# ----------------------------------------------------------------------------
# helpers


def f64(t):
    return None if t is None else t.detach().to(torch.float64).numpy()


def sig(x):
    return 1.0 / (1.0 + np.exp(-x))


def dyadic_decays(B, H, S, C, seed):
    """Per-token log-decays a_t = -k/64 (k small integers) and the chunk
    quantities built from them; every cumulative sum is exact in FP32, so the
    chunked form and the token recurrence see the same numbers."""
    g = torch.Generator().manual_seed(seed)
    nc = (S + C - 1) // C
    Sp = nc * C
    a = -torch.randint(0, 9, (B, H, S), generator=g).to(torch.float32) / 64.0
    a_pad = torch.zeros((B, H, Sp))
    a_pad[:, :, :S] = a
    cs = torch.cumsum(a_pad.view(B, H, nc, C), -1)
    rev = cs[..., C - 1:C] - cs
    seg = cs[..., :, None] - cs[..., None, :]
    up = torch.triu(torch.ones(C, C, dtype=torch.bool), 1)
    return (a, cs.reshape(B, H, Sp)[:, :, :S].contiguous(), rev.reshape(B, H, Sp)[:, :, :S].contiguous(),
            seg.masked_fill(up, float("-inf")).contiguous())


def small_inputs(B, S, H, G, R, N, P, C, div, reduced, has_z, has_d, seed):
    inp = si.make_inputs(B=B, S=S, H=H, G=G, R=R, N=N, P=P, C=C, div=div, reduced=reduced,
                         has_z=has_z, has_d=has_d, seed=seed)
    a, da_cs, da_cs_rev, segsum = dyadic_decays(B, H, S, C, seed + 1000)
    inp.update(da_cs=da_cs, da_cs_rev=da_cs_rev, segsum=segsum)
    return inp, a


def run(inp, **kw):
    return oracle.bwd_fwd(*si.args_of(inp), **kw)


def token_recurrence(inp, a):
    """Independent restatement: the Mamba-3 MIMO recurrence token by token.

    h_t   = e^{a_t} h_{t-1} + factor_t * sum_r k_rot[t,r]^T psi[t,r]
    out_t = q_rot[t] (e^{a_t} h_{t-1}) + gamma_t (qh[t] kh[t]^T) psi[t] + d psi[t]
    states[c] = h_{cC-1}; rotary as complex multiplication of the pairs
    (m, N/2+m) by e^{i theta}; gamma/factor as the trapezoid weights.
    The gradients come from torch autograd of L = sum dout * y with the
    MIMO output projection y (reduced) or per-rank y (non-reduced), gated by
    silu(z * mimo_z) when z is present."""
    q, k, v = f64(inp["q"]), f64(inp["k"]), f64(inp["v"])
    B, S, R, G, N = q.shape
    H, P = v.shape[2:]
    C, div = inp["chunk_size"], inp["rotary_dim_divisor"]
    nc = (S + C - 1) // C
    w, half = N // div, N // 2
    qb, kb, mv = f64(inp["q_bias"]), f64(inp["k_bias"]), f64(inp["mimo_v"])
    ang, dt, trap = f64(inp["angles"]), f64(inp["dt"]), f64(inp["trap"])
    d = f64(inp["d"])
    a = a.to(torch.float64).numpy()
    out = np.zeros((B, H, S, R, P))
    states = np.zeros((B, H, nc, N, P))
    qk = np.zeros((B, H, S, R, R))

    def rotate(x, th):
        zc = (x[:, :w] + 1j * x[:, half:half + w]) * np.exp(1j * th)[None, :]
        y = x.copy()
        y[:, :w] = zc.real
        y[:, half:half + w] = zc.imag
        return y

    for b in range(B):
        for h in range(H):
            g = h // (H // G)
            st = np.zeros((N, P))
            for t in range(S):
                if t % C == 0:
                    states[b, h, t // C] = st
                qh = q[b, t, :, g, :] + qb[h]
                kh = k[b, t, :, g, :] + kb[h]
                qk[b, h, t] = qh @ kh.T
                qr, kr = rotate(qh, ang[b, t, h]), rotate(kh, ang[b, t, h])
                psi = v[b, t, h][None, :] * mv[h]
                gam = dt[b, h, t] * sig(trap[b, h, t])
                sh = dt[b, h, t + 1] * (1.0 - sig(trap[b, h, t + 1])) if t + 1 < S else 0.0
                dec = math.exp(a[b, h, t]) * st
                o = qr @ dec + gam * (qk[b, h, t] @ psi)
                if d is not None:
                    o = o + d[h] * psi
                out[b, h, t] = o
                st = dec + (gam + sh) * (kr.T @ psi)

    res = {"out": out, "states": states, "qk_dot": qk, "dmimo_o": None, "dz": None, "dmimo_z": None}
    reduced, has_z = inp["mimo_o"] is not None, inp["z"] is not None
    if not (reduced or has_z):
        return res
    o_t = torch.tensor(out)
    dout = torch.tensor(f64(inp["dout"]))
    gate = 1.0
    if has_z:
        z = torch.tensor(f64(inp["z"]), requires_grad=True)
        mz = torch.tensor(np.broadcast_to(f64(inp["mimo_z"]), (B, H, R, P)).copy(), requires_grad=True)
        pz = z.permute(0, 2, 1, 3)[:, :, :, None, :] * mz[:, :, None]
        gate = pz * torch.sigmoid(pz)
    if reduced:
        mo = torch.tensor(np.broadcast_to(f64(inp["mimo_o"]), (B, H, R, P)).copy(), requires_grad=True)
        y = (mo[:, :, None] * o_t * gate).sum(3)              # [B,H,S,P]
        L = (dout.permute(0, 2, 1, 3) * y).sum()
    else:
        y = o_t * gate                                        # [B,H,S,R,P]
        L = (dout.permute(0, 3, 1, 2, 4) * y).sum()
    L.backward()
    if reduced:
        res["dmimo_o"] = mo.grad.numpy()
    if has_z:
        res["dz"] = z.grad.numpy()
        res["dmimo_z"] = mz.grad.numpy()
    return res


def rel_max(a, b):
    a, b = np.asarray(a), np.asarray(b)
    return float(np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300))


def rel_rms(a, b):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    return float(np.sqrt(np.mean((a - b) ** 2)) / max(np.sqrt(np.mean(b ** 2)), 1e-300))


# ----------------------------------------------------------------------------
# the BF16 rounding primitive


def test_bf16_rounding_matches_torch_and_ties():
    g = torch.Generator().manual_seed(7)
    x = torch.randn(20000, generator=g) * torch.exp2(torch.randint(-140, 120, (20000,), generator=g).float())
    x = torch.cat([x, torch.tensor([0.0, -0.0, 1e-45, -3e-39, 3.38e38, 3.3895e38, 3.4e38, 1.0 + 2 ** -8])])
    want = x.to(torch.bfloat16).to(torch.float64).numpy()
    got = np.array([oracle.bf16_nearest(float(v)) for v in x.tolist()])
    np.testing.assert_array_equal(got, want)
    # ties go to the even neighbour; 2^-8 is half an ulp at 1.0
    assert oracle.bf16_nearest(1.0 + 2 ** -8) == 1.0
    assert oracle.bf16_nearest(1.0 + 3 * 2 ** -8) == 1.0 + 2 ** -6
    assert oracle.bf16_nearest(-(1.0 + 2 ** -8 + 2 ** -30)) == -(1.0 + 2 ** -7)


# ----------------------------------------------------------------------------
# exact mode against the token recurrence (+ autograd gradients)

RECURRENCE_CASES = [
    # B, S, H, G, R, N, P, C, div, reduced, has_z, has_d
    (1, 37, 2, 1, 2, 8, 6, 8, 4, True, True, True),      # tail chunk, all branches
    (2, 20, 4, 2, 3, 12, 5, 6, 2, False, True, False),   # GQA, odd R, div 2, per-rank dout
    (1, 16, 1, 1, 1, 4, 3, 16, 4, True, False, True),    # R = 1, single chunk, no Z
    (1, 9, 2, 2, 4, 8, 8, 4, 4, False, False, False),    # only states + qk_dot
    (1, 24, 2, 1, 4, 16, 8, 4, 4, True, True, False),
]


@pytest.mark.parametrize("case", RECURRENCE_CASES)
def test_exact_oracle_equals_token_recurrence(case):
    inp, a = small_inputs(*case, seed=11)
    got = run(inp, round_bf16=False, want_out=True)
    ref = token_recurrence(inp, a)
    S = inp["q"].shape[1]
    assert rel_max(got["out"][:, :, :S], ref["out"]) < 1e-11
    assert rel_max(got["states"], ref["states"]) < 1e-11
    assert rel_max(got["qk_dot"], ref["qk_dot"]) < 1e-12
    for name in ("dmimo_o", "dz", "dmimo_z"):
        assert (got[name] is None) == (ref[name] is None), name
        if ref[name] is not None:
            assert rel_max(got[name], ref[name]) < 1e-10, name


def test_states_zero_at_first_chunk_and_entering_semantics():
    inp, a = small_inputs(1, 12, 1, 1, 2, 4, 4, 4, 4, True, True, True, seed=3)
    got = run(inp, round_bf16=True)
    assert np.all(got["states"][:, :, 0] == 0.0)
    assert np.any(got["states"][:, :, 1] != 0.0)


# ----------------------------------------------------------------------------
# chunk-size invariance, zero-decay closed form, tail, GQA, degenerate cases


@pytest.mark.parametrize("S", [16, 13])
def test_chunk_size_invariance(S):
    base, _ = small_inputs(1, S, 2, 1, 2, 8, 4, 1, 4, True, True, True, seed=5)
    g = torch.Generator().manual_seed(99)
    a = -torch.randint(0, 9, (1, 2, S), generator=g).float() / 64.0
    results = {}
    for C in (1, 2, 4, 8):
        nc = (S + C - 1) // C
        a_pad = torch.zeros((1, 2, nc * C))
        a_pad[:, :, :S] = a
        cs = torch.cumsum(a_pad.view(1, 2, nc, C), -1)
        inp = dict(base)
        inp["chunk_size"] = C
        inp["da_cs"] = cs.reshape(1, 2, -1)[:, :, :S].contiguous()
        inp["da_cs_rev"] = (cs[..., C - 1:C] - cs).reshape(1, 2, -1)[:, :, :S].contiguous()
        inp["segsum"] = (cs[..., :, None] - cs[..., None, :]).masked_fill(
            torch.triu(torch.ones(C, C, dtype=torch.bool), 1), float("-inf")).contiguous()
        results[C] = run(inp, round_bf16=False)
    r1 = results[1]
    for C, r in results.items():
        for name in ("qk_dot", "dz", "dmimo_o", "dmimo_z"):
            assert rel_max(r[name], r1[name]) < 1e-11, (C, name)
        for c in range(r["states"].shape[2]):
            assert rel_max(r["states"][:, :, c], r1["states"][:, :, c * C]) < 1e-11 or \
                np.all(r1["states"][:, :, c * C] == 0)


def test_zero_decay_is_one_masked_matmul():
    """a = 0: the scan is causal linear attention over the whole sequence."""
    B, S, H, G, R, N, P, C = 1, 14, 1, 1, 2, 8, 4, 4
    inp = si.make_inputs(B=B, S=S, H=H, G=G, R=R, N=N, P=P, C=C, div=2, reduced=True,
                         has_z=False, has_d=True, seed=21)
    nc = (S + C - 1) // C
    inp["da_cs"] = torch.zeros((B, H, S))
    inp["da_cs_rev"] = torch.zeros((B, H, S))
    inp["segsum"] = torch.zeros((B, H, nc, C, C))
    got = run(inp, round_bf16=False, want_out=True)["out"][0, 0, :S]      # [S,R,P]
    q, k, v = (f64(inp[n])[0, :, :, 0] for n in ("q", "k")), None, f64(inp["v"])[0, :, 0]
    q, k = f64(inp["q"])[0, :, :, 0], f64(inp["k"])[0, :, :, 0]
    qh, kh = q + f64(inp["q_bias"])[0], k + f64(inp["k_bias"])[0]
    th = f64(inp["angles"])[0, :, 0]                                      # [S, N/2]
    cs, sn = np.cos(th)[:, None], np.sin(th)[:, None]
    w = N // 2
    qr = np.concatenate([cs * qh[..., :w] - sn * qh[..., w:], sn * qh[..., :w] + cs * qh[..., w:]], -1)
    kr = np.concatenate([cs * kh[..., :w] - sn * kh[..., w:], sn * kh[..., :w] + cs * kh[..., w:]], -1)
    dt, trap = f64(inp["dt"])[0, 0], f64(inp["trap"])[0, 0]
    gam = dt * sig(trap)
    fac = gam + np.append(dt[1:] * sig(-trap[1:]), 0.0)
    psi = v[:, None, :] * f64(inp["mimo_v"])[0][None]                     # [S,R,P]
    tok = np.repeat(np.arange(S), R)
    mask = tok[:, None] > tok[None, :]
    Qf, Kf, Pf = qr.reshape(S * R, N), (kr * fac[:, None, None]).reshape(S * R, N), psi.reshape(S * R, P)
    same = tok[:, None] == tok[None, :]
    qkd = (qh.reshape(S * R, N) @ kh.reshape(S * R, N).T) * same * np.repeat(gam, R)[:, None]
    want = (np.where(mask, Qf @ Kf.T, 0.0) + qkd) @ Pf + f64(inp["d"])[0] * Pf
    assert rel_max(got.reshape(S * R, P), want) < 1e-11


@pytest.mark.parametrize("round_bf16", [False, True])
def test_tail_equals_explicitly_padded_run(round_bf16):
    B, S, H, G, R, N, P, C = 1, 37, 2, 1, 2, 8, 4, 8
    Sp = 40
    inp, _ = small_inputs(B, S, H, G, R, N, P, C, 4, True, True, True, seed=8)
    pad = dict(inp)
    for name, dim in (("dout", 1), ("q", 1), ("k", 1), ("v", 1), ("z", 1), ("angles", 1), ("dt", 2),
                      ("trap", 2), ("da_cs_rev", 2)):
        x = inp[name]
        shape = list(x.shape)
        shape[dim] = Sp - S
        pad[name] = torch.cat([x, torch.zeros(shape, dtype=x.dtype)], dim)
    last = inp["da_cs"][:, :, -1:]
    pad["da_cs"] = torch.cat([inp["da_cs"], last.expand(B, H, Sp - S)], 2)   # edge-extended cumsum
    r1 = run(inp, round_bf16=round_bf16)
    r2 = run(pad, round_bf16=round_bf16)
    np.testing.assert_array_equal(r1["states"], r2["states"])
    np.testing.assert_array_equal(r1["qk_dot"], r2["qk_dot"][:, :, :S])
    np.testing.assert_array_equal(r1["dz"], r2["dz"][:, :S])
    np.testing.assert_array_equal(r1["dmimo_o"], r2["dmimo_o"])
    np.testing.assert_array_equal(r1["dmimo_z"], r2["dmimo_z"])


@pytest.mark.parametrize("round_bf16", [False, True])
def test_gqa_equals_repeated_groups(round_bf16):
    B, S, H, G, R, N, P, C = 2, 20, 4, 2, 2, 8, 4, 8
    inp, _ = small_inputs(B, S, H, G, R, N, P, C, 4, True, True, True, seed=12)
    rep = dict(inp)
    rep["q"] = inp["q"].repeat_interleave(H // G, dim=3).contiguous()
    rep["k"] = inp["k"].repeat_interleave(H // G, dim=3).contiguous()
    r1, r2 = run(inp, round_bf16=round_bf16), run(rep, round_bf16=round_bf16)
    for name in oracle.OUTPUT_NAMES:
        np.testing.assert_array_equal(r1[name], r2[name])


@pytest.mark.parametrize("round_bf16", [False, True])
def test_zero_value_projection_gives_zero_state_and_gradients(round_bf16):
    inp, _ = small_inputs(1, 20, 2, 1, 3, 8, 4, 8, 4, True, True, True, seed=4)
    inp["mimo_v"] = torch.zeros_like(inp["mimo_v"])
    r = run(inp, round_bf16=round_bf16, want_out=True)
    for name in ("states", "dz", "dmimo_o", "dmimo_z", "out"):
        assert np.all(r[name] == 0.0), name
    assert np.any(r["qk_dot"] != 0.0)


def test_bf16_mode_is_close_to_exact_mode():
    """The rounding points perturb each output by well under a few percent
    (rel. RMS); a missing or doubled term would not."""
    inp = si.workload_inputs(0)
    rb, re_ = run(inp, round_bf16=True), run(inp, round_bf16=False)
    for name in oracle.OUTPUT_NAMES:
        e = rel_rms(rb[name], re_[name])
        assert 1e-5 < e < 2e-2, (name, e)


# ----------------------------------------------------------------------------
# BF16 worked examples derived by hand.  Each sets up a B=S=H=G=1-ish problem
# whose intermediate lands on or near a BF16 tie, so that the pages' rounding
# point changes the answer relative to exact arithmetic.


def tiny_problem(S=1, R=1, N=2, P=2, C=1, div=2, reduced=True, has_z=False):
    bf16, f32 = torch.bfloat16, torch.float32
    nc = (S + C - 1) // C
    return {
        "dout": torch.zeros((1, S, 1, P) if reduced else (1, S, R, 1, P), dtype=bf16),
        "q": torch.zeros((1, S, R, 1, N), dtype=bf16), "k": torch.zeros((1, S, R, 1, N), dtype=bf16),
        "v": torch.zeros((1, S, 1, P), dtype=bf16),
        "q_bias": torch.zeros((1, R, N), dtype=f32), "k_bias": torch.zeros((1, R, N), dtype=f32),
        "mimo_v": torch.ones((1, R, P), dtype=f32),
        "mimo_o": torch.ones((1, R, P), dtype=f32) if reduced else None,
        "z": torch.zeros((1, S, 1, P), dtype=bf16) if has_z else None,
        "mimo_z": torch.ones((1, R, P), dtype=f32) if has_z else None,
        "angles": torch.zeros((1, S, 1, N // div), dtype=f32),
        "da_cs": torch.zeros((1, 1, S), dtype=f32), "da_cs_rev": torch.zeros((1, 1, S), dtype=f32),
        "dt": torch.zeros((1, 1, S), dtype=f32), "trap": torch.zeros((1, 1, S), dtype=bf16),
        "d": None, "segsum": torch.zeros((1, 1, nc, C, C), dtype=f32),
        "chunk_size": C, "rotary_dim_divisor": div,
    }


def both(inp):
    return run(inp, round_bf16=True), run(inp, round_bf16=False)


def test_worked_example_same_token_qk_rounds_to_even():
    # q = (1, 1), k = (1, 2^-8): q.k = 1 + 2^-8, half an ulp above 1.0 -> 1.0
    x = tiny_problem()
    x["q"][0, 0, 0, 0] = torch.tensor([1.0, 1.0])
    x["k"][0, 0, 0, 0] = torch.tensor([1.0, 2 ** -8])
    rb, re_ = both(x)
    assert rb["qk_dot"][0, 0, 0, 0, 0] == 1.0
    assert re_["qk_dot"][0, 0, 0, 0, 0] == 1.0 + 2 ** -8


def test_worked_example_bias_is_rounded_before_the_add():
    # bias = 2^-8 (1 + 2^-9) rounds to 2^-8 first; 1 + 2^-8 is then a tie -> 1.0.
    # Rounding only the sum would give 1 + 2^-7; no rounding 1 + 2^-8 + 2^-17.
    x = tiny_problem()
    x["q"][0, 0, 0, 0] = torch.tensor([1.0, 0.0])
    x["k"][0, 0, 0, 0] = torch.tensor([1.0, 0.0])
    x["q_bias"][0, 0] = torch.tensor([2 ** -8 * (1 + 2 ** -9), 0.0])
    rb, re_ = both(x)
    assert rb["qk_dot"][0, 0, 0, 0, 0] == 1.0
    assert re_["qk_dot"][0, 0, 0, 0, 0] == 1.0 + 2 ** -8 + 2 ** -17


def test_worked_example_diagonal_is_summed_rank_by_rank_in_bf16():
    # R = 3, qk[0, r] = 1 for all r, PsiV = (1, 2^-8, 2^-8), gamma = 2 * sigmoid(0) = 1.
    # Rank-ordered BF16 sum: 1 -> bf16(1 + 2^-8) = 1 -> bf16(1 + 2^-8) = 1.
    # A single FP32 dot would give 1 + 2^-7.  out[0,0,:] = diag; with dout = 1
    # and no Z, dmimo_o[0, :] = out[0, 0, :].
    x = tiny_problem(R=3, P=1)
    x["q"][0, 0, :, 0] = torch.tensor([1.0, 0.0])
    x["k"][0, 0, :, 0] = torch.tensor([1.0, 0.0])
    x["v"][0, 0, 0] = 1.0
    x["mimo_v"][0, :, 0] = torch.tensor([1.0, 2 ** -8, 2 ** -8])
    x["dt"][0, 0, 0] = 2.0
    x["dout"][0, 0, 0] = 1.0
    rb, re_ = both(x)
    assert rb["dmimo_o"][0, 0, 0, 0] == 1.0
    assert re_["dmimo_o"][0, 0, 0, 0] == pytest.approx(1.0 + 2 ** -7, abs=1e-15)


def test_worked_example_dz_is_summed_rank_by_rank_in_bf16():
    # out[0, r, 0] = 1 for every rank (qk[r,0] = 1, PsiV[0] = 1, others 0,
    # gamma = 1); dout = 1, mimo_o = 2 -> pre = 2; z = 0 -> sigmoid = 1/2,
    # silu' = 1/2 -> gzp = 1.  mimo_z = (1, 2^-8, 2^-8): the rank-ordered
    # BF16 sum stays at 1.0, exact arithmetic gives 1 + 2^-7.
    x = tiny_problem(R=3, P=1, has_z=True)
    x["q"][0, 0, :, 0] = torch.tensor([1.0, 0.0])
    x["k"][0, 0, 0, 0] = torch.tensor([1.0, 0.0])
    x["v"][0, 0, 0] = 1.0
    x["mimo_v"][0, :, 0] = torch.tensor([1.0, 0.0, 0.0])
    x["dt"][0, 0, 0] = 2.0
    x["dout"][0, 0, 0] = 1.0
    x["mimo_o"][0, :, 0] = 2.0
    x["mimo_z"][0, :, 0] = torch.tensor([1.0, 2 ** -8, 2 ** -8])
    rb, re_ = both(x)
    assert rb["dz"][0, 0, 0, 0] == 1.0
    assert re_["dz"][0, 0, 0, 0] == pytest.approx(1.0 + 2 ** -7, abs=1e-15)
    assert rb["dmimo_z"][0, 0, 0, 0] == 0.0          # z = 0


def test_worked_example_factor_is_rounded():
    # gamma[0] = 2 * sigmoid(0) = 1; shifted[0] = bf16(2^-7 * sigmoid(0)) = 2^-8;
    # factor = bf16(1 + 2^-8) = 1 (tie to even).  k = (1 + 2^-7, 0), so
    # k_scaled = 1 + 2^-7 with the rounded factor but bf16((1 + 2^-7)(1 + 2^-8))
    # = 1 + 2^-6 without it.  states[1] = k_state^T PsiV with PsiV = (1, 1).
    x = tiny_problem(S=2, C=1)
    x["k"][0, 0, 0, 0] = torch.tensor([1.0 + 2 ** -7, 0.0])
    x["v"][0, 0, 0] = torch.tensor([1.0, 1.0])
    x["dt"][0, 0] = torch.tensor([2.0, 2 ** -7])
    rb, re_ = both(x)
    np.testing.assert_array_equal(rb["states"][0, 0, 1], [[1.0 + 2 ** -7] * 2, [0.0, 0.0]])
    ex = (1 + 2 ** -7) * (1 + 2 ** -8)
    np.testing.assert_allclose(re_["states"][0, 0, 1], [[ex, ex], [0.0, 0.0]], rtol=0, atol=1e-15)
    assert np.all(rb["states"][0, 0, 0] == 0.0)


def test_worked_example_causal_matrix_is_rounded():
    # Two tokens in one chunk, R = 1.  A[1,0] = bf16(q_1 . ks_0 * e^0) with
    # q_1 = (1, 1), ks_0 = k_0 * factor_0 = (1, 2^-8): 1 + 2^-8 -> 1.0.
    # PsiV_0 = 1 + 2^-7, PsiV_1 = 0 and dt_1 = 0 (no own diagonal for token 1):
    # out[1] = bf16(A[1,0] PsiV_0) = 1 + 2^-7, but 1 + 2^-6 if A were not
    # rounded.  With dout = (0, 1) and no Z, dmimo_o = out[1].
    x = tiny_problem(S=2, C=2, P=1)
    x["q"][0, 1, 0, 0] = torch.tensor([1.0, 1.0])
    x["k"][0, 0, 0, 0] = torch.tensor([1.0, 2 ** -8])
    x["v"][0, 0, 0, 0] = 1.0 + 2 ** -7
    x["dt"][0, 0] = torch.tensor([2.0, 0.0])
    x["dout"][0, 1, 0, 0] = 1.0
    rb, re_ = both(x)
    assert rb["dmimo_o"][0, 0, 0, 0] == 1.0 + 2 ** -7
    assert re_["dmimo_o"][0, 0, 0, 0] == pytest.approx((1.0 + 2 ** -8) * (1 + 2 ** -7), abs=1e-15)


def test_worked_example_psi_uses_rounded_mimo_v():
    # mimo_v = 1 + 2^-8 rounds to 1.0 (tie to even) before the product, so
    # PsiV = bf16((1 + 2^-7) * 1) = 1 + 2^-7; the unrounded product
    # (1 + 2^-7)(1 + 2^-8) would round to 1 + 2^-6.  Observed through the
    # diagonal (qk = 1, gamma = 1): out = PsiV = dmimo_o with dout = 1.
    x = tiny_problem(P=1)
    x["q"][0, 0, 0, 0] = torch.tensor([1.0, 0.0])
    x["k"][0, 0, 0, 0] = torch.tensor([1.0, 0.0])
    x["v"][0, 0, 0] = 1.0 + 2 ** -7
    x["mimo_v"][0, 0, 0] = 1.0 + 2 ** -8
    x["dt"][0, 0, 0] = 2.0
    x["dout"][0, 0, 0] = 1.0
    rb, re_ = both(x)
    assert rb["dmimo_o"][0, 0, 0, 0] == 1.0 + 2 ** -7
    assert re_["dmimo_o"][0, 0, 0, 0] == pytest.approx((1.0 + 2 ** -7) * (1 + 2 ** -8), abs=1e-15)


def test_qk_dot_layout_is_token_rout_rin():
    # q[t,r] = (2^(4r + 16 (t%2) - 40), 0), k[t,s] = (2^s, 0): every product is a
    # distinct power of two, exact in BF16, so any transposition shows.
    S, R = 4, 4
    x = tiny_problem(S=S, R=R, C=2)
    for t in range(S):
        for r in range(R):
            x["q"][0, t, r, 0, 0] = 2.0 ** (4 * r + 16 * (t % 2) - 40)
            x["k"][0, t, r, 0, 0] = 2.0 ** r
    rb = run(x, round_bf16=True)
    for t in range(S):
        for r in range(R):
            for s in range(R):
                assert rb["qk_dot"][0, 0, t, r, s] == 2.0 ** (4 * r + 16 * (t % 2) - 40 + s)


def test_worked_example_qk_dot_uses_unrotated_q_and_k():
    # angle 1 rad on the single rotary pair: q = k = (1, 0).  Un-rotated q.k = 1.
    # Rotated, bf16(cos 1)^2 + bf16(sin 1)^2 = 0.5390625^2 + 0.83984375^2
    # = 0.99591064..., which would round to 0.99609375.
    x = tiny_problem()
    x["q"][0, 0, 0, 0] = torch.tensor([1.0, 0.0])
    x["k"][0, 0, 0, 0] = torch.tensor([1.0, 0.0])
    x["angles"][0, 0, 0, 0] = 1.0
    rb = run(x, round_bf16=True)
    assert rb["qk_dot"][0, 0, 0, 0, 0] == 1.0


def test_worked_example_out_is_rounded():
    # out = bf16(diag + d PsiV) = bf16(1 + 2^-8) = 1.0 (tie to even); exact 1 + 2^-8.
    x = tiny_problem(P=1)
    x["q"][0, 0, 0, 0] = torch.tensor([1.0, 0.0])
    x["k"][0, 0, 0, 0] = torch.tensor([1.0, 0.0])
    x["v"][0, 0, 0] = 1.0
    x["dt"][0, 0, 0] = 2.0
    x["d"] = torch.tensor([2 ** -8])
    x["dout"][0, 0, 0] = 1.0
    rb, re_ = both(x)
    assert rb["dmimo_o"][0, 0, 0, 0] == 1.0
    assert re_["dmimo_o"][0, 0, 0, 0] == pytest.approx(1.0 + 2 ** -8, abs=1e-15)


def test_worked_example_diagonal_times_gamma_is_rounded():
    # PsiV = 1 + 2^-7, qk = 1, gamma = bf16(2 - 2^-7) * sigmoid(0) = 1 - 2^-8:
    # diag = bf16((1 + 2^-7)(1 - 2^-8)) = bf16(1 + 2^-8 - 2^-15) = 1.0.
    # d = 2^-9 adds 2^-9 (1 + 2^-7): out = bf16(1 + 2^-9 + 2^-16) = 1.0, while an
    # unrounded diag gives bf16(1 + 2^-8 + 2^-9 + ...) = 1 + 2^-7.
    x = tiny_problem(P=1)
    x["q"][0, 0, 0, 0] = torch.tensor([1.0, 0.0])
    x["k"][0, 0, 0, 0] = torch.tensor([1.0, 0.0])
    x["v"][0, 0, 0] = 1.0 + 2 ** -7
    x["dt"][0, 0, 0] = 2.0 - 2 ** -7
    x["d"] = torch.tensor([2 ** -9])
    x["dout"][0, 0, 0] = 1.0
    rb, re_ = both(x)
    assert rb["dmimo_o"][0, 0, 0, 0] == 1.0
    want = (1 + 2 ** -7) * (1 - 2 ** -8) + 2 ** -9 * (1 + 2 ** -7)
    assert re_["dmimo_o"][0, 0, 0, 0] == pytest.approx(want, abs=1e-15)


def test_worked_example_k_state_is_rounded():
    # One chunk of two tokens, then a third token.  ks_0 = (2, 0) (factor 2),
    # ks_1 = (1, 0); da_cs_rev = (ln(1 + 0.45 * 2^-7), 0).  k_state_0 =
    # bf16(2 e) = 2.0 (0.45 ulp above 2), so with PsiV = (0.5, -1) the state
    # entering chunk 1 cancels to 0; unrounded it is e - 1 = 0.0035...
    x = tiny_problem(S=3, C=2, P=1)
    x["k"][0, 0, 0, 0] = torch.tensor([1.0, 0.0])
    x["k"][0, 1, 0, 0] = torch.tensor([1.0, 0.0])
    x["v"][0, :2, 0, 0] = torch.tensor([0.5, -1.0])
    x["dt"][0, 0] = torch.tensor([2.0, 2.0, 0.0])
    dar = torch.tensor([math.log(1 + 0.45 * 2 ** -7), 0.0, 0.0], dtype=torch.float32)
    x["da_cs_rev"][0, 0] = dar
    rb, re_ = both(x)
    assert rb["states"][0, 0, 1, 0, 0] == 0.0
    assert re_["states"][0, 0, 1, 0, 0] == pytest.approx(math.exp(float(dar[0])) - 1.0, abs=1e-12)


def test_worked_example_rotary_is_rounded():
    # Token 1 has angle 1 rad and q = (1, 0): q_rot = (bf16(cos 1), bf16(sin 1))
    # = (0.5390625, 0.83984375).  ks_0 = (1, 1).  A[1,0] = bf16(1.37890625)
    # = 1.375 (a tie, to even); unrounded rotation gives cos 1 + sin 1 =
    # 1.38177... -> 1.3828125.  out[1] = A[1,0] PsiV_0 with PsiV_0 = 1.
    x = tiny_problem(S=2, C=2, P=1)
    x["q"][0, 1, 0, 0] = torch.tensor([1.0, 0.0])
    x["k"][0, 0, 0, 0] = torch.tensor([1.0, 1.0])
    x["angles"][0, 1, 0, 0] = 1.0
    x["v"][0, 0, 0, 0] = 1.0
    x["dt"][0, 0] = torch.tensor([2.0, 0.0])
    x["dout"][0, 1, 0, 0] = 1.0
    rb, re_ = both(x)
    assert rb["dmimo_o"][0, 0, 0, 0] == 1.375
    assert re_["dmimo_o"][0, 0, 0, 0] == pytest.approx(math.cos(1.0) + math.sin(1.0), abs=1e-14)


def test_worked_example_pre_gate_gradient_is_rounded():
    # out = 1; dout = 1 + 2^-7; mimo_o = 1 + 2^-8 rounds to 1 -> pre = 1 + 2^-7
    # (unrounded chain: bf16((1 + 2^-7)(1 + 2^-8)) = 1 + 2^-6).  mimo_z = 0
    # makes pz = 0, so gzp = pre / 2 and dmimo_z = gzp z = pre with z = 2.
    x = tiny_problem(P=1, has_z=True)
    x["q"][0, 0, 0, 0] = torch.tensor([1.0, 0.0])
    x["k"][0, 0, 0, 0] = torch.tensor([1.0, 0.0])
    x["v"][0, 0, 0] = 1.0
    x["dt"][0, 0, 0] = 2.0
    x["dout"][0, 0, 0] = 1.0 + 2 ** -7
    x["mimo_o"][0, 0, 0] = 1.0 + 2 ** -8
    x["mimo_z"][0, 0, 0] = 0.0
    x["z"][0, 0, 0] = 2.0
    rb, re_ = both(x)
    assert rb["dmimo_z"][0, 0, 0, 0] == 1.0 + 2 ** -7
    assert re_["dmimo_z"][0, 0, 0, 0] == pytest.approx((1 + 2 ** -7) * (1 + 2 ** -8), abs=1e-15)
    assert rb["dmimo_o"][0, 0, 0, 0] == 0.0           # silu(0) = 0


def test_worked_example_inter_uses_rounded_state():
    # Chunk 0: state = k_state^T PsiV = (1 + 2^-7)^2 = 1 + 2^-6 + 2^-14, so
    # states[1] = 1 + 2^-6.  Chunk 1: q = (1, 0), inter = bf16(state) = 1 + 2^-6,
    # d PsiV_1 = -(1 + 2^-6): out_1 = 0 with the rounded state, 2^-14 without.
    x = tiny_problem(S=2, C=1, P=1)
    x["k"][0, 0, 0, 0] = torch.tensor([1.0 + 2 ** -7, 0.0])
    x["v"][0, :, 0, 0] = torch.tensor([1.0 + 2 ** -7, -1.0])
    x["q"][0, 1, 0, 0] = torch.tensor([1.0, 0.0])
    x["dt"][0, 0] = torch.tensor([2.0, 0.0])
    x["d"] = torch.tensor([1.0 + 2 ** -6])
    x["dout"][0, 1, 0, 0] = 1.0
    rb, re_ = both(x)
    assert rb["states"][0, 0, 1, 0, 0] == 1.0 + 2 ** -6
    assert rb["dmimo_o"][0, 0, 0, 0] == 0.0
    assert re_["dmimo_o"][0, 0, 0, 0] == pytest.approx(2 ** -14, abs=1e-16)


def test_worked_example_gamma_uses_bf16_dt():
    # dt = 2 + 2^-7 is a BF16 tie and loads as 2.0: gamma = 1 and
    # diag = bf16((1 + 2^-7) * 1); with dt unrounded gamma = 1 + 2^-8 and
    # diag = bf16((1 + 2^-7)(1 + 2^-8)) = 1 + 2^-6.
    x = tiny_problem(P=1)
    x["q"][0, 0, 0, 0] = torch.tensor([1.0, 0.0])
    x["k"][0, 0, 0, 0] = torch.tensor([1.0, 0.0])
    x["v"][0, 0, 0] = 1.0 + 2 ** -7
    x["dt"][0, 0, 0] = 2.0 + 2 ** -7
    x["dout"][0, 0, 0] = 1.0
    rb, re_ = both(x)
    assert rb["dmimo_o"][0, 0, 0, 0] == 1.0 + 2 ** -7
    assert re_["dmimo_o"][0, 0, 0, 0] == pytest.approx((1 + 2 ** -7) * (1 + 2 ** -8), abs=1e-15)


def test_worked_example_k_bias_is_rounded_before_the_add():
    # mirror of the q_bias example on the k side
    x = tiny_problem()
    x["q"][0, 0, 0, 0] = torch.tensor([1.0, 0.0])
    x["k"][0, 0, 0, 0] = torch.tensor([1.0, 0.0])
    x["k_bias"][0, 0] = torch.tensor([2 ** -8 * (1 + 2 ** -9), 0.0])
    rb, re_ = both(x)
    assert rb["qk_dot"][0, 0, 0, 0, 0] == 1.0
    assert re_["qk_dot"][0, 0, 0, 0, 0] == 1.0 + 2 ** -8 + 2 ** -17


def test_worked_example_diagonal_product_is_rounded_per_rank():
    # qk[0,:] = (1, 1.140625), PsiV = (1 + 2^-7, 1.75 * 2^-9), gamma = 1.
    # Rank 1's product 1.140625 * 1.75 * 2^-9 = 2^-8 - 2^-17 rounds to 2^-8, so
    # the running sum hits the tie 1 + 2^-7 + 2^-8 and goes to even 1 + 2^-6;
    # with an unrounded product it stays below the tie: 1 + 2^-7.
    x = tiny_problem(R=2, P=1)
    x["q"][0, 0, 0, 0] = torch.tensor([1.0, 0.0])
    x["k"][0, 0, 0, 0] = torch.tensor([1.0, 0.0])
    x["k"][0, 0, 1, 0] = torch.tensor([1.140625, 0.0])
    x["v"][0, 0, 0] = 1.0
    x["mimo_v"][0, :, 0] = torch.tensor([1.0 + 2 ** -7, 1.75 * 2 ** -9])
    x["dt"][0, 0, 0] = 2.0
    x["dout"][0, 0, 0] = 1.0
    rb, re_ = both(x)
    assert rb["dmimo_o"][0, 0, 0, 0] == 1.0 + 2 ** -6
    assert re_["dmimo_o"][0, 0, 0, 0] == pytest.approx(1 + 2 ** -7 + 2 ** -8 - 2 ** -17, abs=1e-15)


def test_worked_example_k_scaled_is_rounded():
    # factor = gamma = bf16(2 + 2^-6) sigmoid(0) = 1 + 2^-7 on token 0, R = 2,
    # k = (1 + 2^-7, 0) and (1 + 2^-6, 0), PsiV = (1, -1):
    # k_scaled = (1 + 2^-6, 1 + 3 2^-7) after rounding, so states[1][0,0] =
    # -2^-7; unrounded it is (1 + 2^-7)(2^-7 - 2^-6) = -2^-7 - 2^-14.
    x = tiny_problem(S=2, C=1, R=2, P=1)
    x["k"][0, 0, 0, 0] = torch.tensor([1.0 + 2 ** -7, 0.0])
    x["k"][0, 0, 1, 0] = torch.tensor([1.0 + 2 ** -6, 0.0])
    x["v"][0, 0, 0, 0] = 1.0
    x["mimo_v"][0, :, 0] = torch.tensor([1.0, -1.0])
    x["dt"][0, 0] = torch.tensor([2.0 + 2 ** -6, 0.0])
    rb, re_ = both(x)
    assert rb["states"][0, 0, 1, 0, 0] == -(2 ** -7)
    assert re_["states"][0, 0, 1, 0, 0] == pytest.approx(-(2 ** -7) - 2 ** -14, abs=1e-16)


def test_worked_example_shifted_gamma_is_rounded():
    # gamma_0 = 1 + 2^-7; shifted_0 = bf16(2^-7 sigmoid(-2^-9)) where the product
    # is 2^-8 - 2^-18 (+ O(2^-40)) and rounds to 2^-8.  factor_0 =
    # bf16(1 + 2^-7 + 2^-8) is a tie -> 1 + 2^-6; without rounding shifted_0 the
    # sum sits just below the tie -> 1 + 2^-7.  k = (1, 0), PsiV = 1, so
    # states[1][0,0] = factor_0.
    x = tiny_problem(S=3, C=1, P=1)
    x["k"][0, 0, 0, 0] = torch.tensor([1.0, 0.0])
    x["v"][0, 0, 0, 0] = 1.0
    x["dt"][0, 0] = torch.tensor([2.0 + 2 ** -6, 2 ** -7, 0.0])
    x["trap"][0, 0] = torch.tensor([0.0, 2 ** -9, 0.0], dtype=torch.bfloat16)
    rb, re_ = both(x)
    assert rb["states"][0, 0, 1, 0, 0] == 1.0 + 2 ** -6
    want = (2.0 + 2 ** -6) * 0.5 + 2 ** -7 / (1.0 + math.exp(2 ** -9))
    assert re_["states"][0, 0, 1, 0, 0] == pytest.approx(want, abs=1e-15)


def test_worked_example_k_scaled_is_rounded_in_the_causal_matrix():
    # factor_0 = 1 + 2^-7; k_0 = (1 + 2^-7, 1 + 2^-6) -> k_scaled_0 =
    # (1 + 2^-6, 1 + 3 2^-7) after rounding.  q_1 = (1, -1): A[1,0] = -2^-7, but
    # -(1 + 2^-7) 2^-7 with an unrounded k_scaled.  out_1 = A[1,0] PsiV_0.
    x = tiny_problem(S=2, C=2, P=1)
    x["k"][0, 0, 0, 0] = torch.tensor([1.0 + 2 ** -7, 1.0 + 2 ** -6])
    x["q"][0, 1, 0, 0] = torch.tensor([1.0, -1.0])
    x["v"][0, 0, 0, 0] = 1.0
    x["dt"][0, 0] = torch.tensor([2.0 + 2 ** -6, 0.0])
    x["dout"][0, 1, 0, 0] = 1.0
    rb, re_ = both(x)
    assert rb["dmimo_o"][0, 0, 0, 0] == -(2 ** -7)
    assert re_["dmimo_o"][0, 0, 0, 0] == pytest.approx(-(1 + 2 ** -7) * 2 ** -7, abs=1e-16)


@pytest.mark.parametrize("side", ["q", "k"])
def test_worked_example_biased_input_is_rounded(side):
    # x = (1, 1 + 2^-7), bias = (2^-8 + 2^-10, 0): biased x_0 = bf16(1 + 2^-8 +
    # 2^-10) = 1 + 2^-7, so with the other operand (1, -1) the same-token dot
    # is exactly 0; unrounded it is -2^-8 + 2^-10.
    other = "k" if side == "q" else "q"
    x = tiny_problem()
    x[side][0, 0, 0, 0] = torch.tensor([1.0, 1.0 + 2 ** -7])
    x[side + "_bias"][0, 0] = torch.tensor([2 ** -8 + 2 ** -10, 0.0])
    x[other][0, 0, 0, 0] = torch.tensor([1.0, -1.0])
    rb, re_ = both(x)
    assert rb["qk_dot"][0, 0, 0, 0, 0] == 0.0
    assert re_["qk_dot"][0, 0, 0, 0, 0] == -(2 ** -8) + 2 ** -10


def test_worked_example_shifted_gamma_uses_bf16_dt():
    # dt_1 = 2^-7 (1 + 2^-8) is a BF16 tie and loads as 2^-7; trap_1 = -2^-8,
    # sigmoid(2^-8) = (1 + 2^-9 - O(2^-26)) / 2.  shifted_0 = bf16(2^-8 (1 + 2^-9 - ..))
    # = 2^-8 and factor_0 = bf16(1 + 2^-8) = 1; with dt_1 unrounded shifted_0
    # rounds to 2^-8 (1 + 2^-7) and factor_0 to 1 + 2^-7.  states[1] = factor_0.
    x = tiny_problem(S=3, C=1, P=1)
    x["k"][0, 0, 0, 0] = torch.tensor([1.0, 0.0])
    x["v"][0, 0, 0, 0] = 1.0
    x["dt"][0, 0] = torch.tensor([2.0, 2 ** -7 * (1 + 2 ** -8), 0.0])
    x["trap"][0, 0] = torch.tensor([0.0, -(2 ** -8), 0.0], dtype=torch.bfloat16)
    rb, re_ = both(x)
    assert rb["states"][0, 0, 1, 0, 0] == 1.0
    want = 1.0 + 2 ** -7 * (1 + 2 ** -8) / (1.0 + math.exp(-(2 ** -8)))
    assert re_["states"][0, 0, 1, 0, 0] == pytest.approx(want, abs=1e-15)


def test_worked_example_k_rotary_is_rounded():
    # Token 0: k = (1, 0) at angle 1 rad -> k_rot = (0.5390625, 0.83984375);
    # token 1: q = (1, 1) at angle 0.  A[1,0] = bf16(1.37890625) = 1.375 (tie,
    # to even); unrounded cos 1 + sin 1 -> 1.3828125.
    x = tiny_problem(S=2, C=2, P=1)
    x["k"][0, 0, 0, 0] = torch.tensor([1.0, 0.0])
    x["angles"][0, 0, 0, 0] = 1.0
    x["q"][0, 1, 0, 0] = torch.tensor([1.0, 1.0])
    x["v"][0, 0, 0, 0] = 1.0
    x["dt"][0, 0] = torch.tensor([2.0, 0.0])
    x["dout"][0, 1, 0, 0] = 1.0
    rb, re_ = both(x)
    assert rb["dmimo_o"][0, 0, 0, 0] == 1.375
    assert re_["dmimo_o"][0, 0, 0, 0] == pytest.approx(math.cos(1.0) + math.sin(1.0), abs=1e-14)


@pytest.mark.parametrize("component, dt0, want_bf16", [
    # factor 131/128: bf16(cos 1) * f = 141.23 ulps -> 141; cos 1 * f = 141.56 -> 142
    (0, 2 * 131 / 128, 141 / 256),
    # factor 137/128: bf16(sin 1) * f = 230.12 ulps -> 230; sin 1 * f = 230.56 -> 231
    (1, 2 * 137 / 128, 230 / 256),
])
def test_worked_example_k_rotary_is_rounded_before_scaling(component, dt0, want_bf16):
    # Token 0: k = (1, 0) at angle 1 rad, factor_0 = dt_0 / 2; token 1 selects one
    # k_scaled component with q_1 = e_component: out_1 = A[1,0] = k_scaled_0[comp].
    x = tiny_problem(S=2, C=2, P=1)
    x["k"][0, 0, 0, 0] = torch.tensor([1.0, 0.0])
    x["angles"][0, 0, 0, 0] = 1.0
    qv = [0.0, 0.0]
    qv[component] = 1.0
    x["q"][0, 1, 0, 0] = torch.tensor(qv)
    x["v"][0, 0, 0, 0] = 1.0
    x["dt"][0, 0] = torch.tensor([dt0, 0.0])
    x["dout"][0, 1, 0, 0] = 1.0
    rb, re_ = both(x)
    assert rb["dmimo_o"][0, 0, 0, 0] == want_bf16
    trig = math.cos(1.0) if component == 0 else math.sin(1.0)
    assert re_["dmimo_o"][0, 0, 0, 0] == pytest.approx(trig * dt0 / 2, abs=1e-14)


@pytest.mark.parametrize("reduced", [True, False])
def test_worked_example_pre_gate_product_with_out_is_rounded(reduced):
    # out = PsiV = 1 + 2^-7 (qk = 1, gamma = 1); the dout-side factor is
    # 1 + 2^-7 too, so pre = bf16((1 + 2^-7)^2) = 1 + 2^-6, not 1 + 2^-6 + 2^-14.
    # mimo_z = 0 and z = 2 make dmimo_z = pre.
    x = tiny_problem(P=1, has_z=True, reduced=reduced)
    x["q"][0, 0, 0, 0] = torch.tensor([1.0, 0.0])
    x["k"][0, 0, 0, 0] = torch.tensor([1.0, 0.0])
    x["v"][0, 0, 0] = 1.0 + 2 ** -7
    x["dt"][0, 0, 0] = 2.0
    x["dout"].fill_(1.0 + 2 ** -7)
    x["mimo_z"][0, 0, 0] = 0.0
    x["z"][0, 0, 0] = 2.0
    rb, re_ = both(x)
    assert rb["dmimo_z"][0, 0, 0, 0] == 1.0 + 2 ** -6
    assert re_["dmimo_z"][0, 0, 0, 0] == pytest.approx((1 + 2 ** -7) ** 2, abs=1e-15)


def test_worked_example_pre_gate_dout_projection_is_rounded():
    # dout * bf16(mimo_o) = (1 + 2^-7)^2 rounds to 1 + 2^-6; times out = 1.25 that
    # is 1.26953125, a tie -> 1.265625.  Without the inner rounding the product
    # sits above the tie -> 1.2734375.
    x = tiny_problem(P=1, has_z=True)
    x["q"][0, 0, 0, 0] = torch.tensor([1.0, 0.0])
    x["k"][0, 0, 0, 0] = torch.tensor([1.0, 0.0])
    x["v"][0, 0, 0] = 1.25
    x["dt"][0, 0, 0] = 2.0
    x["dout"][0, 0, 0] = 1.0 + 2 ** -7
    x["mimo_o"][0, 0, 0] = 1.0 + 2 ** -7
    x["mimo_z"][0, 0, 0] = 0.0
    x["z"][0, 0, 0] = 2.0
    rb, re_ = both(x)
    assert rb["dmimo_z"][0, 0, 0, 0] == 1.265625
    assert re_["dmimo_z"][0, 0, 0, 0] == pytest.approx((1 + 2 ** -7) ** 2 * 1.25, abs=1e-15)


# --- the layer's forward output y ---------------------------------------------
# y is pinned to the op's own gradients (themselves pinned by the token
# recurrence above): y is linear in mimo_o, and its derivative along mimo_z is
# what dmimo_z accumulates.

@pytest.mark.parametrize("has_z", [True, False])
def test_forward_y_pairs_with_dmimo_o(has_z):
    # <dout, y> = sum_t,p dout sum_r mimo_o out g = sum_r,p mimo_o dmimo_o  (exact)
    inp, _ = small_inputs(2, 37, 3, 3, 4, 8, 12, 8, 4, True, has_z, True, seed=11)
    r = oracle.bwd_fwd(*si.args_of(inp), round_bf16=False, want_y=True)
    assert r["y"].shape == tuple(inp["dout"].shape)
    lhs = float((f64(inp["dout"]) * r["y"]).sum())
    rhs = float((f64(inp["mimo_o"])[None] * r["dmimo_o"]).sum())
    assert abs(lhs - rhs) <= 1e-11 * max(abs(rhs), 1.0)


@pytest.mark.parametrize("reduced", [True, False])
def test_forward_y_gate_derivative_along_mimo_z(reduced):
    # d/ds <dout, y(mimo_z (1 + s))> at s = 0 equals sum_r,p mimo_z dmimo_z  (exact)
    inp, _ = small_inputs(1, 29, 2, 1, 3, 8, 10, 8, 4, reduced, True, False, seed=5)
    # mimo_z with 8 significant bits, so mimo_z * (1 +- 2^-12) is exact in FP32
    inp["mimo_z"] = inp["mimo_z"].to(torch.bfloat16).float()

    def f(scale):
        x = dict(inp)
        x["mimo_z"] = inp["mimo_z"] * scale
        r = oracle.bwd_fwd(*si.args_of(x), round_bf16=False, want_y=True)
        return float((f64(inp["dout"]) * r["y"]).sum()), r

    eps = 2.0 ** -12
    fp, _ = f(1.0 + eps)
    fm, _ = f(1.0 - eps)
    _, r0 = f(1.0)
    fd = (fp - fm) / (2 * eps)
    want = float((f64(inp["mimo_z"])[None] * r0["dmimo_z"]).sum())
    assert abs(fd - want) <= 1e-6 * max(abs(want), 1.0)


def test_forward_y_layout_and_bf16_rounding():
    # per-rank dout layout [B,S,R,H,P] without mimo_o; BF16 mode rounds y once
    inp, _ = small_inputs(1, 19, 2, 2, 2, 8, 6, 8, 2, False, True, True, seed=9)
    ex = oracle.bwd_fwd(*si.args_of(inp), round_bf16=True, want_y=True, want_out=True)
    y = ex["y"]
    assert y.shape == tuple(inp["dout"].shape)
    assert np.array_equal(y, oracle.bf16_nearest_array(y))
    # y[b,t,r,h,p] has out[b,h,t,r,p] as a factor: zero out -> zero y
    inp0 = dict(inp)
    inp0["mimo_v"] = torch.zeros_like(inp["mimo_v"])
    inp0["d"] = None
    y0 = oracle.bwd_fwd(*si.args_of(inp0), round_bf16=True, want_y=True)["y"]
    assert np.count_nonzero(y0) == 0
