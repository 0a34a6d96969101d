"""A second, independent pin of the second-stage oracle (oracle/bwd_bwd.py):
torch autograd of the Mamba-3 MIMO forward written token by token.

The forward here is the recurrence, not the chunked form the oracle
differentiates by hand:

    h_t   = e^{a_t} h_{t-1} + factor_t * sum_r k_rot[t,r]^T psi[t,r]
    out_t = q_rot[t] (e^{a_t} h_{t-1}) + gamma_t (qh[t] kh[t]^T) psi[t] + d psi[t]

with the rotary as a complex multiplication of the pairs (m, N/2 + m),
gamma_t = dt_t sigmoid(trap_t) and factor_t = gamma_t + dt_{t+1}
sigmoid(-trap_{t+1}).  L = sum dPhiO * out, dPhiO = dout * mimo_o (reduce-O)
or dout per rank.  Autograd of L gives the total gradient with respect to
every input; the oracle's 12 outputs must reproduce them:

* q, k, v, mimo_v, angles, d and the biases directly (DQ / DK summed over the
  tokens for the biases, DMIMO_V and DD summed over the batch);
* dt and trap through gamma and factor (DGAMMA, DFACTOR);
* the per-token log decay a through the chunk quantities built from it:
  da_cs (inclusive within the chunk), da_cs_rev (the later tokens of the
  chunk), segsum[c, i, j] = da_cs[i] - da_cs[j] and the chunk decay at the
  last valid token (DDA_CS, DDA_CS_REV, DSSDA, DDA).

Everything is float64, so the two agree to rounding (1e-9 relative).
"""

import numpy as np
import pytest
import torch

from oracle import bwd_bwd as bb


def _chunk_quantities(a, C):
    """da_cs, da_cs_rev [B,H,S] and segsum [B,H,nc,C,C] from per-token log
    decays a [B,H,S] (padded positions carry a = 0)."""
    B, H, S = a.shape
    nc = (S + C - 1) // C
    ap = np.zeros((B, H, nc * C))
    ap[:, :, :S] = a
    cs = np.cumsum(ap.reshape(B, H, nc, C), axis=-1)
    rev = cs[..., -1:] - cs
    seg = cs[..., :, None] - cs[..., None, :]
    seg = np.where(np.tril(np.ones((C, C), dtype=bool), -1), seg, -np.inf)
    return cs.reshape(B, H, -1)[:, :, :S], rev.reshape(B, H, -1)[:, :, :S], seg


def _forward_loss(t, C, div, reduced):
    """L of the token recurrence; t holds torch float64 leaves."""
    q, k, v = t["q"], t["k"], t["v"]
    B, S, R, G, N = q.shape
    H, P = v.shape[2], v.shape[3]
    w, half = N // div, N // 2

    def rotate(x, th):  # rows of x [R, N], angles th [w]
        re, im = x[:, :w], x[:, half:half + w]
        c, s = torch.cos(th)[None, :], torch.sin(th)[None, :]
        return torch.cat([re * c - im * s, x[:, w:half], re * s + im * c, x[:, half + w:]], dim=1)

    loss = torch.zeros((), dtype=torch.float64)
    for b in range(B):
        for h in range(H):
            g = h // (H // G)
            st = torch.zeros((N, P), dtype=torch.float64)
            for s in range(S):
                qh = q[b, s, :, g, :] + t["q_bias"][h]
                kh = k[b, s, :, g, :] + t["k_bias"][h]
                th = t["angles"][b, s, h]
                qr, kr = rotate(qh, th), rotate(kh, th)
                psi = v[b, s, h][None, :] * t["mimo_v"][h]
                gam = t["dt"][b, h, s] * torch.sigmoid(t["trap"][b, h, s])
                shifted = (t["dt"][b, h, s + 1] * torch.sigmoid(-t["trap"][b, h, s + 1])
                           if s + 1 < S else torch.zeros((), dtype=torch.float64))
                factor = gam + shifted
                dec = torch.exp(t["a"][b, h, s]) * st
                out = qr @ dec + gam * (qh @ kh.T) @ psi
                if t.get("d") is not None:
                    out = out + t["d"][h] * psi
                if reduced:
                    dphi = t["dout"][b, s, h][None, :] * t["mimo_o"][h]
                else:
                    dphi = t["dout"][b, s, :, h, :]
                loss = loss + (dphi * out).sum()
                st = dec + factor * (kr.T @ psi)
    return loss


def _case(B, S, H, G, R, N, P, C, div, reduced, has_d, seed):
    rng = np.random.default_rng(seed)
    x = {
        "q": rng.standard_normal((B, S, R, G, N)),
        "k": rng.standard_normal((B, S, R, G, N)),
        "v": rng.standard_normal((B, S, H, P)),
        "q_bias": 0.1 * rng.standard_normal((H, R, N)),
        "k_bias": 0.1 * rng.standard_normal((H, R, N)),
        "mimo_v": rng.standard_normal((H, R, P)) / R,
        "mimo_o": rng.standard_normal((H, R, P)) / R,
        "angles": rng.uniform(-np.pi, np.pi, (B, S, H, N // div)),
        "dt": rng.uniform(1e-3, 0.1, (B, H, S)),
        "trap": rng.uniform(0.0, 1.0, (B, H, S)),
        "a": -rng.uniform(0.01, 0.3, (B, H, S)),
        "d": rng.standard_normal((H,)) if has_d else None,
        "dout": rng.standard_normal((B, S, H, P) if reduced else (B, S, R, H, P)),
    }
    return x


def _oracle(x, C, div, reduced):
    """The oracle's 12 gradients, with its caches from the same recurrence."""
    B, S, R, G, N = x["q"].shape
    H, P = x["v"].shape[2], x["v"].shape[3]
    da_cs, da_cs_rev, seg = _chunk_quantities(x["a"], C)
    a_in = {k: x[k] for k in ("dout", "q", "k", "v", "q_bias", "k_bias", "mimo_v", "mimo_o", "d", "dt",
                              "trap", "angles")}
    a_in.update(da_cs=da_cs, da_cs_rev=da_cs_rev, segsum=seg)
    if not reduced:
        a_in["mimo_o"] = None
    nc = (S + C - 1) // C
    states = np.zeros((B, H, nc, N, P))
    qk = np.zeros((B, H, S, R, R))
    for b in range(B):
        for h in range(H):
            _, st, q_, _ = bb.forward(a_in, b, h, C, div)
            states[b, h], qk[b, h] = st, q_[:S]
    return bb.bwd_bwd(x["dout"], x["q"], x["k"], x["v"], x["q_bias"], x["k_bias"], x["mimo_v"], states, qk,
                      da_cs, da_cs_rev, x["dt"], x["trap"], seg, x["angles"],
                      mimo_o=x["mimo_o"] if reduced else None, d=x["d"], chunk_size=C, rotary_dim_divisor=div)


def _decay_gradient(g, C, S):
    """dL/da_t from the oracle's DDA_CS, DDA_CS_REV, DSSDA and DDA by the
    chain rule through the chunk quantities."""
    B, H = g["DDA_CS"].shape[:2]
    out = np.zeros((B, H, S))
    for t in range(S):
        c, tl = t // C, t % C
        lo, hi = c * C, min(c * C + C, S)
        for s in range(lo, hi):
            sl = s - lo
            if tl <= sl:  # a_t is inside da_cs[s] (and the chunk decay at s)
                out[:, :, t] += g["DDA_CS"][:, :, s] + g["DDA"][:, :, s]
            else:  # a_t is inside da_cs_rev[s]
                out[:, :, t] += g["DDA_CS_REV"][:, :, s]
        # segsum[c, i, j] = da_cs[i] - da_cs[j] contains a_t iff j < tl <= i
        dss = g["DSSDA"][:, :, c]
        out[:, :, t] += dss[:, :, tl:, :tl].sum(axis=(-2, -1))
    return out


def _close(got, want, tol=1e-9):
    scale = max(np.max(np.abs(want)), 1e-12)
    err = np.max(np.abs(got - want)) / scale
    assert err < tol, f"max |oracle - autograd| / max |autograd| = {err:.3e}"


@pytest.mark.parametrize("case", [
    dict(B=1, S=7, H=2, G=2, R=2, N=8, P=4, C=3, div=2, reduced=True, has_d=True),
    dict(B=2, S=6, H=2, G=1, R=3, N=8, P=3, C=4, div=4, reduced=False, has_d=False),
    dict(B=1, S=5, H=1, G=1, R=1, N=4, P=2, C=5, div=2, reduced=True, has_d=True),
], ids=["reduced_D_tail", "per_rank_GQA", "R1_one_chunk"])
def test_oracle_gradients_equal_autograd_of_the_token_recurrence(case):
    C, div, reduced = case["C"], case["div"], case["reduced"]
    x = _case(**case, seed=hash(tuple(case.values())) % 1000)
    g = _oracle(x, C, div, reduced)

    leaves = {k: torch.tensor(v, dtype=torch.float64, requires_grad=True) for k, v in x.items() if v is not None}
    loss = _forward_loss(leaves, C, div, reduced)
    loss.backward()
    ag = {k: v.grad.numpy() for k, v in leaves.items() if v.grad is not None}

    B, S, R, G, N = x["q"].shape
    H = x["v"].shape[2]
    hpg = H // G
    dq = g["DQ"].reshape(B, S, R, H, N)
    dk = g["DK"].reshape(B, S, R, H, N)
    # q and k: per-head gradients summed over each group's heads
    _close(np.stack([dq[:, :, :, gi * hpg:(gi + 1) * hpg].sum(axis=3) for gi in range(G)], axis=3), ag["q"])
    _close(np.stack([dk[:, :, :, gi * hpg:(gi + 1) * hpg].sum(axis=3) for gi in range(G)], axis=3), ag["k"])
    # biases: the per-head gradients summed over batch and tokens
    _close(dq.sum(axis=(0, 1)).transpose(1, 0, 2), ag["q_bias"])
    _close(dk.sum(axis=(0, 1)).transpose(1, 0, 2), ag["k_bias"])
    _close(g["DV"], ag["v"])
    _close(g["DMIMO_V"].sum(axis=0), ag["mimo_v"])
    _close(g["DANGLES"], ag["angles"])
    if case["has_d"]:
        _close(g["DD"].sum(axis=0), ag["d"])
    # dt and trap through gamma_t = dt_t s(trap_t), factor_t = gamma_t + dt_{t+1} s(-trap_{t+1})
    sg = 1.0 / (1.0 + np.exp(-x["trap"]))
    dgam, dfac = g["DGAMMA"], g["DFACTOR"]
    prev = np.concatenate([np.zeros_like(dfac[..., :1]), dfac[..., :-1]], axis=-1)  # DFACTOR_{t-1}
    _close((dgam + dfac) * sg + prev * (1.0 - sg), ag["dt"])
    _close((dgam + dfac) * x["dt"] * sg * (1.0 - sg) - prev * x["dt"] * sg * (1.0 - sg), ag["trap"])
    # the per-token log decay through da_cs, da_cs_rev, segsum and the chunk decay
    _close(_decay_gradient(g, C, S), ag["a"])
