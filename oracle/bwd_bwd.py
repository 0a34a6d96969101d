"""CPU oracle for ``mamba_mimo_bwd_bwd``: the second backward stage of the
Mamba-3 MIMO chunked scan (the reverse scan over chunks and its 12 gradients).

TEST INFRASTRUCTURE ONLY.  Only ``tests/`` and ``bench.py``'s CPU legs may
import this module.  The CUDA library never calls it and shares no code with
it.

Source of the definition (page "MindSpeed-Ops PR #100", second stage):
  [api]    the op document "mamba3_mimo_bwd_bwd 算子迁移说明": signature,
           the input and output tables (shapes, dtypes; DQ/DK laid out as
           [B, S*R, H, N]), and its reverse-scan paragraph (dPhiO and PsiV).
  [cache]  the practice document "mamba3_mimo_bwd_bwd Triton-Ascend 实践",
           section "输入缓存的语义": states[c] is the state entering chunk
           c, with state_out = state_in * exp(da_cs_sum) + K_state^T PsiV and
           dstates_in = dstates_out * exp(da_cs_sum) + Q^T (dPhiO exp(da_cs));
           qk_dot is the same-token R x R q.k block used by the diagonal term
           gamma * qk_dot * PsiV.
  [groups] the same document, "梯度分组": which gradients are chunk-local,
           which follow the state chain, which are the rotary post-pass.
  [tail]   the same document, "非整 chunk": inputs zero-padded to whole
           chunks, sequence outputs cropped, DSSDA's invalid rows and columns
           in the last chunk zeroed.
  The forward these gradients differentiate is the first stage's chunked
  computation (page "feat: add Triton-Ascend implementation of Mamba-3
  mamba_mimo_bwd_fwd #125", the FP32 reference) without rounding points.

Readings (the pages name the outputs but print no formula for them):
  - Every output is the exact derivative, in float64, of
        L = sum_{t < S, r, p} dPhiO[t, r, p] * out[t, r, p]
    where out is the chunk output of the first stage, with dPhiO =
    dout[t,p] * mimo_o[r,p] (reduce-O) or dout[t,r,p] [api], and the states
    carried by the forward recurrence (the given ``states`` are those values
    and stand in for them [cache]).  No Z gating: the first stage has folded
    it into dout [api, "支持范围"].
  - gamma = dt * sigmoid(trap); factor = gamma + dt[t+1] * sigmoid(-trap[t+1])
    (0 at the last padded position), dt unrounded (the FP32 reference).
    DGAMMA and DFACTOR are the gradients with respect to these two.
  - da_cs enters twice: exp(da_cs[t]) on the inter term of token t, and
    exp(da_cs[last valid token of the chunk]) as the chunk's state decay
    (da_cs_sum).  DDA_CS is the gradient through the first use; DDA the
    gradient through the second, reported at each chunk's last valid token
    (zero at every other token).  DDA + DDA_CS is the whole gradient with
    respect to da_cs.
  - DQ and DK are per head (not summed over the heads of a GQA group), with
    row t*R + r; DMIMO_V and DD are per batch (not summed over B).
  - DSSDA[b,h,c,i,j] sums the gradient of the masked segsum entry (t_i > t_j)
    over the R x R rank pairs of the two tokens; it is 0 on and above the
    diagonal and in the last chunk's rows and columns past S.

Parity pins of this module live in tests/test_oracle_bwd_bwd.py.
"""

from __future__ import annotations

import numpy as np
import torch

OUTPUT_NAMES = ("DQ", "DK", "DV", "DMIMO_V", "DANGLES", "DFACTOR", "DGAMMA", "DDA", "DSSDA",
                "DDA_CS_REV", "DDA_CS", "DD")


def _f64(t):
    if t is None:
        return None
    if isinstance(t, torch.Tensor):
        return t.detach().to("cpu", torch.float64).numpy()
    return np.asarray(t, dtype=np.float64)


def _sigmoid(x):
    return 1.0 / (1.0 + np.exp(-x))


def _rotate(x, th, w):
    """Rotary on the pairs (i, N/2 + i), i < w, with angles th[..., i]
    (page #125, the rotary helper of the FP32 reference); other columns pass."""
    half = x.shape[-1] // 2
    y = x.copy()
    c, s = np.cos(th), np.sin(th)
    a, b = x[..., :w], x[..., half:half + w]
    y[..., :w] = c * a - s * b
    y[..., half:half + w] = s * a + c * b
    return y


def _rotate_back(dy, y, th, w):
    """Gradient of _rotate: the input gradient (transposed rotation) and the
    angle gradient d/dth = dy_lo * (-y_hi) + dy_hi * y_lo, per pair."""
    half = dy.shape[-1] // 2
    dx = dy.copy()
    c, s = np.cos(th), np.sin(th)
    dlo, dhi = dy[..., :w], dy[..., half:half + w]
    dx[..., :w] = c * dlo + s * dhi
    dx[..., half:half + w] = -s * dlo + c * dhi
    dth = dlo * (-y[..., half:half + w]) + dhi * y[..., :w]
    return dx, dth


def token_scalars(dt, trap, S, Sp):
    """gamma and factor over the padded sequence of one (b,h) (reading above)."""
    dtp = np.zeros(Sp)
    trp = np.zeros(Sp)
    dtp[:S], trp[:S] = dt, trap
    gamma = dtp * _sigmoid(trp)
    shifted = np.zeros(Sp)
    shifted[:-1] = dtp[1:] * _sigmoid(-trp[1:])
    return gamma, gamma + shifted


class _Pair:
    """Inputs of one (b,h) over the padded sequence (zero past S)."""

    def __init__(self, a, b, h, C, div, gamma=None, factor=None, da_cs_dec=None):
        B, S, R, G, N = a["q"].shape
        H, P = a["v"].shape[2], a["v"].shape[3]
        nc = (S + C - 1) // C
        Sp = nc * C
        g = h // (H // G)
        w = N // div
        self.S, self.Sp, self.nc, self.C, self.R, self.N, self.P, self.w = S, Sp, nc, C, R, N, P, w

        def pad(x, shape):
            y = np.zeros((Sp,) + shape)
            y[:S] = x
            return y

        self.q = pad(a["q"][b, :, :, g, :], (R, N))
        self.k = pad(a["k"][b, :, :, g, :], (R, N))
        self.qh = self.q + a["q_bias"][h][None]            # biased q [page #125]
        self.kh = self.k + a["k_bias"][h][None]
        self.th = pad(a["angles"][b, :, h, :], (w,))[:, None, :]
        self.qr = _rotate(self.qh, self.th, w)
        self.kr = _rotate(self.kh, self.th, w)
        self.v = pad(a["v"][b, :, h, :], (P,))
        self.mv = a["mimo_v"][h]
        self.psi = self.v[:, None, :] * self.mv[None]      # PsiV [t, r, p]   [api]
        if a["mimo_o"] is not None:                        # dPhiO            [api]
            self.gphi = pad(a["dout"][b, :, h, :], (P,))[:, None, :] * a["mimo_o"][h][None]
        else:
            self.gphi = pad(a["dout"][b, :, :, h, :], (R, P))
        gam, fac = token_scalars(a["dt"][b, h], a["trap"][b, h], S, Sp)
        self.gamma = gam if gamma is None else gamma
        self.factor = fac if factor is None else factor
        self.da_cs = pad(a["da_cs"][b, h], ())
        self.da_cs_dec = self.da_cs if da_cs_dec is None else da_cs_dec
        self.da_cs_rev = pad(a["da_cs_rev"][b, h], ())
        self.ks = self.kr * self.factor[:, None, None]                        # k_scaled
        self.kst = self.ks * np.exp(self.da_cs_rev)[:, None, None]            # k_state
        self.seg = a["segsum"][b, h]
        self.d = 0.0 if a["d"] is None else float(a["d"][h])

    def chunk(self, x, c):
        """Rows j = t*R + r of chunk c."""
        C = self.C
        return x[c * C:(c + 1) * C].reshape(C * self.R, *x.shape[2:])

    def alpha(self, c):
        last = min((c + 1) * self.C, self.S) - 1
        return np.exp(self.da_cs_dec[last])

    def masks(self, c):
        """Strict causal mask on token index and exp(segsum) on rows x cols."""
        C, R = self.C, self.R
        tok = np.arange(C * R) // R
        mask = tok[:, None] > tok[None, :]
        ex = np.where(mask, np.exp(np.where(mask, self.seg[c][tok[:, None], tok[None, :]], 0.0)), 0.0)
        return mask, ex


def forward(a, b, h, C, div, *, gamma=None, factor=None, da_cs_dec=None):
    """The first stage's forward for one (b,h) in float64 with no rounding
    points: returns (L, states [nc,N,P], qk [Sp,R,R], out [Sp,R,P]).  gamma,
    factor and the da_cs of the chunk decay may be given separately (the pins
    differentiate through each)."""
    pr = _Pair(a, b, h, C, div, gamma, factor, da_cs_dec)
    R, N, P, nc = pr.R, pr.N, pr.P, pr.nc
    qk = np.einsum("trn,tsn->trs", pr.qh, pr.kh)           # same-token, un-rotated
    states = np.zeros((nc, N, P))
    out = np.zeros((pr.Sp, R, P))
    hst = np.zeros((N, P))
    for c in range(nc):
        states[c] = hst
        qc, ksc, kstc, psic = pr.chunk(pr.qr, c), pr.chunk(pr.ks, c), pr.chunk(pr.kst, c), pr.chunk(pr.psi, c)
        ea = np.repeat(np.exp(pr.da_cs[c * C:(c + 1) * C]), R)
        mask, ex = pr.masks(c)
        amat = (qc @ ksc.T) * ex
        inter = ea[:, None] * (qc @ hst)
        intra = amat @ psic
        gam = pr.gamma[c * C:(c + 1) * C]
        diag = gam[:, None, None] * np.einsum("tor,trp->top", qk[c * C:(c + 1) * C],
                                              pr.psi[c * C:(c + 1) * C])
        out[c * C:(c + 1) * C] = (inter + intra + pr.d * psic).reshape(C, R, P) + diag
        hst = pr.alpha(c) * hst + kstc.T @ psic
    L = float(np.sum(pr.gphi[:pr.S] * out[:pr.S]))
    return L, states, qk, out


def bwd_bwd(dout, q, k, v, q_bias, k_bias, mimo_v, states, qk_dot, da_cs, da_cs_rev, dt, trap,
            segsum, angles, mimo_o=None, d=None, chunk_size=16, rotary_dim_divisor=4) -> dict:
    """The 12 gradients in float64.  Arguments follow the pages' order [api];
    ``states`` and ``qk_dot`` are the first stage's caches."""
    a = {k_: _f64(v_) for k_, v_ in dict(dout=dout, q=q, k=k, v=v, q_bias=q_bias, k_bias=k_bias,
                                            mimo_v=mimo_v, mimo_o=mimo_o, d=d, da_cs=da_cs,
                                            da_cs_rev=da_cs_rev, dt=dt, trap=trap, segsum=segsum,
                                            angles=angles).items()}
    st = _f64(states)
    qkd = _f64(qk_dot)
    B, S, R, G, N = a["q"].shape
    H, P = a["v"].shape[2], a["v"].shape[3]
    C = int(chunk_size)
    div = int(rotary_dim_divisor)
    nc = (S + C - 1) // C
    w = N // div
    out = {
        "DQ": np.zeros((B, S * R, H, N)), "DK": np.zeros((B, S * R, H, N)), "DV": np.zeros((B, S, H, P)),
        "DMIMO_V": np.zeros((B, H, R, P)), "DANGLES": np.zeros((B, S, H, w)),
        "DFACTOR": np.zeros((B, H, S)), "DGAMMA": np.zeros((B, H, S)), "DDA": np.zeros((B, H, S)),
        "DSSDA": np.zeros((B, H, nc, C, C)), "DDA_CS_REV": np.zeros((B, H, S)),
        "DDA_CS": np.zeros((B, H, S)), "DD": None if d is None else np.zeros((B, H)),
    }
    for b in range(B):
        for h in range(H):
            g = _pair_grads(a, st[b, h], qkd[b, h], b, h, C, div)
            Sx = S
            out["DQ"][b, :, h] = g["dqh"][:Sx].reshape(Sx * R, N)
            out["DK"][b, :, h] = g["dkh"][:Sx].reshape(Sx * R, N)
            out["DV"][b, :, h] = g["dv"][:Sx]
            out["DMIMO_V"][b, h] = g["dmv"]
            out["DANGLES"][b, :, h] = g["dth"][:Sx]
            for name, key in (("DFACTOR", "dfac"), ("DGAMMA", "dgam"), ("DDA", "dda"),
                              ("DDA_CS_REV", "ddar"), ("DDA_CS", "ddac")):
                out[name][b, h] = g[key][:Sx]
            out["DSSDA"][b, h] = g["dseg"]
            if d is not None:
                out["DD"][b, h] = g["dd"]
    return out


def _pair_grads(a, states, qk_dot, b, h, C, div) -> dict:
    """All gradients of one (b,h): a reverse scan for dstates, then each
    chunk's gradients given the state entering it and the dstates leaving it."""
    pr = _Pair(a, b, h, C, div)
    R, N, P, nc, S, Sp, w = pr.R, pr.N, pr.P, pr.nc, pr.S, pr.Sp, pr.w
    qk = np.zeros((Sp, R, R))
    qk[:S] = qk_dot
    # reverse scan [cache]: D_c = alpha_c D_{c+1} + (Q exp(da_cs))^T dPhiO;
    # dn[c] is the gradient with respect to the state leaving chunk c.
    dn = np.zeros((nc, N, P))
    dcur = np.zeros((N, P))
    for c in range(nc - 1, -1, -1):
        dn[c] = dcur
        ea = np.repeat(np.exp(pr.da_cs[c * C:(c + 1) * C]), R)
        dcur = pr.alpha(c) * dcur + (pr.chunk(pr.qr, c) * ea[:, None]).T @ pr.chunk(pr.gphi, c)
    dqr = np.zeros((Sp, R, N))
    dks = np.zeros((Sp, R, N))
    dpsi = np.zeros((Sp, R, P))
    dqh_diag = np.zeros((Sp, R, N))
    dkh_diag = np.zeros((Sp, R, N))
    res = {k_: np.zeros(Sp) for k_ in ("dfac", "dgam", "dda", "ddar", "ddac")}
    dseg = np.zeros((nc, C, C))
    dd = 0.0
    for c in range(nc):
        sl = slice(c * C, (c + 1) * C)
        hc = states[c]
        qc, ksc, kstc, psic, gc = (pr.chunk(x, c) for x in (pr.qr, pr.ks, pr.kst, pr.psi, pr.gphi))
        ea = np.repeat(np.exp(pr.da_cs[sl]), R)
        mask, ex = pr.masks(c)
        smat = qc @ ksc.T
        amat = smat * ex
        # inter: out += exp(da_cs) Q h_c
        inter = ea[:, None] * (qc @ hc)
        dq = ea[:, None] * (gc @ hc.T)
        res["ddac"][sl] = np.sum((inter * gc).reshape(C, R, P), axis=(1, 2))
        # intra: out += A PsiV, A = mask * (Q Ks^T) * exp(segsum)
        dA = gc @ psic.T
        dS = dA * ex
        dq += dS @ ksc
        dk = dS.T @ qc
        dp = amat.T @ gc
        dseg[c] = np.add.reduceat(np.add.reduceat(dA * amat, np.arange(0, C * R, R), axis=0),
                                  np.arange(0, C * R, R), axis=1)
        # state update: h_{c+1} = alpha_c h_c + Kst^T PsiV
        dkst = psic @ dn[c].T
        dp += kstc @ dn[c]
        last = min((c + 1) * C, S) - 1
        res["dda"][last] += pr.alpha(c) * np.sum(hc * dn[c])
        res["ddar"][sl] = np.sum((dkst * kstc).reshape(C, R, N), axis=(1, 2))
        dk += dkst * np.repeat(np.exp(pr.da_cs_rev[sl]), R)[:, None]
        # D skip
        dd += float(np.sum(gc * psic))
        dp += pr.d * gc
        # diagonal: out[t,o,p] += gamma_t sum_r qk[t,o,r] PsiV[t,r,p]
        g3 = gc.reshape(C, R, P)
        p3 = psic.reshape(C, R, P)
        res["dgam"][sl] = np.einsum("top,tor,trp->t", g3, qk[sl], p3)
        gam = pr.gamma[sl]
        dp3 = gam[:, None, None] * np.einsum("tor,top->trp", qk[sl], g3)
        dqk = gam[:, None, None] * np.einsum("top,trp->tor", g3, p3)
        dqh_diag[sl] = np.einsum("tor,trn->ton", dqk, pr.kh[sl])
        dkh_diag[sl] = np.einsum("tor,ton->trn", dqk, pr.qh[sl])
        dqr[sl] = dq.reshape(C, R, N)
        dks[sl] = dk.reshape(C, R, N)
        dpsi[sl] = dp.reshape(C, R, P) + dp3
    # k_scaled = k_rot * factor
    res["dfac"] = np.sum(dks * pr.kr, axis=(1, 2))
    dkr = dks * pr.factor[:, None, None]
    # rotary post-pass [groups]
    dqh, dthq = _rotate_back(dqr, pr.qr, pr.th, w)
    dkh, dthk = _rotate_back(dkr, pr.kr, pr.th, w)
    dqh += dqh_diag
    dkh += dkh_diag
    dth = np.sum(dthq + dthk, axis=1)
    dv = np.einsum("trp,rp->tp", dpsi, pr.mv)
    dmv = np.einsum("trp,tp->rp", dpsi[:S], pr.v[:S])
    # DSSDA: zero on/above the diagonal (masked) and past S in the last chunk [tail]
    valid = np.arange(nc * C).reshape(nc, C) < S
    dseg *= valid[:, :, None] & valid[:, None, :]
    return dict(dqh=dqh, dkh=dkh, dv=dv, dmv=dmv, dth=dth, dseg=dseg, dd=dd, **res)
