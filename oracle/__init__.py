"""CPU oracle for ``mamba_mimo_bwd_fwd`` (Mamba-3 MIMO chunked scan, first
backward stage).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import this package.  The CUDA
library never calls it and shares no code with it.

The arithmetic lives in ``mmbf_oracle.c`` (plain C, double precision between
the BF16 rounding points of the pages' BF16 reference; see that file's header
for the passages it follows and the readings it takes).  This module only
marshals tensors into it and reassembles the per-(b,h) results into the
layouts of the op document's output table:

    dmimo_o [B,H,R,P] f64 | None     states [B,H,nchunks,N,P]
    dz      [B,S,H,P]     | None     dmimo_z [B,H,R,P]  | None
    qk_dot  [B,H,S,R,R]              out [B,H,Sp,R,P]   (optional, never an
                                                          output of the op)

and, on request, the layer's forward output y (``forward_y``), laid out like
dout: [B,S,H,P] with mimo_o, [B,S,R,H,P] without.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mmbf_oracle.c")
_LIB = os.path.join(_HERE, "libmmbf_oracle.so")
_lock = threading.Lock()
_lib = None


class _Dims(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int64) for n in (
        "B", "S", "H", "G", "R", "N", "P", "C", "div", "reduced", "has_z", "has_d", "round_bf16")]


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (OpenMP over (b,h) pairs; no FMA contraction,
    so x86 and Arm hosts give the same doubles)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".{os.getpid()}.tmp"
        subprocess.run(
            ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fopenmp",
             "-shared", "-fPIC", _SRC, "-o", tmp, "-lm"],
            check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            lib.oracle_bwd_fwd.restype = ctypes.c_int
            lib.oracle_bf16_nearest.restype = ctypes.c_double
            lib.oracle_bf16_nearest.argtypes = [ctypes.c_double]
            _lib = lib
    return _lib


def bf16_nearest(x: float) -> float:
    """The oracle's BF16 rounding of one double (nearest, ties to even)."""
    return _load().oracle_bf16_nearest(float(x))


def _bits(t: torch.Tensor | None) -> np.ndarray | None:
    """A CPU tensor as the numpy array the C oracle reads: BF16 as its raw
    16-bit patterns, FP32 as float32."""
    if t is None:
        return None
    t = t.detach().to("cpu").contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    if t.dtype == torch.float32:
        return t.numpy()
    raise TypeError(f"oracle inputs are bfloat16 or float32, got {t.dtype}")


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def bwd_fwd(dout, q, k, v, q_bias, k_bias, mimo_v, mimo_o, z, mimo_z, angles, da_cs,
            da_cs_rev, dt, trap, d, segsum, chunk_size=16, rotary_dim_divisor=4, *,
            round_bf16: bool = True, pairs=None, want_out: bool = False, want_y: bool = False) -> dict:
    """Run the oracle.  Arguments follow the pages' positional order.

    ``pairs``: None for every (b,h) pair (results in full layouts), or a list
    of (b,h) pairs (results compact, leading axis = pair index:
    states [n,nc,N,P], qk_dot [n,S,R,R], dz [n,S,P], dmimo_o/dmimo_z [n,R,P],
    out [n,Sp,R,P]).  Values are float64; with ``round_bf16`` the BF16
    outputs hold BF16 values.  ``want_y`` adds the forward output "y"
    (see forward_y; full layouts only)."""
    if want_y:
        if pairs is not None:
            raise ValueError("want_y needs the full problem (pairs=None)")
        res = bwd_fwd(dout, q, k, v, q_bias, k_bias, mimo_v, mimo_o, z, mimo_z, angles, da_cs,
                      da_cs_rev, dt, trap, d, segsum, chunk_size, rotary_dim_divisor,
                      round_bf16=round_bf16, want_out=True)
        res["y"] = forward_y(res["out"], mimo_o, z, mimo_z, q.shape[1], round_bf16=round_bf16)
        if not want_out:
            res["out"] = None
        return res
    B, S, R, G, N = q.shape
    H, P = v.shape[2], v.shape[3]
    C = int(chunk_size)
    nc = (S + C - 1) // C
    Sp = nc * C
    reduced, has_z, has_d = mimo_o is not None, z is not None, d is not None
    dims = _Dims(B, S, H, G, R, N, P, C, int(rotary_dim_divisor), int(reduced), int(has_z),
                 int(has_d), int(bool(round_bf16)))
    full = pairs is None
    if full:
        pairs = [(b, h) for b in range(B) for h in range(H)]
    pr = np.ascontiguousarray(np.array(pairs, dtype=np.int64).reshape(-1, 2))
    n = pr.shape[0]
    arrs = [_bits(x) for x in (dout, q, k, v, q_bias, k_bias, mimo_v, mimo_o, z, mimo_z, angles,
                               da_cs, da_cs_rev, dt, trap, d, segsum)]
    states = np.zeros((n, nc, N, P))
    qk = np.zeros((n, S, R, R))
    dz = np.zeros((n, S, P)) if has_z else None
    dmo = np.zeros((n, R, P)) if reduced else None
    dmz = np.zeros((n, R, P)) if has_z else None
    out = np.zeros((n, Sp, R, P)) if want_out else None
    rc = _load().oracle_bwd_fwd(
        ctypes.byref(dims), *[_ptr(a) for a in arrs], ctypes.c_int64(n), _ptr(pr), _ptr(states),
        _ptr(qk), _ptr(dz), _ptr(dmo), _ptr(dmz), _ptr(out))
    if rc != 0:
        raise MemoryError(f"oracle failed on {rc} (b,h) pairs")
    res = {"dmimo_o": dmo, "states": states, "dz": dz, "dmimo_z": dmz, "qk_dot": qk, "out": out}
    if not full:
        return res
    # Compact per-pair slots -> the op's layouts (pairs are in (b,h) order).
    res["states"] = states.reshape(B, H, nc, N, P)
    res["qk_dot"] = qk.reshape(B, H, S, R, R)
    if dz is not None:
        res["dz"] = dz.reshape(B, H, S, P).transpose(0, 2, 1, 3).copy()
    if dmo is not None:
        res["dmimo_o"] = dmo.reshape(B, H, R, P)
    if dmz is not None:
        res["dmimo_z"] = dmz.reshape(B, H, R, P)
    if out is not None:
        res["out"] = out.reshape(B, H, Sp, R, P)
    return res


OUTPUT_NAMES = ("dmimo_o", "states", "dz", "dmimo_z", "qk_dot")


def forward_y(out, mimo_o, z, mimo_z, S: int, *, round_bf16: bool = True):
    """The layer's forward output y, from the chunk output ``out`` [B,H,Sp,R,P]
    (BF16 values in BF16 mode) of a problem of length S.  It is the function
    whose gradients with respect to mimo_o, z and mimo_z the op returns (op
    document, gradient formulas of the Z / projection branch):

        gate  g[t,r,p] = silu(z[t,p] * mimo_z[r,p])   (1 without z)
        y[t,p]         = sum over r, in rank order, of mimo_o[r,p] out[t,r,p] g[t,r,p]
                                                      (with mimo_o: [B,S,H,P])
        y[t,r,p]       = out[t,r,p] g[t,r,p]          (without:     [B,S,R,H,P])

    In double; with ``round_bf16`` the result is rounded to BF16 once (the
    activations' type)."""
    B, H, Sp, R, P = out.shape
    o = out[:, :, :S]                                            # [B,H,S,R,P]
    if z is not None:
        zd = z.double().numpy()                                  # [B,S,H,P]
        mz = mimo_z.double().numpy()                             # [H,R,P]
        pz = zd.transpose(0, 2, 1, 3)[:, :, :, None, :] * mz[None, :, None, :, :]
        g = pz / (1.0 + np.exp(-pz))                             # silu, [B,H,S,R,P]
    else:
        g = np.ones_like(o)
    if mimo_o is not None:
        mo = mimo_o.double().numpy()                             # [H,R,P]
        y = np.zeros((B, H, S, P))
        for r in range(R):                                       # rank order
            y = y + mo[None, :, None, r, :] * o[:, :, :, r, :] * g[:, :, :, r, :]
        y = y.transpose(0, 2, 1, 3)                              # [B,S,H,P]
    else:
        y = (o * g).transpose(0, 2, 3, 1, 4)                     # [B,S,R,H,P]
    y = np.ascontiguousarray(y)
    return bf16_nearest_array(y) if round_bf16 else y


def bf16_nearest_array(x: np.ndarray) -> np.ndarray:
    """bf16_nearest applied to every element."""
    f = _load().oracle_bf16_nearest
    flat = np.asarray(x, dtype=np.float64).ravel()
    return np.fromiter((f(float(v)) for v in flat), dtype=np.float64, count=flat.size).reshape(np.shape(x))
