"""Seeded synthetic inputs for ``mamba_mimo_bwd_fwd``.

This module only draws random tensors with the shapes, dtypes and value
distributions of the workloads; it holds none of the op's arithmetic.  Both
the CPU oracle (``oracle/``) and the CUDA path (tests, ``bench.py``) take
their inputs from here; neither imports the other.

Two value recipes:

``"workload"`` -- the synthetic workload recipe:
    q, k, v, dout, z  ~ N(0, 1), stored as BF16
    q_bias, k_bias    ~ N(0, 0.1^2)                 FP32
    mimo_v/o/z        ~ N(0, (1/R)^2)               FP32
    angles            ~ U(-pi, pi)                  FP32
    dt                ~ U(1e-3, 0.1)                FP32
    per-token log-decay a = -dt * U(0.5, 2), zero at padded positions;
    da_cs      = inclusive cumulative sum of a within each chunk,
    da_cs_rev  = sum of a over the later tokens of the same chunk,
    segsum[c,i,j] = cs[i] - cs[j] for j <= i and -inf above the diagonal,
                    cs being the chunk cumsum over the padded chunk;
    trap ~ U(0, 1) stored as BF16;  d ~ N(0, 1).
    With this recipe the chunked scan equals the token-by-token recurrence
    with decay exp(a_t).

``"unit"`` -- the value ranges of the unit tests on the PR #125 page
    (q/k/v/dout/z randn, q_bias randn/8, k_bias randn, mimo_* randn/4,
    angles U(0,1), da_cs/da_cs_rev/segsum independent randn/8, dt
    U(0.05, 0.15), trap randn, d randn/8): decays are not consistent with
    one another, as there.

``make_inputs`` returns a dict keyed by the op's argument names in the pages'
positional order (``ARG_NAMES``) plus ``chunk_size`` and
``rotary_dim_divisor``.
"""

from __future__ import annotations

import math
from dataclasses import dataclass

import torch

ARG_NAMES = ("dout", "q", "k", "v", "q_bias", "k_bias", "mimo_v", "mimo_o", "z", "mimo_z",
             "angles", "da_cs", "da_cs_rev", "dt", "trap", "d", "segsum")


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    S: int
    H: int
    G: int
    R: int
    N: int
    P: int
    C: int
    div: int = 4
    reduced: bool = True
    has_z: bool = True
    has_d: bool = True

    @property
    def nchunks(self) -> int:
        return (self.S + self.C - 1) // self.C

    def shape_kwargs(self) -> dict:
        return dict(B=self.B, S=self.S, H=self.H, G=self.G, R=self.R, N=self.N, P=self.P,
                    C=self.C, div=self.div, reduced=self.reduced, has_z=self.has_z,
                    has_d=self.has_d)


# The five synthetic workloads: tiny, tail + GQA, the pages' timed shape,
# wide state, throughput.
WORKLOADS = (
    Workload("tiny_b1_s64_h2_r2_n16", 1, 64, 2, 1, 2, 16, 16, 16, 4, True, True, True),
    Workload("tail_gqa_b2_s1000_h8_g2_r4_n32", 2, 1000, 8, 2, 4, 32, 32, 16, 4, False, False, False),
    Workload("mimo_b1_s8192_h16_r4_n64_p64_c16", 1, 8192, 16, 1, 4, 64, 64, 16, 4, True, True, True),
    Workload("wide_b2_s16384_h32_g4_r4_n128_p64_c32", 2, 16384, 32, 4, 4, 128, 64, 32, 2, True, True, True),
    Workload("throughput_b8_s32768_h32_g8_r8_n64_p64_c16", 8, 32768, 32, 8, 8, 64, 64, 16, 4, True, True, True),
)
WORKLOAD_SEED_BASE = 0x4D4D4246


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def make_inputs(*, B, S, H, G, R, N, P, C, div=4, reduced=True, has_z=True, has_d=True,
                seed=0, recipe="workload", device="cpu") -> dict:
    """Draw one seeded input set (see the module docstring for the recipes)."""
    dev = torch.device(device)
    g = _gen(seed, dev)
    bf16, f32 = torch.bfloat16, torch.float32
    nc = (S + C - 1) // C
    Sp = nc * C

    def randn(shape, scale=1.0, dtype=f32):
        x = torch.randn(shape, generator=g, device=dev, dtype=f32)
        if scale != 1.0:
            x = x * scale
        return x.to(dtype)

    def uniform(shape, lo, hi, dtype=f32):
        x = torch.rand(shape, generator=g, device=dev, dtype=f32) * (hi - lo) + lo
        return x.to(dtype)

    w = N // div
    out = {}
    q = randn((B, S, R, G, N), dtype=bf16)
    k = randn((B, S, R, G, N), dtype=bf16)
    v = randn((B, S, H, P), dtype=bf16)
    dout = randn((B, S, H, P) if reduced else (B, S, R, H, P), dtype=bf16)
    z = randn((B, S, H, P), dtype=bf16) if has_z else None
    if recipe == "workload":
        q_bias = randn((H, R, N), 0.1)
        k_bias = randn((H, R, N), 0.1)
        mimo_v = randn((H, R, P), 1.0 / R)
        mimo_o = randn((H, R, P), 1.0 / R) if reduced else None
        mimo_z = randn((H, R, P), 1.0 / R) if has_z else None
        angles = uniform((B, S, H, w), -math.pi, math.pi)
        dt = uniform((B, H, S), 1e-3, 0.1)
        a = -dt * uniform((B, H, S), 0.5, 2.0)
        a_pad = torch.zeros((B, H, Sp), device=dev, dtype=f32)
        a_pad[:, :, :S] = a
        cs = torch.cumsum(a_pad.view(B, H, nc, C), dim=-1)          # inclusive, per chunk
        rev = cs[..., C - 1:C] - cs                                   # later tokens of the chunk
        da_cs = cs.reshape(B, H, Sp)[:, :, :S].contiguous()
        da_cs_rev = rev.reshape(B, H, Sp)[:, :, :S].contiguous()
        seg = cs[..., :, None] - cs[..., None, :]
        upper = torch.triu(torch.ones((C, C), dtype=torch.bool, device=dev), diagonal=1)
        segsum = seg.masked_fill(upper, float("-inf")).contiguous()
        trap = uniform((B, H, S), 0.0, 1.0, dtype=bf16)
        d = randn((H,)) if has_d else None
    elif recipe == "unit":
        q_bias = randn((H, R, N), 1.0 / 8)
        k_bias = randn((H, R, N))
        mimo_v = randn((H, R, P), 0.25)
        mimo_o = randn((H, R, P), 0.25) if reduced else None
        mimo_z = randn((H, R, P), 0.25) if has_z else None
        angles = uniform((B, S, H, w), 0.0, 1.0)
        da_cs = randn((B, H, S), 1.0 / 8)
        da_cs_rev = randn((B, H, S), 1.0 / 8)
        dt = uniform((B, H, S), 0.05, 0.15)
        trap = randn((B, H, S), dtype=bf16)
        d = randn((H,), 1.0 / 8) if has_d else None
        segsum = randn((B, H, nc, C, C), 1.0 / 8)
    else:
        raise ValueError(f"unknown recipe {recipe!r}")
    vals = dict(dout=dout, q=q, k=k, v=v, q_bias=q_bias, k_bias=k_bias, mimo_v=mimo_v,
                mimo_o=mimo_o, z=z, mimo_z=mimo_z, angles=angles, da_cs=da_cs,
                da_cs_rev=da_cs_rev, dt=dt, trap=trap, d=d, segsum=segsum)
    out.update({n: vals[n] for n in ARG_NAMES})
    out["chunk_size"] = C
    out["rotary_dim_divisor"] = div
    return out


def workload_inputs(index: int, device="cpu") -> dict:
    wl = WORKLOADS[index]
    return make_inputs(**wl.shape_kwargs(), seed=WORKLOAD_SEED_BASE + index, device=device)


def args_of(inputs: dict) -> tuple:
    """Positional argument tuple in the pages' order (17 tensors, chunk_size,
    rotary_dim_divisor)."""
    return tuple(inputs[n] for n in ARG_NAMES) + (inputs["chunk_size"], inputs["rotary_dim_divisor"])


def head_slice(inputs: dict, b: int, h: int) -> dict:
    """The inputs one (b,h) pair reads, as a B=1, H=1, G=1 problem (tensor
    slicing only): q/k of the head's group, the head's v/dout/z/angles,
    decays, segsum and parameters."""
    q = inputs["q"]
    H = inputs["v"].shape[2]
    G = q.shape[3]
    g = h // (H // G)
    out = dict(inputs)
    out["q"] = q[b:b + 1, :, :, g:g + 1].contiguous()
    out["k"] = inputs["k"][b:b + 1, :, :, g:g + 1].contiguous()
    out["v"] = inputs["v"][b:b + 1, :, h:h + 1].contiguous()
    dout = inputs["dout"]
    out["dout"] = (dout[b:b + 1, :, h:h + 1] if dout.dim() == 4 else dout[b:b + 1, :, :, h:h + 1]).contiguous()
    if inputs["z"] is not None:
        out["z"] = inputs["z"][b:b + 1, :, h:h + 1].contiguous()
    out["angles"] = inputs["angles"][b:b + 1, :, h:h + 1].contiguous()
    for n in ("da_cs", "da_cs_rev", "dt", "trap", "segsum"):
        out[n] = inputs[n][b:b + 1, h:h + 1].contiguous()
    for n in ("q_bias", "k_bias", "mimo_v", "mimo_o", "mimo_z", "d"):
        if inputs[n] is not None:
            out[n] = inputs[n][h:h + 1].contiguous()
    return out


def make_stage1_caches(*, B, S, H, R, N, P, C, seed, device="cpu") -> tuple:
    """Seeded stand-ins for the first stage's caches that the second stage
    reads as given inputs: states [B,H,nchunks,N,P] ~ N(0, 1) and qk_dot
    [B,H,S,R,R] ~ N(0, N), both stored as BF16 (the first stage's output
    dtype).  For tests and benchmarks at sizes where the caches are not
    derived from a forward pass."""
    dev = torch.device(device)
    g = _gen(seed, dev)
    nc = (S + C - 1) // C
    states = torch.randn((B, H, nc, N, P), generator=g, device=dev).to(torch.bfloat16)
    qk = (torch.randn((B, H, S, R, R), generator=g, device=dev) * math.sqrt(N)).to(torch.bfloat16)
    return states, qk
