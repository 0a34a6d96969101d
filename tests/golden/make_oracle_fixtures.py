"""Writes oracle_fixtures.json: a small text summary of both oracles' outputs
on seeded synthetic inputs, so that a later change to an oracle's arithmetic
shows up as a failing test (tests/test_oracle_fixtures.py) and has to be
justified.  Calls only oracle/ (and the seeded input generators).

    python tests/golden/make_oracle_fixtures.py
"""

import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import oracle  # noqa: E402
import synthetic_inputs as si  # noqa: E402
from oracle import bwd_bwd as bb  # noqa: E402

OUT = os.path.join(os.path.dirname(os.path.abspath(__file__)), "oracle_fixtures.json")
SAMPLES = 8


def summary(x):
    """Sum, L2 norm and SAMPLES entries at fixed, spread flat indices."""
    x = np.asarray(x, dtype=np.float64).ravel()
    idx = np.linspace(0, x.size - 1, SAMPLES).round().astype(int)
    return {"size": int(x.size), "sum": float(x.sum()), "l2": float(np.sqrt((x * x).sum())),
            "idx": idx.tolist(), "val": [float(v) for v in x[idx]]}


def first_stage_case():
    """The tiny workload, B1 S64 H2 R2 N=P=16 C16, every branch on."""
    return si.workload_inputs(0)


def second_stage_case():
    """B1 S20 H2 G1 R2 N=8 P=4 C8 (tail of 4), reduce-O and D, caches from
    the oracle's own forward."""
    inp = si.make_inputs(B=1, S=20, H=2, G=1, R=2, N=8, P=4, C=8, div=4, reduced=True, has_z=False,
                         has_d=True, seed=77, recipe="workload")
    keys = ("dout", "q", "k", "v", "q_bias", "k_bias", "mimo_v", "mimo_o", "d", "da_cs", "da_cs_rev", "dt",
            "trap", "segsum", "angles")
    a = {k: bb._f64(inp[k]) for k in keys}
    nc = (20 + 8 - 1) // 8
    states, qk = np.zeros((1, 2, nc, 8, 4)), np.zeros((1, 2, 20, 2, 2))
    for h in range(2):
        _, st, q_, _ = bb.forward(a, 0, h, 8, 4)
        states[0, h], qk[0, h] = st, q_[:20]
    return a, states, qk


def compute():
    res = {}
    inp = first_stage_case()
    for mode, kw in (("bf16", {}), ("exact", {"round_bf16": False})):
        out = oracle.bwd_fwd(*si.args_of(inp), **kw)
        res[f"bwd_fwd_{mode}"] = {n: summary(out[n]) for n in oracle.OUTPUT_NAMES if out[n] is not None}
    a, states, qk = second_stage_case()
    g = bb.bwd_bwd(a["dout"], a["q"], a["k"], a["v"], a["q_bias"], a["k_bias"], a["mimo_v"], states, qk,
                   a["da_cs"], a["da_cs_rev"], a["dt"], a["trap"], a["segsum"], a["angles"], mimo_o=a["mimo_o"],
                   d=a["d"], chunk_size=8, rotary_dim_divisor=4)
    res["bwd_bwd"] = {n: summary(g[n]) for n in bb.OUTPUT_NAMES if g[n] is not None}
    return res


if __name__ == "__main__":
    with open(OUT, "w") as f:
        json.dump(compute(), f, indent=1, sort_keys=True)
        f.write("\n")
    print("wrote", OUT)
