"""The benchmark's FLOP accounting (the roofline numerators) against a
brute-force count of the multiply-adds each stage's dense products perform,
token pair by token pair, with the masked upper triangle not counted."""

import os
import sys
from types import SimpleNamespace

import pytest

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402


def _pairs(C):
    """Strictly causal token pairs (t_i > t_j) of one chunk."""
    return sum(1 for ti in range(C) for tj in range(C) if ti > tj)


def _first_stage_macs(wl):
    per_chunk = 0
    CR = wl.C * wl.R
    per_chunk += CR * wl.N * wl.P                      # state update k_state^T PsiV
    per_chunk += CR * wl.N * wl.P                      # inter: q_rot . state
    rank_pairs = _pairs(wl.C) * wl.R * wl.R
    per_chunk += rank_pairs * wl.N                     # strictly causal Q K^T
    per_chunk += rank_pairs * wl.P                     # A PsiV
    per_chunk += wl.C * wl.R * wl.R * wl.N             # same-token qk_dot
    per_chunk += wl.C * wl.R * wl.R * wl.P             # diagonal qk_dot PsiV
    return per_chunk * (wl.S // wl.C) * wl.B * wl.H


def _second_stage_macs(wl):
    CR = wl.C * wl.R
    rank_pairs = _pairs(wl.C) * wl.R * wl.R
    causal = rank_pairs * (wl.N + wl.P + wl.P + wl.N + wl.N)  # Q Ks^T, A^T dPhiO, dPhiO PsiV^T, dS Ks, dS^T Q
    state = 4 * CR * wl.N * wl.P                              # dPhiO Hc^T, k_state D, PsiV D^T, Q Hc
    return (causal + state) * (wl.S // wl.C) * wl.B * wl.H


SHAPES = [dict(B=1, S=64, H=2, R=2, N=16, P=16, C=16), dict(B=2, S=96, H=3, R=4, N=32, P=8, C=8),
          dict(B=1, S=8192, H=16, R=4, N=64, P=64, C=16)]


@pytest.mark.parametrize("shape", SHAPES)
def test_flop_accounting_equals_two_flop_per_counted_multiply_add(shape):
    wl = SimpleNamespace(**shape)
    assert bench.algorithmic_flop(wl) == 2 * _first_stage_macs(wl)
    assert bench.bb_grad_flop(wl) == 2 * _second_stage_macs(wl)


def test_timed_shape_figures():
    wl = SimpleNamespace(**SHAPES[-1])
    assert bench.algorithmic_flop(wl) == 13_153_337_344
    assert bench.bb_grad_flop(wl) == 27_246_198_784
