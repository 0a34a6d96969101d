"""Both oracles against their stored summaries (tests/golden/
oracle_fixtures.json, written by tests/golden/make_oracle_fixtures.py from
the oracles alone).  A regression guard, not a pin: any change to an
oracle's arithmetic fails here until the fixtures are regenerated."""

import importlib.util
import json
import os

import numpy as np
import pytest

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _generator():
    spec = importlib.util.spec_from_file_location("make_oracle_fixtures",
                                                  os.path.join(GOLDEN, "make_oracle_fixtures.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


@pytest.fixture(scope="module")
def stored_and_now():
    with open(os.path.join(GOLDEN, "oracle_fixtures.json")) as f:
        stored = json.load(f)
    return stored, _generator().compute()


@pytest.mark.parametrize("group", ["bwd_fwd_bf16", "bwd_fwd_exact", "bwd_bwd"])
def test_oracle_outputs_match_the_stored_summaries(stored_and_now, group):
    stored, now = stored_and_now
    assert sorted(stored[group]) == sorted(now[group])
    for name, want in stored[group].items():
        got = now[group][name]
        assert got["size"] == want["size"] and got["idx"] == want["idx"], name
        scale = max(want["l2"], 1e-300)
        if group == "bwd_fwd_bf16":
            # BF16 rounding points: a libm result one ulp apart on another
            # machine can move an isolated value by one BF16 ulp (2^-8
            # relative); a changed formula moves far more
            tol, rel = 1e-4 * scale, 2.0 ** -7
        else:  # float64 throughout: agreement to rounding
            tol, rel = 1e-10 * scale, 0.0
        assert abs(got["l2"] - want["l2"]) <= tol, name
        assert abs(got["sum"] - want["sum"]) <= tol, name
        for g, w in zip(got["val"], want["val"]):
            assert abs(g - w) <= rel * abs(w) + 1e-10 * scale, (name, g, w)
