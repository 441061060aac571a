"""The oracle against its stored outputs on the tiny configuration.

The pages print no worked numeric example of this path, so the fixtures under tests/golden/ are the
oracle's own float64 outputs on the seeded tiny inputs, written by tests/golden/make_golden.py (which
calls nothing but `oracle/` and the input generators).  They guard the oracle against unintended edits of
its arithmetic; its correctness pins are the closed forms, brute force, finite differences and invariants
of test_oracle*.py.  Tolerances cover libm's last-place differences between hosts; the argmax is exact.
"""
import json
import os
import sys

import numpy as np
import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.join(HERE, "golden"))

import make_golden  # noqa: E402

RTOL, ATOL = 1e-12, 1e-15


@pytest.fixture(scope="module")
def stored_and_fresh():
    with open(os.path.join(HERE, "golden", "config1_oracle.json")) as f:
        return json.load(f), make_golden.compute()


def close(a, b):
    np.testing.assert_allclose(np.asarray(a, dtype=np.float64), np.asarray(b, dtype=np.float64), rtol=RTOL, atol=ATOL)


def test_pooled_tiny_matches_the_stored_oracle_outputs(stored_and_fresh):
    stored, fresh = stored_and_fresh
    s, f = stored["pooled"], fresh["pooled"]
    for k in ("loss", "dt", "db", "de_sum", "de_sum_sq"):
        close(s[k], f[k])
    assert s["de_rows"].keys() == f["de_rows"].keys()
    for k in s["de_rows"]:
        close(s["de_rows"][k], f["de_rows"][k])


@pytest.mark.parametrize("mode", ["sum", "mean"])
def test_maxsim_tiny_matches_the_stored_oracle_outputs(stored_and_fresh, mode):
    stored, fresh = stored_and_fresh
    s, f = stored["maxsim"][mode], fresh["maxsim"][mode]
    close(s["scores"], f["scores"])
    close(s["dq_sum_sq"], f["dq_sum_sq"])
    close(s["dd_sum_sq"], f["dd_sum_sq"])
    for key in ("dq_rows", "dd_rows"):
        assert s[key].keys() == f[key].keys()
        for k in s[key]:
            close(s[key][k], f[key][k])
    if mode == "sum":
        assert s["argmax"] == f["argmax"]


def test_stored_values_are_consistent_with_the_definitions(stored_and_fresh):
    """Relations between stored numbers that the definitions fix: mean scores are sum scores over |q|
    (every tiny query has 8 rows), and the pooled loss of 256 anchors with t = 10, b = -10 and unit rows
    lies between the all-repel and all-attract extremes of one anchor's 255 cells."""
    stored, _ = stored_and_fresh
    ssum = np.asarray(stored["maxsim"]["sum"]["scores"])
    smean = np.asarray(stored["maxsim"]["mean"]["scores"])
    np.testing.assert_allclose(smean, ssum / 8.0, rtol=1e-14, atol=0)
    loss = stored["pooled"]["loss"]
    assert 0.0 < loss < 255 * np.log1p(np.exp(20.0))
