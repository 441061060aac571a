"""Pins of the oracle's `balanced` and `ranked` pair-loss forms over a score matrix (no GPU).

The pages define both forms in words only ("Training", `uform_pair_loss_form_t`): balanced normalises a
row's attract and repel halves apart; ranked scores every positive over every negative and the bias
cancels.  The pins below check the properties those words fix (bias cancellation, shift invariance,
normalisation apart, reduction to the sigmoid form) plus closed forms and finite differences.
"""

import math

import numpy as np
import pytest

import oracle
from contrastive_late_interaction_gb300 import synth
from tests.test_oracle import to_csr


def _rel(rng, n, p_att=0.2, p_rep=0.3, p_ign=0.1):
    att, rep, ign = {}, {}, set()
    for i in range(n):
        for j in range(n):
            u = rng.random()
            if u < p_att:
                att[(i, j)] = float(rng.uniform(0.3, 2.0))
            elif u < p_att + p_rep:
                rep[(i, j)] = float(rng.uniform(0.3, 2.0))
            elif u < p_att + p_rep + p_ign:
                ign.add((i, j))
    return to_csr(n, att.keys(), att), to_csr(n, rep.keys(), rep), to_csr(n, ign)


def test_ranked_bias_cancels_and_row_shifts_do_not_matter():
    rng = np.random.default_rng(1)
    n = 7
    s = rng.normal(size=(n, n))
    A, R, I = _rel(rng, n)
    a = oracle.pair_loss_scores_form("ranked", s, 3.0, 0.0, A, R, I, ambient_weight=0.5)
    c = oracle.pair_loss_scores_form("ranked", s, 3.0, -7.5, A, R, I, ambient_weight=0.5)
    shift = rng.normal(size=(n, 1))
    e = oracle.pair_loss_scores_form("ranked", s + shift, 3.0, 2.0, A, R, I, ambient_weight=0.5)
    for x in (c, e):
        assert x["loss"] == pytest.approx(a["loss"], rel=1e-12)
        assert x["dt"] == pytest.approx(a["dt"], rel=1e-10, abs=1e-14)
        np.testing.assert_allclose(x["dscores"], a["dscores"], rtol=1e-10, atol=1e-14)
    assert a["db"] == 0.0
    # every row's gradient sums to zero (a shift of the row changes nothing)
    np.testing.assert_allclose(a["dscores"].sum(axis=1), 0.0, atol=1e-14)


def test_ranked_one_positive_one_negative_closed_form():
    s = np.array([[0.7, -0.2], [0.1, 0.4]])
    att = to_csr(2, [(0, 0), (1, 1)])
    rep = to_csr(2, [(0, 1), (1, 0)])
    t = 2.5
    r = oracle.pair_loss_scores_form("ranked", s, t, 0.0, att, rep, negatives_named=True)
    expect = 0.5 * (math.log1p(math.exp(-t * (0.7 + 0.2))) + math.log1p(math.exp(-t * (0.4 - 0.1))))
    assert r["loss"] == pytest.approx(expect, rel=1e-14)


def test_balanced_equal_scores_closed_form():
    """One attract cell and k repel cells, all at the same score: each half's mean is its cell loss."""
    n = 5
    s = np.full((n, n), 0.3)
    t, b = 4.0, -1.0
    z = t * 0.3 + b
    att = synth.diagonal_edges(n)
    r = oracle.pair_loss_scores_form("balanced", s, t, b, att, ambient_weight=2.0)
    expect = math.log1p(math.exp(-z)) + math.log1p(math.exp(z))
    assert r["loss"] == pytest.approx(expect, rel=1e-13)


def test_balanced_halves_are_normalised_apart():
    """Scaling every attract weight, or every repel weight, by a constant changes nothing."""
    rng = np.random.default_rng(2)
    n = 8
    s = rng.normal(size=(n, n))
    A, R, I = _rel(rng, n)
    base = oracle.pair_loss_scores_form("balanced", s, 2.0, -0.5, A, R, I, negatives_named=True)
    A2 = synth.Edges(A.offsets, A.ids, A.weights * 3.7)
    R2 = synth.Edges(R.offsets, R.ids, R.weights * 0.25)
    x = oracle.pair_loss_scores_form("balanced", s, 2.0, -0.5, A2, R2, I, negatives_named=True)
    assert x["loss"] == pytest.approx(base["loss"], rel=1e-12)
    np.testing.assert_allclose(x["dscores"], base["dscores"], rtol=1e-10, atol=1e-15)


def test_balanced_reduces_to_sigmoid_with_one_cell_per_half():
    """A row with exactly one attract and one repel cell (weights one) has the sigmoid form's row loss."""
    rng = np.random.default_rng(3)
    n = 6
    s = rng.normal(size=(n, n))
    att = synth.diagonal_edges(n)
    rep = to_csr(n, [(i, (i + 1) % n) for i in range(n)])
    a = oracle.pair_loss_scores_form("balanced", s, 1.5, 0.25, att, rep, negatives_named=True)
    c = oracle.pair_loss_sigmoid_scores(s, 1.5, 0.25, att, rep, negatives_named=True)
    for k in ("loss", "dt", "db"):
        assert a[k] == pytest.approx(c[k], rel=1e-13)
    np.testing.assert_allclose(a["dscores"], c["dscores"], rtol=1e-13)


@pytest.mark.parametrize("form", ["balanced", "ranked"])
def test_forms_finite_differences(form):
    rng = np.random.default_rng(4 + (form == "ranked"))
    n = 6
    s = rng.normal(size=(n, n))
    A, R, I = _rel(rng, n)
    t, b = 2.0, -0.7

    def loss(s_, t_, b_):
        return oracle.pair_loss_scores_form(form, s_, t_, b_, A, R, I, ambient_weight=0.8)["loss"]

    base = oracle.pair_loss_scores_form(form, s, t, b, A, R, I, ambient_weight=0.8)
    h = 1e-6
    for i in range(n):
        for j in range(n):
            sp, sm = s.copy(), s.copy()
            sp[i, j] += h
            sm[i, j] -= h
            assert (loss(sp, t, b) - loss(sm, t, b)) / (2 * h) == pytest.approx(base["dscores"][i, j], rel=1e-6,
                                                                                abs=1e-9)
    assert (loss(s, t + h, b) - loss(s, t - h, b)) / (2 * h) == pytest.approx(base["dt"], rel=1e-6, abs=1e-9)
    assert (loss(s, t, b + h) - loss(s, t, b - h)) / (2 * h) == pytest.approx(base["db"], rel=1e-6, abs=1e-9)


@pytest.mark.parametrize("form", ["balanced", "ranked"])
def test_forms_sides_equal_explicit_ignores(form):
    rng = np.random.default_rng(6)
    n = 9
    s = rng.normal(size=(n, n))
    sides = rng.integers(1, 4, size=n).astype(np.uint8)
    diag = synth.diagonal_edges(n)
    a = oracle.pair_loss_scores_form(form, s, 1.0, 0.0, diag, sides=sides)
    ign = {(i, j) for i in range(n) for j in range(n) if not (sides[i] & 1) or not (sides[j] & 2)}
    c = oracle.pair_loss_scores_form(form, s, 1.0, 0.0, diag, ignore=to_csr(n, ign))
    assert a["loss"] == c["loss"] and a["dt"] == c["dt"]
    np.testing.assert_array_equal(a["dscores"], c["dscores"])
