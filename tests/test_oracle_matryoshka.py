"""Pins of the oracle's Matryoshka prefixes under the sigmoid pair loss (no GPU).

"Training", `uform_contrastive_t` (`matryoshka_dimensions`) and "UForm", section "Matryoshka-Like
Multi-Scale Embedders": every listed prefix is scored under the SigLIP loss on cosine similarities.  The
pins check what that fixes: the normalisation's gradient (closed form, finite differences), invariance to
the scale of a row, additivity over prefixes, and the bf16 rounding of the scored prefixes.
"""

import numpy as np
import pytest

import oracle
from tests.test_oracle import to_csr


def _case(seed, n, d, p_att=0.2):
    rng = np.random.default_rng(seed)
    e = rng.normal(size=(n, d))
    att = {(i, j): float(rng.uniform(0.5, 2.0)) for i in range(n) for j in range(n) if i != j and rng.random() < p_att}
    if not att:
        att = {(0, 1): 1.0}
    return e, to_csr(n, att.keys(), att)


def test_full_width_of_unit_rows_is_the_plain_loss_projected():
    """One prefix, the full width, unit rows: the loss is the plain loss and dE is its gradient with the
    radial component removed (the closed form of the normalisation's Jacobian at |e| = 1)."""
    e, att = _case(1, 7, 10)
    e /= np.linalg.norm(e, axis=1, keepdims=True)
    m = oracle.pair_loss_sigmoid_matryoshka(e, [10], 3.0, -1.0, att, round_prefix=False)
    p = oracle.pair_loss_sigmoid(e, 3.0, -1.0, att)
    assert m["loss"] == pytest.approx(p["loss"], rel=1e-14)
    assert m["dt"] == pytest.approx(p["dt"], rel=1e-13)
    assert m["db"] == pytest.approx(p["db"], rel=1e-13)
    g = p["de"]
    expect = g - np.sum(g * e, axis=1, keepdims=True) * e
    np.testing.assert_allclose(m["de"], expect, rtol=1e-12, atol=1e-15)
    # the radial component of every row's gradient vanishes
    np.testing.assert_allclose(np.sum(m["de"] * e, axis=1), 0.0, atol=1e-14)


def test_scaling_a_row_changes_only_its_gradient_scale():
    e, att = _case(2, 8, 12)
    base = oracle.pair_loss_sigmoid_matryoshka(e, [4, 8, 12], 2.0, -0.5, att, round_prefix=False)
    e2 = e.copy()
    e2[3] *= 7.5
    x = oracle.pair_loss_sigmoid_matryoshka(e2, [4, 8, 12], 2.0, -0.5, att, round_prefix=False)
    assert x["loss"] == pytest.approx(base["loss"], rel=1e-12)
    assert x["dt"] == pytest.approx(base["dt"], rel=1e-11)
    np.testing.assert_allclose(x["de"][3], base["de"][3] / 7.5, rtol=1e-10, atol=1e-15)
    np.testing.assert_allclose(np.delete(x["de"], 3, 0), np.delete(base["de"], 3, 0), rtol=1e-10, atol=1e-15)


def test_prefixes_add():
    e, att = _case(3, 9, 16)
    both = oracle.pair_loss_sigmoid_matryoshka(e, [8, 16], 1.5, 0.25, att)
    a = oracle.pair_loss_sigmoid_matryoshka(e, [8], 1.5, 0.25, att)
    c = oracle.pair_loss_sigmoid_matryoshka(e, [16], 1.5, 0.25, att)
    for k in ("loss", "dt", "db"):
        assert both[k] == pytest.approx(a[k] + c[k], rel=1e-13)
    np.testing.assert_allclose(both["de"], a["de"] + c["de"], rtol=1e-12, atol=1e-15)
    assert not np.any(a["de"][:, 8:]), "a prefix moves no feature past its width"


def test_finite_differences():
    e, att = _case(4, 6, 12)
    prefixes = [4, 8, 12]
    t, b = 2.0, -0.7
    rep = to_csr(6, [(0, 3), (2, 5)], {(0, 3): 0.8, (2, 5): 1.3})
    base = oracle.pair_loss_sigmoid_matryoshka(e, prefixes, t, b, att, rep, round_prefix=False)

    def loss(e_, t_, b_):
        return oracle.pair_loss_sigmoid_matryoshka(e_, prefixes, t_, b_, att, rep, round_prefix=False)["loss"]

    h = 1e-6
    for i in range(6):
        for k in range(12):
            ep, em = e.copy(), e.copy()
            ep[i, k] += h
            em[i, k] -= h
            assert (loss(ep, t, b) - loss(em, t, b)) / (2 * h) == pytest.approx(base["de"][i, k], rel=1e-6, abs=1e-9)
    assert (loss(e, t + h, b) - loss(e, t - h, b)) / (2 * h) == pytest.approx(base["dt"], rel=1e-6, abs=1e-9)
    assert (loss(e, t, b + h) - loss(e, t, b - h)) / (2 * h) == pytest.approx(base["db"], rel=1e-6, abs=1e-9)


def test_rounding_is_exact_where_the_prefix_is_representable():
    """Rows whose normalised prefixes are exactly bf16 (entries +-1/2 over a width of 4, +-1/4 over 16)
    score the same with and without the rounding step; the rounding itself is nearest-even."""
    rng = np.random.default_rng(5)
    e = rng.choice([-1.0, 1.0], size=(6, 16)) * 3.0
    att = to_csr(6, [(i, (i + 1) % 6) for i in range(6)])
    a = oracle.pair_loss_sigmoid_matryoshka(e, [4, 16], 4.0, -2.0, att, round_prefix=True)
    c = oracle.pair_loss_sigmoid_matryoshka(e, [4, 16], 4.0, -2.0, att, round_prefix=False)
    assert a["loss"] == c["loss"]
    np.testing.assert_array_equal(a["de"], c["de"])
    assert oracle.round_bf16(np.array([1.0 / 3.0]))[0] != 1.0 / 3.0
    assert oracle.round_bf16(np.array([1.0 + 2.0 ** -8]))[0] == 1.0            # a tie rounds to even
    assert oracle.round_bf16(np.array([1.0 + 3 * 2.0 ** -8]))[0] == 1.0 + 2.0 ** -6
