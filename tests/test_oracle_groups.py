"""Pins of the oracle's temperature groups under the sigmoid pair loss (no GPU).

"Training", `uform_contrastive_t` (`temperature_groups`: learnable (inverse temperature, bias) pairs, one
per group a step's items select).  Read as: a cell takes its anchor's pair.  The dense float64 formulation
is pinned to the C oracle (one group, every relation mode), to finite differences, and to invariances
that any per-anchor reading must keep.
"""

import numpy as np
import pytest

import oracle
from tests.test_oracle import random_relations as _random_dicts, to_csr


def random_relations(rng, n):
    att, rep, ign = _random_dicts(rng, n)
    return to_csr(n, att.keys(), att), to_csr(n, rep.keys(), rep), to_csr(n, ign)


@pytest.mark.parametrize("named", [False, True])
def test_one_group_is_the_c_oracle(named):
    rng = np.random.default_rng(1 + named)
    n = 12
    e = rng.normal(size=(n, 7))
    att, rep, ign = random_relations(rng, n)
    a = oracle.pair_loss_sigmoid_groups(e, np.zeros(n, int), [3.0], [-1.5], att, rep, ign, named, 0.6)
    c = oracle.pair_loss_sigmoid(e, 3.0, -1.5, att, rep, ign, named, 0.6)
    assert a["loss"] == pytest.approx(c["loss"], rel=1e-12)
    assert a["dt"][0] == pytest.approx(c["dt"], rel=1e-11)
    assert a["db"][0] == pytest.approx(c["db"], rel=1e-11)
    np.testing.assert_allclose(a["de"], c["de"], rtol=1e-10, atol=1e-14)


def test_equal_pairs_split_nothing_and_unused_groups_get_no_gradient():
    rng = np.random.default_rng(3)
    n = 10
    e = rng.normal(size=(n, 5))
    att, rep, ign = random_relations(rng, n)
    g = rng.integers(0, 3, size=n)
    g[g == 2] = 0                                  # group 2 selected by no item
    a = oracle.pair_loss_sigmoid_groups(e, g, [2.0, 2.0, 2.0], [0.5, 0.5, 0.5], att, rep, ign)
    c = oracle.pair_loss_sigmoid(e, 2.0, 0.5, att, rep, ign)
    assert a["loss"] == pytest.approx(c["loss"], rel=1e-12)
    np.testing.assert_allclose(a["de"], c["de"], rtol=1e-10, atol=1e-14)
    assert np.sum(a["dt"]) == pytest.approx(c["dt"], rel=1e-11)
    assert np.sum(a["db"]) == pytest.approx(c["db"], rel=1e-11)
    assert a["dt"][2] == 0.0 and a["db"][2] == 0.0


def test_relabelling_groups_permutes_their_gradients():
    rng = np.random.default_rng(4)
    n = 11
    e = rng.normal(size=(n, 6))
    att, rep, ign = random_relations(rng, n)
    g = rng.integers(0, 3, size=n)
    t, b = np.array([1.0, 4.0, -2.0]), np.array([0.3, -1.0, 2.0])
    perm = np.array([2, 0, 1])                     # old label k becomes perm[k]
    a = oracle.pair_loss_sigmoid_groups(e, g, t, b, att, rep, ign)
    tp, bp = np.empty(3), np.empty(3)
    tp[perm], bp[perm] = t, b
    c = oracle.pair_loss_sigmoid_groups(e, perm[g], tp, bp, att, rep, ign)
    assert c["loss"] == pytest.approx(a["loss"], rel=1e-13)
    np.testing.assert_allclose(c["dt"][perm], a["dt"], rtol=1e-12)
    np.testing.assert_allclose(c["db"][perm], a["db"], rtol=1e-12)
    np.testing.assert_allclose(c["de"], a["de"], rtol=1e-12, atol=1e-15)


def test_a_group_reaches_only_its_anchors_rows():
    """Changing group 1's pair changes the loss by exactly the change of the rows its items anchor."""
    rng = np.random.default_rng(5)
    n = 9
    e = rng.normal(size=(n, 4))
    att = to_csr(n, [(i, (i + 2) % n) for i in range(n)])
    g = np.array([0, 1, 0, 1, 1, 0, 0, 1, 0])
    a = oracle.pair_loss_sigmoid_groups(e, g, [2.0, 3.0], [-1.0, 0.5], att)
    c = oracle.pair_loss_sigmoid_groups(e, g, [2.0, -1.0], [-1.0, 2.0], att)
    rows0 = np.where(g == 0)[0]
    r_a = oracle.pair_loss_sigmoid(e, 2.0, -1.0, att, rows=rows0)
    r1_a = oracle.pair_loss_sigmoid(e, 3.0, 0.5, att, rows=np.where(g == 1)[0])
    r1_c = oracle.pair_loss_sigmoid(e, -1.0, 2.0, att, rows=np.where(g == 1)[0])
    assert a["loss"] == pytest.approx(r_a["loss"] + r1_a["loss"], rel=1e-12)
    assert c["loss"] - a["loss"] == pytest.approx(r1_c["loss"] - r1_a["loss"], rel=1e-10)


def test_finite_differences():
    rng = np.random.default_rng(6)
    n = 7
    e = rng.normal(size=(n, 5))
    att, rep, ign = random_relations(rng, n)
    g = np.array([0, 1, 1, 0, 2, 2, 1])
    t, b = np.array([1.5, -0.5, 2.5]), np.array([0.2, 0.7, -1.1])
    base = oracle.pair_loss_sigmoid_groups(e, g, t, b, att, rep, ign, False, 0.9)

    def loss(e_, t_, b_):
        return oracle.pair_loss_sigmoid_groups(e_, g, t_, b_, att, rep, ign, False, 0.9)["loss"]

    h = 1e-6
    for i in range(n):
        for k in range(5):
            ep, em = e.copy(), e.copy()
            ep[i, k] += h
            em[i, k] -= h
            assert (loss(ep, t, b) - loss(em, t, b)) / (2 * h) == pytest.approx(base["de"][i, k], rel=1e-6, abs=1e-9)
    for q in range(3):
        tp, tm, bp, bm = t.copy(), t.copy(), b.copy(), b.copy()
        tp[q] += h
        tm[q] -= h
        bp[q] += h
        bm[q] -= h
        assert (loss(e, tp, b) - loss(e, tm, b)) / (2 * h) == pytest.approx(base["dt"][q], rel=1e-6, abs=1e-9)
        assert (loss(e, t, bp) - loss(e, t, bm)) / (2 * h) == pytest.approx(base["db"][q], rel=1e-6, abs=1e-9)


# ---------------------------------------------------------------------------
# Anchor bands: one device's rows when the loss is sharded across devices ("UForm", section
# "Matryoshka-Like Multi-Scale Embedders": embeddings all-gathered into one similarity band, gradients
# reduce-scattered back), read as each rank scoring its own items' rows against every gathered column.
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("named", [False, True])
def test_band_shares_are_the_c_oracles_anchor_rows(named):
    """The C oracle evaluates listed anchors' rows on its own: a band's L, dt, db must be those rows'
    shares (this separates a band of rows from a band of columns)."""
    rng = np.random.default_rng(11 + named)
    n = 13
    e = rng.normal(size=(n, 6))
    att, rep, ign = random_relations(rng, n)
    for lo, cnt in ((0, 4), (4, 1), (5, 8)):
        a = oracle.pair_loss_sigmoid_groups(e, np.zeros(n, int), [2.0], [-1.0], att, rep, ign, named, 0.8,
                                            band=(lo, cnt))
        c = oracle.pair_loss_sigmoid(e, 2.0, -1.0, att, rep, ign, named, 0.8, rows=np.arange(lo, lo + cnt))
        assert a["loss"] == pytest.approx(c["loss"], rel=1e-12)
        assert a["dt"][0] == pytest.approx(c["dt"], rel=1e-11, abs=1e-15)
        assert a["db"][0] == pytest.approx(c["db"], rel=1e-11, abs=1e-15)


def test_bands_that_partition_the_rows_add_up():
    rng = np.random.default_rng(21)
    n = 11
    e = rng.normal(size=(n, 4))
    att, rep, ign = random_relations(rng, n)
    g = rng.integers(0, 3, size=n)
    t, b = np.array([1.5, -0.5, 2.5]), np.array([0.2, 0.7, -1.1])
    full = oracle.pair_loss_sigmoid_groups(e, g, t, b, att, rep, ign, False, 0.9)
    parts = [oracle.pair_loss_sigmoid_groups(e, g, t, b, att, rep, ign, False, 0.9, band=bd)
             for bd in ((0, 3), (3, 5), (8, 3))]
    assert sum(p["loss"] for p in parts) == pytest.approx(full["loss"], rel=1e-12)
    np.testing.assert_allclose(sum(p["dt"] for p in parts), full["dt"], rtol=1e-11, atol=1e-15)
    np.testing.assert_allclose(sum(p["db"] for p in parts), full["db"], rtol=1e-11, atol=1e-15)
    np.testing.assert_allclose(sum(p["de"] for p in parts), full["de"], rtol=1e-11, atol=1e-14)
    # a band's gradient reaches rows outside it (through the columns its anchors score)
    assert np.abs(parts[0]["de"][3:]).max() > 0


def test_band_finite_differences():
    """A band's dE, dt and db are the gradients of that band's loss share."""
    rng = np.random.default_rng(31)
    n, w = 7, 4
    e = rng.normal(size=(n, w))
    att, rep, ign = random_relations(rng, n)
    g = np.array([0, 1, 1, 0, 1, 0, 1])
    t, b = np.array([1.5, -0.5]), np.array([0.2, 0.7])
    band = (2, 3)
    base = oracle.pair_loss_sigmoid_groups(e, g, t, b, att, rep, ign, False, 0.9, band=band)

    def loss(e_, t_, b_):
        return oracle.pair_loss_sigmoid_groups(e_, g, t_, b_, att, rep, ign, False, 0.9, band=band)["loss"]

    h = 1e-6
    for i in range(n):
        for k in range(w):
            ep, em = e.copy(), e.copy()
            ep[i, k] += h
            em[i, k] -= h
            assert (loss(ep, t, b) - loss(em, t, b)) / (2 * h) == pytest.approx(base["de"][i, k], rel=1e-6, abs=1e-9)
    for q in range(2):
        tp, tm, bp, bm = t.copy(), t.copy(), b.copy(), b.copy()
        tp[q] += h
        tm[q] -= h
        bp[q] += h
        bm[q] -= h
        assert (loss(e, tp, b) - loss(e, tm, b)) / (2 * h) == pytest.approx(base["dt"][q], rel=1e-6, abs=1e-9)
        assert (loss(e, t, bp) - loss(e, t, bm)) / (2 * h) == pytest.approx(base["db"][q], rel=1e-6, abs=1e-9)
