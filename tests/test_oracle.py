"""Pins of the float64 oracle to facts outside itself (no GPU).

Each test states what it pins the oracle to: a closed form, a brute-force
second formulation, central finite differences, or an invariant.  Together
they are chosen so that a dropped term, a wrong sign, a wrong index, a
transposed operand or a wrong resolution order in the oracle fails one of
them.
"""

import itertools
import math

import numpy as np
import pytest

import oracle
from contrastive_late_interaction_gb300 import synth

LN2 = math.log(2.0)


# ---------------------------------------------------------------------------
# helpers written independently of the oracle
# ---------------------------------------------------------------------------

def dense_resolution(n, att, rep, ign, named, ambient, diagonal_skipped=True):
    """Brute-force per-pair resolution, following the documented order:
    ignore, then attract, then repel, then the run's negatives.
    att/rep: dict (i, j) -> weight; ign: set of (i, j).  Returns y, w arrays (w=0: skipped)."""
    y = np.zeros((n, n))
    w = np.zeros((n, n))
    for i in range(n):
        for j in range(n):
            if diagonal_skipped and i == j:
                continue
            if (i, j) in ign:
                continue
            if (i, j) in att:
                y[i, j], w[i, j] = 1.0, att[(i, j)]
            elif (i, j) in rep:
                y[i, j], w[i, j] = -1.0, rep[(i, j)]
            elif not named:
                y[i, j], w[i, j] = -1.0, ambient
    return y, w


def to_csr(n, pairs, weights=None):
    rows = [[] for _ in range(n)]
    for (i, j) in sorted(pairs):
        rows[i].append(j)
    off = np.zeros(n + 1, dtype=np.uint64)
    off[1:] = np.cumsum([len(r) for r in rows])
    ids = np.array([j for r in rows for j in r], dtype=np.uint32)
    w = None
    if weights is not None:
        w = np.array([weights[(i, j)] for i in range(n) for j in rows[i]], dtype=np.float64)
    return synth.Edges(off, ids, w)


def random_relations(rng, n, p=0.3, weighted=True):
    att, rep, ign = {}, {}, set()
    for i in range(n):
        for j in range(n):
            if rng.random() < p:
                att[(i, j)] = float(rng.uniform(0.2, 2.0)) if weighted else 1.0
            if rng.random() < p:
                rep[(i, j)] = float(rng.uniform(0.2, 2.0)) if weighted else 1.0
            if rng.random() < p / 2:
                ign.add((i, j))
    return att, rep, ign


def run_pooled(e, t, b, att, rep, ign, named, ambient, **kw):
    n = len(e)
    return oracle.pair_loss_sigmoid(e, t, b, to_csr(n, att.keys(), att), to_csr(n, rep.keys(), rep),
                                    to_csr(n, ign), named, ambient, **kw)


# ---------------------------------------------------------------------------
# scalar pieces: closed forms of sigma and softplus
# ---------------------------------------------------------------------------

def test_sigmoid_softplus_closed_forms():
    assert oracle.sigmoid(0.0) == 0.5
    assert oracle.softplus(0.0) == pytest.approx(LN2, rel=1e-15)
    assert oracle.softplus(10.0) == pytest.approx(10.0 + math.log1p(math.exp(-10.0)), rel=1e-15)
    assert oracle.softplus(-10.0) == pytest.approx(math.log1p(math.exp(-10.0)), rel=1e-15)
    for z in range(-30, 31):
        s, sm = oracle.sigmoid(z), oracle.sigmoid(-z)
        assert s + sm == pytest.approx(1.0, abs=1e-15)
        assert oracle.softplus(z) - oracle.softplus(-z) == pytest.approx(z, abs=1e-12)
        # -log sigma(z) = softplus(-z), and its derivative is sigma(z) - 1 = -sigma(-z)
        assert oracle.softplus(-z) == pytest.approx(math.log1p(math.exp(-z)), rel=1e-14)
        h = 1e-5
        fd = (oracle.softplus(-(z + h)) - oracle.softplus(-(z - h))) / (2 * h)
        assert fd == pytest.approx(-sm, rel=1e-7, abs=1e-12)


# ---------------------------------------------------------------------------
# pooled loss: closed forms
# ---------------------------------------------------------------------------

def test_collapsed_batch_closed_form():
    """All rows the same unit vector and t=10, b=-10: every z is 0, so each scored ordered pair costs
    w ln 2 and pulls/pushes with dl/dz = -w y / 2."""
    rng = np.random.default_rng(1)
    n, d = 10, 7
    e = np.zeros((n, d))
    e[:, 3] = 1.0
    att = {(i, i ^ 1): float(rng.uniform(0.5, 1.5)) for i in range(n)}
    rep = {(0, 5): 2.0, (7, 2): 0.25}
    ign = {(1, 4), (4, 1), (0, 1)}
    for named, ambient in ((False, 0.7), (True, 0.7)):
        y, w = dense_resolution(n, att, rep, ign, named, ambient)
        r = run_pooled(e, 10.0, -10.0, att, rep, ign, named, ambient)
        assert r["loss"] == pytest.approx(w.sum() * LN2 / n, rel=1e-14)
        g = -w * y / 2.0 / n          # dL/dz per ordered pair
        assert r["db"] == pytest.approx(g.sum(), rel=1e-13, abs=1e-15)
        assert r["dt"] == pytest.approx(g.sum(), rel=1e-13, abs=1e-15)   # s = 1 everywhere
        expect = 10.0 * (g.sum(axis=1) + g.sum(axis=0))[:, None] * e
        np.testing.assert_allclose(r["de"], expect, rtol=1e-13, atol=1e-15)


def test_orthogonal_batch_closed_form():
    """Basis rows (N <= D): every off-diagonal s is 0, so z = b; with b = -10 an attract costs
    softplus(10) and a repel softplus(-10); dE_i[k] = t (g_ik + g_ki)."""
    n, d = 6, 9
    e = np.eye(n, d)
    att = {(0, 1): 1.0, (1, 0): 1.0, (2, 3): 0.5, (5, 4): 3.0}
    rep = {(3, 2): 2.0}
    ign = {(4, 5)}
    t, b = 10.0, -10.0
    y, w = dense_resolution(n, att, rep, ign, False, 1.0)
    r = run_pooled(e, t, b, att, rep, ign, False, 1.0)
    sp_att, sp_rep = math.log1p(math.exp(-10.0)) + 10.0, math.log1p(math.exp(-10.0))
    loss = (w[y > 0].sum() * sp_att + w[y < 0].sum() * sp_rep) / n
    assert r["loss"] == pytest.approx(loss, rel=1e-14)
    sig = 1.0 / (1.0 + math.exp(10.0))      # sigma(b) for b = -10
    g = np.where(y > 0, -w * (1.0 - sig), np.where(y < 0, w * sig, 0.0)) / n
    assert r["db"] == pytest.approx(g.sum(), rel=1e-13)
    assert r["dt"] == 0.0
    expect = np.zeros((n, d))
    expect[:, :n] = t * (g + g.T)
    np.testing.assert_allclose(r["de"], expect, rtol=1e-13, atol=1e-16)


def test_two_items_one_attract_pair():
    """N = 2 with one attract pair named both ways: L = softplus(-(t s + b))."""
    rng = np.random.default_rng(2)
    e = rng.normal(size=(2, 5))
    e /= np.linalg.norm(e, axis=1, keepdims=True)
    s = float(e[0] @ e[1])
    for t, b in ((10.0, -10.0), (1.0, 0.0), (3.5, 1.25)):
        r = run_pooled(e, t, b, {(0, 1): 1.0, (1, 0): 1.0}, {}, set(), False, 1.0)
        z = t * s + b
        assert r["loss"] == pytest.approx(math.log1p(math.exp(-z)), rel=1e-13)


# ---------------------------------------------------------------------------
# pooled loss: finite differences, brute-force resolution, invariants
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("named", [False, True])
def test_pooled_gradients_finite_differences(named):
    rng = np.random.default_rng(3 + named)
    n, d = 6, 5
    e = rng.normal(size=(n, d))
    e /= np.linalg.norm(e, axis=1, keepdims=True)
    att, rep, ign = random_relations(rng, n)
    t, b, amb = 4.0, -1.5, 0.8
    base = run_pooled(e, t, b, att, rep, ign, named, amb)

    def loss(e_, t_, b_):
        return run_pooled(e_, t_, b_, att, rep, ign, named, amb, want_de=False)["loss"]

    h = 1e-6
    for i in range(n):
        for k in range(d):
            ep, em = e.copy(), e.copy()
            ep[i, k] += h
            em[i, k] -= h
            fd = (loss(ep, t, b) - loss(em, t, b)) / (2 * h)
            assert fd == pytest.approx(base["de"][i, k], rel=1e-6, abs=1e-8)
    fd_t = (loss(e, t + h, b) - loss(e, t - h, b)) / (2 * h)
    fd_b = (loss(e, t, b + h) - loss(e, t, b - h)) / (2 * h)
    assert fd_t == pytest.approx(base["dt"], rel=1e-6, abs=1e-8)
    assert fd_b == pytest.approx(base["db"], rel=1e-6, abs=1e-8)


def test_resolution_against_brute_force_enumeration():
    """For N <= 6 and random memberships in all three edge sets, the CSR-driven resolution must equal
    running with the brute-force resolved pairs spelled out as explicit attract/repel edges."""
    rng = np.random.default_rng(4)
    for trial in range(40):
        n = int(rng.integers(2, 7))
        att, rep, ign = random_relations(rng, n, p=0.35)
        named = bool(trial % 2)
        amb = float(rng.uniform(0.3, 1.7))
        e = rng.normal(size=(n, 4))
        e /= np.linalg.norm(e, axis=1, keepdims=True)
        t, b = float(rng.uniform(0.5, 12)), float(rng.uniform(-10, 2))
        got = run_pooled(e, t, b, att, rep, ign, named, amb)
        y, w = dense_resolution(n, att, rep, ign, named, amb)
        ea = {(i, j): w[i, j] for i in range(n) for j in range(n) if y[i, j] > 0}
        er = {(i, j): w[i, j] for i in range(n) for j in range(n) if y[i, j] < 0}
        ref = run_pooled(e, t, b, ea, er, set(), True, 123.0)
        for key in ("loss", "dt", "db"):
            assert got[key] == pytest.approx(ref[key], rel=1e-13, abs=1e-15)
        np.testing.assert_allclose(got["de"], ref["de"], rtol=1e-12, atol=1e-15)


def test_self_edges_have_no_effect():
    rng = np.random.default_rng(5)
    n = 5
    e = rng.normal(size=(n, 3))
    att = {(0, 1): 1.0, (1, 0): 1.0}
    a = run_pooled(e, 2.0, -1.0, att, {}, set(), False, 1.0)
    att2 = dict(att)
    att2.update({(i, i): 1.0 for i in range(n)})
    c = run_pooled(e, 2.0, -1.0, att2, {(2, 2): 5.0}, set(), False, 1.0)
    assert a["loss"] == c["loss"] and a["dt"] == c["dt"] and a["db"] == c["db"]


def test_permuting_items_permutes_gradients():
    inp = synth.pooled_bags(7, 48, 16, ignore_p=0.05)
    perm = np.random.default_rng(6).permutation(inp.count)
    inv = np.argsort(perm)
    e = inp.e_rounded

    def remap(edges):
        pairs = {}
        for i in range(edges.count):
            for k in range(int(edges.offsets[i]), int(edges.offsets[i + 1])):
                pairs[(int(inv[i]), int(inv[edges.ids[k]]))] = 1.0
        return pairs

    a = oracle.pair_loss_sigmoid(e, inp.t, inp.b, inp.attract, inp.repel, inp.ignore)
    pa, pi = remap(inp.attract), remap(inp.ignore)
    c = run_pooled(e[perm], inp.t, inp.b, pa, {}, set(pi.keys()), False, 1.0)
    assert c["loss"] == pytest.approx(a["loss"], rel=1e-12)
    assert c["dt"] == pytest.approx(a["dt"], rel=1e-12)
    assert c["db"] == pytest.approx(a["db"], rel=1e-12)
    np.testing.assert_allclose(c["de"], a["de"][perm], rtol=1e-10, atol=1e-14)


def test_zero_padding_width_changes_nothing():
    inp = synth.pooled_bags(8, 40, 12)
    e = inp.e_rounded
    a = oracle.pair_loss_sigmoid(e, inp.t, inp.b, inp.attract)
    c = oracle.pair_loss_sigmoid(np.hstack([e, np.zeros((40, 5))]), inp.t, inp.b, inp.attract)
    assert (a["loss"], a["dt"], a["db"]) == (c["loss"], c["dt"], c["db"])
    np.testing.assert_array_equal(c["de"][:, :12], a["de"])
    np.testing.assert_array_equal(c["de"][:, 12:], 0.0)


def test_thread_count_and_row_subsets_agree():
    inp = synth.pooled_bags(9, 64, 8, ignore_p=0.1)
    e = inp.e_rounded
    a = oracle.pair_loss_sigmoid(e, inp.t, inp.b, inp.attract, ignore=inp.ignore, threads=1)
    c = oracle.pair_loss_sigmoid(e, inp.t, inp.b, inp.attract, ignore=inp.ignore, threads=7)
    assert (a["loss"], a["dt"], a["db"]) == (c["loss"], c["dt"], c["db"])
    rows = np.array([5, 0, 63, 17])
    s = oracle.pair_loss_sigmoid(e, inp.t, inp.b, inp.attract, ignore=inp.ignore, rows=rows)
    np.testing.assert_array_equal(s["de"], a["de"][rows])
    np.testing.assert_array_equal(s["row_loss"], a["row_loss"][rows])


# ---------------------------------------------------------------------------
# loss over a given score matrix
# ---------------------------------------------------------------------------

def test_score_matrix_loss_matches_pooled_on_gram_matrix():
    """The score-matrix form on S = E E^T, with the diagonal ignored, is the pooled loss; and the chain
    rule through S gives dE = (dS + dS^T) E."""
    inp = synth.pooled_bags(10, 30, 6, ignore_p=0.1)
    e = inp.e_rounded
    pooled = oracle.pair_loss_sigmoid(e, inp.t, inp.b, inp.attract, ignore=inp.ignore)
    n = inp.count
    ign = {(i, int(inp.ignore.ids[k])) for i in range(n)
           for k in range(int(inp.ignore.offsets[i]), int(inp.ignore.offsets[i + 1]))}
    ign |= {(i, i) for i in range(n)}
    sc = oracle.pair_loss_sigmoid_scores(e @ e.T, inp.t, inp.b, inp.attract, ignore=to_csr(n, ign))
    assert sc["loss"] == pytest.approx(pooled["loss"], rel=1e-12)
    assert sc["dt"] == pytest.approx(pooled["dt"], rel=1e-12)
    assert sc["db"] == pytest.approx(pooled["db"], rel=1e-12)
    np.testing.assert_allclose((sc["dscores"] + sc["dscores"].T) @ e, pooled["de"], rtol=1e-10, atol=1e-14)


def test_score_matrix_sides_equal_explicit_ignores():
    rng = np.random.default_rng(11)
    n = 9
    s = rng.normal(size=(n, n))
    sides = rng.integers(1, 4, size=n).astype(np.uint8)
    diag = synth.diagonal_edges(n)
    a = oracle.pair_loss_sigmoid_scores(s, 1.0, 0.0, diag, sides=sides)
    ign = {(i, j) for i in range(n) for j in range(n) if not (sides[i] & 1) or not (sides[j] & 2)}
    c = oracle.pair_loss_sigmoid_scores(s, 1.0, 0.0, diag, ignore=to_csr(n, ign))
    assert a["loss"] == c["loss"] and a["dt"] == c["dt"] and a["db"] == c["db"]
    np.testing.assert_array_equal(a["dscores"], c["dscores"])


def test_score_matrix_zero_scores_closed_form():
    n = 7
    diag = synth.diagonal_edges(n)
    r = oracle.pair_loss_sigmoid_scores(np.zeros((n, n)), 1.0, 0.0, diag)
    assert r["loss"] == pytest.approx(n * n * LN2 / n, rel=1e-14)
    assert r["db"] == pytest.approx((n * (n - 1) * 0.5 - n * 0.5) / n, rel=1e-14)


def test_score_matrix_finite_differences():
    rng = np.random.default_rng(12)
    n = 5
    s = rng.normal(size=(n, n))
    att, rep, ign = random_relations(rng, n)
    A, R, I = to_csr(n, att.keys(), att), to_csr(n, rep.keys(), rep), to_csr(n, ign)
    t, b = 2.5, -0.5
    base = oracle.pair_loss_sigmoid_scores(s, t, b, A, R, I, ambient_weight=0.6)
    h = 1e-6
    for i, j in itertools.product(range(n), range(n)):
        sp, sm = s.copy(), s.copy()
        sp[i, j] += h
        sm[i, j] -= h
        fd = (oracle.pair_loss_sigmoid_scores(sp, t, b, A, R, I, ambient_weight=0.6)["loss"] -
              oracle.pair_loss_sigmoid_scores(sm, t, b, A, R, I, ambient_weight=0.6)["loss"]) / (2 * h)
        assert fd == pytest.approx(base["dscores"][i, j], rel=1e-6, abs=1e-9)


# ---------------------------------------------------------------------------
# hard MaxSim
# ---------------------------------------------------------------------------

def brute_maxsim(q_off, q, d_off, d, mean=False):
    """Second formulation: the full Q D^T matrix, then a max over each document's column slice."""
    full = q @ d.T
    nq, nd = len(q_off) - 1, len(d_off) - 1
    s = np.zeros((nq, nd))
    arg = np.zeros((nd, len(q)), dtype=np.int64)
    for j in range(nd):
        blk = full[:, int(d_off[j]):int(d_off[j + 1])]
        arg[j] = np.argmax(blk, axis=1)        # first occurrence: lowest index
        m = blk.max(axis=1)
        for i in range(nq):
            seg = m[int(q_off[i]):int(q_off[i + 1])]
            s[i, j] = seg.sum() / (len(seg) if mean else 1.0)
    return s, arg


@pytest.mark.parametrize("mean", [False, True])
def test_maxsim_forward_against_full_matrix(mean):
    mi = synth.maxsim_random(13, 7, 9, 16, (1, 6), (1, 11))
    s, arg, gap = oracle.maxsim_forward(mi.q_offsets, mi.q, mi.d_offsets, mi.d, mean)
    bs, barg = brute_maxsim(mi.q_offsets, mi.q, mi.d_offsets, mi.d, mean)
    np.testing.assert_allclose(s, bs, rtol=1e-12, atol=1e-14)
    sure = gap > 1e-9
    np.testing.assert_array_equal(arg[sure], barg[sure])
    assert sure.mean() > 0.9


def test_maxsim_single_row_document():
    mi = synth.maxsim_random(14, 5, 4, 8, (1, 5), (1, 1))
    s, arg, _ = oracle.maxsim_forward(mi.q_offsets, mi.q, mi.d_offsets, mi.d)
    for i in range(mi.nq):
        qs = mi.q[int(mi.q_offsets[i]):int(mi.q_offsets[i + 1])].sum(axis=0)
        for j in range(mi.nd):
            assert s[i, j] == pytest.approx(float(qs @ mi.d[int(mi.d_offsets[j])]), rel=1e-12, abs=1e-14)
    assert (arg == 0).all()


def test_maxsim_width_one():
    rng = np.random.default_rng(15)
    q = rng.normal(size=(6, 1))
    d = rng.normal(size=(10, 1))
    q_off = np.array([0, 2, 6], dtype=np.uint64)
    d_off = np.array([0, 3, 10], dtype=np.uint64)
    s, arg, _ = oracle.maxsim_forward(q_off, q, d_off, d)
    for i in range(2):
        for j in range(2):
            dv = d[int(d_off[j]):int(d_off[j + 1]), 0]
            exp = sum(x * (dv.max() if x > 0 else dv.min()) for x in q[int(q_off[i]):int(q_off[i + 1]), 0])
            assert s[i, j] == pytest.approx(exp, rel=1e-14)
    for t in range(6):
        dv = d[0:3, 0]
        assert arg[0, t] == (int(np.argmax(dv)) if q[t, 0] > 0 else int(np.argmin(dv)))


def test_maxsim_query_copied_from_document():
    """Exact unit rows (distinct basis vectors): a query made of rows of a document scores |q| against
    it, and the argmax points at the copied positions."""
    d = np.eye(12)[[3, 7, 1, 9, 0, 5, 11, 2]]
    d_off = np.array([0, 5, 8], dtype=np.uint64)
    pick = [4, 1, 2]
    q = d[pick]
    q_off = np.array([0, 3], dtype=np.uint64)
    s, arg, gap = oracle.maxsim_forward(q_off, q, d_off, d)
    assert s[0, 0] == 3.0
    assert list(arg[0]) == pick
    assert (gap[0] == 1.0).all()


def test_maxsim_ties_go_to_the_lowest_index():
    d = np.array([[0.5, 0.5], [1.0, 0.0], [0.5, 0.5], [1.0, 0.0]])
    q = np.array([[1.0, 0.0], [0.0, 1.0]])
    s, arg, gap = oracle.maxsim_forward(np.array([0, 2], np.uint64), q, np.array([0, 4], np.uint64), d)
    assert list(arg[0]) == [1, 0]
    assert (gap[0] == 0.0).all()


def test_maxsim_permutations():
    mi = synth.maxsim_random(16, 6, 5, 8, (2, 5), (2, 7))
    s, arg, _ = oracle.maxsim_forward(mi.q_offsets, mi.q, mi.d_offsets, mi.d)
    # permuting documents permutes the columns of S
    perm = np.array([3, 0, 4, 1, 2])
    lens = np.diff(mi.d_offsets.astype(np.int64))
    d2 = np.concatenate([mi.d[int(mi.d_offsets[j]):int(mi.d_offsets[j + 1])] for j in perm])
    s2, arg2, _ = oracle.maxsim_forward(mi.q_offsets, mi.q, synth.ragged_offsets(lens[perm]), d2)
    np.testing.assert_allclose(s2, s[:, perm], rtol=1e-13)
    np.testing.assert_array_equal(arg2, arg[perm])
    # permuting the rows inside one document leaves S alone and remaps the argmax
    rows = np.arange(len(mi.d))
    j = 2
    o0, o1 = int(mi.d_offsets[j]), int(mi.d_offsets[j + 1])
    local = np.random.default_rng(17).permutation(o1 - o0)
    rows[o0:o1] = o0 + local
    s3, arg3, gap3 = oracle.maxsim_forward(mi.q_offsets, mi.q, mi.d_offsets, mi.d[rows])
    np.testing.assert_allclose(s3, s, rtol=1e-13)
    sure = gap3[j] > 1e-9
    np.testing.assert_array_equal(local[arg3[j]][sure], arg[j][sure])


@pytest.mark.parametrize("mean", [False, True])
def test_maxsim_mean_and_sum_agree(mean):
    mi = synth.maxsim_random(18, 4, 6, 8, (1, 9), (3, 8))
    s_sum, a_sum, _ = oracle.maxsim_forward(mi.q_offsets, mi.q, mi.d_offsets, mi.d, False)
    s_mean, a_mean, _ = oracle.maxsim_forward(mi.q_offsets, mi.q, mi.d_offsets, mi.d, True)
    lens = np.diff(mi.q_offsets.astype(np.int64))
    np.testing.assert_allclose(s_mean * lens[:, None], s_sum, rtol=1e-13)
    np.testing.assert_array_equal(a_mean, a_sum)


@pytest.mark.parametrize("mean", [False, True])
def test_maxsim_backward_finite_differences(mean):
    """sum(dS * S) is piecewise linear in Q and D; away from ties its finite-difference gradient is
    the argmax-routed one."""
    mi = synth.maxsim_random(19, 3, 4, 6, (2, 4), (2, 5))
    rng = np.random.default_rng(20)
    ds = rng.normal(size=(mi.nq, mi.nd))
    s, arg, gap = oracle.maxsim_forward(mi.q_offsets, mi.q, mi.d_offsets, mi.d, mean)
    assert gap.min() > 1e-4
    dq, dd = oracle.maxsim_backward(mi.q_offsets, mi.q, mi.d_offsets, mi.d, arg, ds, mean)

    def obj(q, d):
        return float((ds * oracle.maxsim_forward(mi.q_offsets, q, mi.d_offsets, d, mean)[0]).sum())

    h = 1e-7
    for (mat, grad, which) in ((mi.q, dq, 0), (mi.d, dd, 1)):
        for r in range(mat.shape[0]):
            for k in range(mat.shape[1]):
                p, m = mat.copy(), mat.copy()
                p[r, k] += h
                m[r, k] -= h
                fd = (obj(p, mi.d) - obj(m, mi.d)) / (2 * h) if which == 0 else \
                     (obj(mi.q, p) - obj(mi.q, m)) / (2 * h)
                assert fd == pytest.approx(grad[r, k], rel=1e-6, abs=1e-7)


def test_maxsim_sampled_helpers_match_full_oracle():
    mi = synth.maxsim_random(21, 5, 6, 8, (1, 5), (1, 9))
    rng = np.random.default_rng(22)
    ds = rng.normal(size=(mi.nq, mi.nd))
    s, arg, gap = oracle.maxsim_forward(mi.q_offsets, mi.q, mi.d_offsets, mi.d)
    dq, dd = oracle.maxsim_backward(mi.q_offsets, mi.q, mi.d_offsets, mi.d, arg, ds)
    ps, pa, pg = oracle.maxsim_pairs(mi.q_offsets, mi.q, mi.d_offsets, mi.d, [0, 4, 2], [5, 1, 1])
    for k, (i, j) in enumerate([(0, 5), (4, 1), (2, 1)]):
        assert ps[k] == s[i, j]
        np.testing.assert_array_equal(pa[k], arg[j, int(mi.q_offsets[i]):int(mi.q_offsets[i + 1])])
    for i in range(mi.nq):
        np.testing.assert_allclose(oracle.maxsim_grad_query(mi.q_offsets, mi.q, mi.d_offsets, mi.d, i, ds[i]),
                                   dq[int(mi.q_offsets[i]):int(mi.q_offsets[i + 1])], rtol=1e-13, atol=1e-15)
    for j in range(mi.nd):
        np.testing.assert_allclose(oracle.maxsim_grad_doc(mi.q_offsets, mi.q, mi.d_offsets, mi.d, j, ds[:, j]),
                                   dd[int(mi.d_offsets[j]):int(mi.d_offsets[j + 1])], rtol=1e-13, atol=1e-15)


def test_tiny_workloads_run():
    p = synth.pooled_tiny()
    r = oracle.pair_loss_sigmoid(p.e_rounded, p.t, p.b, p.attract)
    assert np.isfinite(r["loss"]) and r["de"].shape == (256, 64)
    # 128 bags of 2, ambient repel, diagonal skipped: 256 attract and 256*254 repel ordered pairs
    assert int(p.attract.offsets[-1]) == 256
    m = synth.maxsim_tiny()
    s, arg, gap = oracle.maxsim_forward(m.q_offsets, m.q, m.d_offsets, m.d)
    assert s.shape == (16, 16) and arg.shape == (16, 128)
