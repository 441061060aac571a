"""CUDA path (through the C ABI) against the float64 oracle, on the same seeded inputs.

Small cases compare every output; the full-size workloads compare sampled outputs the oracle can
compute one at a time, plus properties that hold at any size.
"""

import numpy as np
import pytest
import torch

import oracle
from contrastive_late_interaction_gb300 import synth

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

if torch.cuda.is_available():
    import contrastive_late_interaction_gb300 as cli
    from tests.gpu_util import (GRAD_RL2, LOSS_RTOL, assert_rel, bf16, check_argmax, check_scores, i64, rel_l2,
                                routed_argmax, run_maxsim, run_pooled, scalar, dev)


# ---------------------------------------------------------------------------
# pooled sigmoid pair loss
# ---------------------------------------------------------------------------

def compare_pooled(p, g, ref):
    assert g["status"] == 0, cli.status_name(g["status"])
    assert_rel(g["loss"], ref["loss"], LOSS_RTOL, "loss")
    assert_rel(g["dt"], ref["dt"], GRAD_RL2, "dt")
    assert_rel(g["db"], ref["db"], GRAD_RL2, "db")
    e = rel_l2(g["de"], ref["de"])
    assert e <= GRAD_RL2, f"dE rel L2 {e:.3e}"


def test_pooled_tiny():
    """N=256, D=64, 128 bags of two, ambient repel, t=10, b=-10."""
    p = synth.pooled_tiny()
    g = run_pooled(p)
    ref = oracle.pair_loss_sigmoid(p.e_rounded, p.t, p.b, p.attract)
    compare_pooled(p, g, ref)


def test_pooled_config2_full():
    """N=4096, D=512, bags U{1..4}, 1% ignored ordered pairs: every output against the full oracle."""
    p = synth.pooled_config2()
    g = run_pooled(p)
    ref = oracle.pair_loss_sigmoid(p.e_rounded, p.t, p.b, p.attract, ignore=p.ignore)
    compare_pooled(p, g, ref)


@pytest.mark.parametrize("n,width,named", [(300, 72, False), (129, 8, True), (1000, 200, False), (2, 64, False),
                                            (200, 1024, False), (130, 4096, True)])   # up to the widest width
def test_pooled_ragged_weighted(n, width, named):
    """Ragged tiles (N and D not multiples of the tile), weighted attract and repel edges, ignores,
    both negatives modes, padded input and output row strides."""
    rng = np.random.default_rng(n + width)
    p = synth.pooled_bags(3, n, width, ignore_p=0.02, bag_size=2 if n == 2 else None)
    p.attract.weights = rng.uniform(0.2, 2.0, size=p.attract.ids.size).astype(np.float32)
    rep_lists = [sorted(set(rng.choice(n, size=min(n, 3), replace=False).tolist()) - {i}) for i in range(n)]
    rep = synth.edges_from_lists(rep_lists)
    rep.weights = rng.uniform(0.1, 3.0, size=rep.ids.size).astype(np.float32)
    p.repel = rep
    p.negatives_named = named
    p.ambient_weight = 0.75
    p.t, p.b = 7.0, -3.0
    g = run_pooled(p, ld=width + 8, ld_de=width + 4)
    ref = oracle.pair_loss_sigmoid(p.e_rounded, p.t, p.b, p.attract, p.repel, p.ignore, named, 0.75)
    compare_pooled(p, g, ref)
    pad = g["raw"]["d_embeddings"].as_strided((n, 4), (width + 4, 1), width)
    assert torch.all(pad == 7.0), "columns past the width were written"


@pytest.mark.parametrize("t,b", [(10.0, 10.0), (-10.0, -10.0), (1.0, 0.0), (-4.0, 6.0)])
def test_pooled_score_regimes(t, b):
    """Every regime of z = t s + b the epilogue distinguishes: all cells far positive, far negative with a
    negative temperature, near zero, and a mix."""
    p = synth.pooled_bags(5, 300, 64, ignore_p=0.01)
    p.t, p.b = t, b
    g = run_pooled(p)
    ref = oracle.pair_loss_sigmoid(p.e_rounded, t, b, p.attract, None, p.ignore, p.negatives_named, p.ambient_weight)
    compare_pooled(p, g, ref)


def test_pooled_config4_full():
    """N=32768, D=768, bags of four: L, dt, db and every dE row against the full oracle (every anchor)."""
    p = synth.pooled_config4()
    g = run_pooled(p)
    ref = oracle.pair_loss_sigmoid(p.e_rounded, p.t, p.b, p.attract)
    compare_pooled(p, g, ref)


def test_pooled_config4_permutation_invariance():
    """The items of config 4 permuted: L, dt and db unchanged, dE permuted (GPU against GPU, the rows
    landing in other tiles and blocks)."""
    p = synth.pooled_config4()
    g = run_pooled(p)
    assert g["status"] == 0
    perm = np.random.default_rng(0).permutation(p.count)
    inv = np.argsort(perm)
    bag = np.arange(p.count) // 4
    q = synth.PooledInputs(p.count, p.width, p.e_f32[perm], p.e_bf16[perm], p.t, p.b,
                           synth.attract_within_bags(bag[perm]), synth.empty_edges(p.count),
                           synth.empty_edges(p.count))
    g2 = run_pooled(q)
    assert_rel(g2["loss"], g["loss"], 1e-4, "permuted loss")
    assert_rel(g2["dt"], g["dt"], 1e-3, "permuted dt")
    assert_rel(g2["db"], g["db"], 1e-3, "permuted db")
    assert rel_l2(g2["de"][inv], g["de"]) <= 1e-3
    assert np.isfinite(g["loss"]) and g["loss"] > 0


def test_pooled_malformed_edges_report_on_device():
    """ids out of order or out of range are found by the validation kernel; the call reports
    CLI_MALFORMED in the device status and the compute kernels do nothing."""
    p = synth.pooled_tiny()
    lists = [[5, 3]] + [[(i + 1) % 256] for i in range(1, 256)]
    unsorted = synth.Edges(synth.ragged_offsets([len(x) for x in lists]),
                           np.array([j for x in lists for j in x], dtype=np.uint32))
    ids = p.attract.ids.copy()
    ids[3] = 999
    out_of_range = synth.Edges(p.attract.offsets.copy(), ids)
    for edges in (unsorted, out_of_range):
        q = synth.PooledInputs(p.count, p.width, p.e_f32, p.e_bf16, p.t, p.b, edges, p.repel, p.ignore)
        g = run_pooled(q)
        assert g["status"] == 5, cli.status_name(g["status"])


def test_pooled_refuses_a_step_without_attract_edges():
    p = synth.pooled_tiny()
    e = bf16(p.e_bf16)
    with pytest.raises(cli.InvalidArgumentError):
        cli.pair_loss_sigmoid_fwd_bwd(e, scalar(10), scalar(-10), None)


# ---------------------------------------------------------------------------
# MaxSim
# ---------------------------------------------------------------------------

def compare_maxsim_full(m, mean=False):
    g = run_maxsim(m, mean=mean)
    assert g["status_f"] == 0 and g["status_b"] == 0
    s, arg, gap = oracle.maxsim_forward(m.q_offsets, m.q, m.d_offsets, m.d, mean)
    check_scores(g["scores"], s)
    decided = check_argmax(g["argmax"], arg, gap)
    assert decided > 0.9 * arg.size
    arg = routed_argmax(m, g["argmax"], arg, gap)
    dq, dd = oracle.maxsim_backward(m.q_offsets, m.q, m.d_offsets, m.d, arg, m.d_scores, mean)
    assert rel_l2(g["dq"], dq) <= GRAD_RL2
    assert rel_l2(g["dd"], dd) <= GRAD_RL2
    return g


@pytest.mark.parametrize("mean", [False, True])
def test_maxsim_tiny(mean):
    compare_maxsim_full(synth.maxsim_tiny(), mean)


@pytest.mark.parametrize("seed,nq,nd,width,ql,dl", [
    (1, 40, 30, 128, (1, 70), (1, 300)),      # queries straddle 128-row blocks; one-row documents
    (2, 7, 50, 72, (3, 9), (1, 5)),           # many documents per tile, width not a multiple of 64
    (3, 3, 4, 256, (100, 200), (500, 900)),   # long queries and documents, the widest width
    (4, 300, 3, 8, (1, 3), (1000, 1300)),     # width 8
    (6, 5000, 3, 64, (1, 2), (5, 40)),        # more queries than the backward's shared table of c(q, d)
    (7, 70000, 2, 64, (1, 1), (3, 20)),       # more queries than its list entries can name
    (8, 6, 3, 128, (5, 40), (5000, 9000)),    # documents longer than the backward's 4096-row window
    (9, 4, 2, 64, (8, 16), (70000, 70000)),   # argmax indices past 16 bits
])
def test_maxsim_ragged(seed, nq, nd, width, ql, dl):
    compare_maxsim_full(synth.maxsim_random(seed, nq, nd, width, ql, dl))


def test_maxsim_backward_routes_a_given_argmax():
    """With the same (valid, random) argmax on both sides the backward is a pure routing: it must agree
    to fp32 accumulation error."""
    m = synth.maxsim_random(5, 60, 45, 128, (4, 40), (10, 200))
    am = synth.random_argmax(6, m)
    g = run_maxsim(m, argmax=am)
    dq, dd = oracle.maxsim_backward(m.q_offsets, m.q, m.d_offsets, m.d, am, m.d_scores)
    assert rel_l2(g["dq"], dq) <= 1e-5
    assert rel_l2(g["dd"], dd) <= 1e-5


@pytest.mark.parametrize("mean", [False, True])
def test_maxsim_backward_skips_inactive_queries_and_documents(mean):
    """dS with whole rows (queries) and columns (documents) zero, as a loss that ignores them gives: the
    backward skips those queries' warps and documents' blocks and walks the list of active documents; dQ
    and dD (zeros included) equal the oracle's routing of the same argmax, and an argmax entry that
    only zero-c pairs would read is not checked."""
    m = synth.maxsim_random(8, 90, 70, 128, (3, 50), (5, 260))
    am = synth.random_argmax(9, m)
    ds = np.array(m.d_scores, dtype=np.float32)
    rng = np.random.default_rng(10)
    dead_q = rng.random(m.nq) < 0.35
    dead_d = rng.random(m.nd) < 0.35
    ds[dead_q, :] = 0.0
    ds[:, dead_d] = 0.0
    d0 = int(np.nonzero(dead_d)[0][0])
    am[d0, 0] = 10 ** 6                      # outside its document, but only zero-c pairs would read it
    q, qo, d, do = bf16(m.q_bf16), i64(m.q_offsets), bf16(m.d_bf16), i64(m.d_offsets)
    g = cli.maxsim_backward(q, qo, d, do, torch.from_numpy(am).to(dev()), torch.from_numpy(ds).to(dev()),
                            mean=mean)
    torch.cuda.synchronize()
    assert int(g["device_status"].item()) == 0
    am[d0, 0] = 0
    dq, dd = oracle.maxsim_backward(m.q_offsets, m.q, m.d_offsets, m.d, am, ds.astype(np.float64), mean)
    gq, gd = g["d_queries"].double().cpu().numpy(), g["d_documents"].double().cpu().numpy()
    assert rel_l2(gq, dq) <= 1e-5 and rel_l2(gd, dd) <= 1e-5
    rq = np.repeat(np.arange(m.nq), np.diff(m.q_offsets.astype(np.int64)))
    rd = np.repeat(np.arange(m.nd), np.diff(m.d_offsets.astype(np.int64)))
    assert np.all(gq[dead_q[rq]] == 0.0) and np.all(gd[dead_d[rd]] == 0.0)


def test_maxsim_copied_queries_find_themselves():
    """A query made of rows copied from a document matches them exactly there (config-5 structure)."""
    j = synth.joint(0, pooled_count=256, pooled_width=64, items=24, d_len=(8, 40), q_len=(2, 8))
    g = run_maxsim(j.maxsim)
    m = j.maxsim
    for i in range(m.nq):
        t0, t1 = int(m.q_offsets[i]), int(m.q_offsets[i + 1])
        assert np.array_equal(g["argmax"][i, t0:t1], np.arange(t1 - t0))


def test_maxsim_config3_full():
    """512 x 512, |q| U{8..64}, |d| U{32..1024}, D=128: the whole score matrix, every decided argmax entry,
    and the whole dQ and dD against the full oracle."""
    compare_maxsim_full(synth.maxsim_config3())


def test_maxsim_device_faults_are_reported():
    m = synth.maxsim_tiny()
    q, qo, d, do = bf16(m.q_bf16), i64(m.q_offsets), bf16(m.d_bf16), i64(m.d_offsets)
    bad = m.d_offsets.copy()
    bad[3] = bad[2]                          # an empty document
    f = cli.maxsim_scores(q, qo, d, i64(bad))
    assert int(f["device_status"].item()) == 1
    bad = m.d_offsets.copy()
    bad[5], bad[6] = bad[6], bad[5]          # offsets going backwards
    f = cli.maxsim_scores(q, qo, d, i64(bad))
    assert int(f["device_status"].item()) == 5
    f = cli.maxsim_scores(q, qo, d, do)
    am = f["argmax"].clone()
    am[2, 7] = 32                            # outside its document (row 7 is query 0's)
    ds = torch.ones(16, 16, device=dev())
    g = cli.maxsim_backward(q, qo, d, do, am, ds)
    assert int(g["device_status"].item()) == 5
    ds[0, 2] = 0.0                           # the entry's pair has c = 0: it is not read, nor checked
    g = cli.maxsim_backward(q, qo, d, do, am, ds)
    assert int(g["device_status"].item()) == 0


# ---------------------------------------------------------------------------
# loss over a score matrix, and the joint step
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("with_sides", [False, True])
def test_score_matrix_loss(with_sides):
    rng = np.random.default_rng(7)
    n = 300
    s = rng.normal(scale=3.0, size=(n, n)).astype(np.float32)
    sides = rng.integers(1, 4, size=n).astype(np.uint8) if with_sides else None
    diag = synth.diagonal_edges(n)
    ign = synth.ignore_bernoulli(8, n, 0.05)
    S = torch.from_numpy(s).to(dev())
    r = cli.pair_loss_sigmoid_scores_fwd_bwd(S, scalar(1.5), scalar(-0.5), cli.device_edges(diag),
                                             ignore=cli.device_edges(ign),
                                             sides=None if sides is None else torch.from_numpy(sides).to(dev()))
    torch.cuda.synchronize()
    assert int(r["device_status"].item()) == 0
    ref = oracle.pair_loss_sigmoid_scores(s.astype(np.float64), 1.5, -0.5, diag, ignore=ign, sides=sides)
    assert_rel(r["loss"].item(), ref["loss"], LOSS_RTOL, "loss")
    assert_rel(r["d_inverse_temperature"].item(), ref["dt"], GRAD_RL2, "dt")
    assert_rel(r["d_bias"].item(), ref["db"], GRAD_RL2, "db")
    assert rel_l2(r["d_scores"].double().cpu().numpy(), ref["dscores"]) <= GRAD_RL2


def maxsim_rows_of_query(m, g_arg, qi, d_scores):
    """dQ rows of query qi from the oracle's backward over (query qi, every document), routed through the
    GPU's argmax where the oracle's choice is open."""
    t0, t1 = int(m.q_offsets[qi]), int(m.q_offsets[qi + 1])
    alld = np.arange(m.nd)
    _, pa, pg = oracle.maxsim_pairs(m.q_offsets, m.q, m.d_offsets, m.d, np.full(m.nd, qi), alld)
    check_argmax(g_arg[:, t0:t1], np.stack(pa), np.stack(pg))
    arg = routed_argmax(m, g_arg[:, t0:t1], np.stack(pa), np.stack(pg), rows=np.arange(t0, t1))
    ref, _ = oracle.maxsim_backward(np.array([0, t1 - t0], np.uint64), m.q[t0:t1], m.d_offsets, m.d, arg,
                                    d_scores[qi:qi + 1])
    return ref


def maxsim_rows_of_document(m, g_arg, di, d_scores):
    """dD rows of document di from the oracle's backward over (every query, document di), routed the same
    way."""
    r0, r1 = int(m.d_offsets[di]), int(m.d_offsets[di + 1])
    allq = np.arange(m.nq)
    _, pa, pg = oracle.maxsim_pairs(m.q_offsets, m.q, m.d_offsets, m.d, allq, np.full(m.nq, di))
    check_argmax(g_arg[di:di + 1], np.concatenate(pa)[None, :], np.concatenate(pg)[None, :])
    sub = synth.MaxSimInputs(m.width, m.q_offsets, m.q_bf16, np.array([0, r1 - r0], np.uint64),
                             m.d_bf16[r0:r1], d_scores[:, di:di + 1])
    arg = routed_argmax(sub, g_arg[di:di + 1], np.concatenate(pa)[None, :], np.concatenate(pg)[None, :])
    _, ref = oracle.maxsim_backward(m.q_offsets, m.q, sub.d_offsets, sub.d, arg, sub.d_scores)
    return ref


def test_joint_step_config5():
    """Pooled N=16384, D=512 and MaxSim over 2048 x 2048 items (queries copied from their documents,
    sides 1/3 each), all enqueued on one stream.  The pooled L, dt, db and every dE row against the full
    oracle; the score-matrix loss's L, dt, db and its whole dS against the oracle on the GPU's score matrix;
    that score matrix on 2,000 sampled pairs; 16 queries' dQ and 16 documents' dD against the oracle's
    backward of the same dS."""
    j = synth.joint_config5()
    p, m = j.pooled, j.maxsim
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        e = bf16(p.e_bf16)
        q, qo, d, do = bf16(m.q_bf16), i64(m.q_offsets), bf16(m.d_bf16), i64(m.d_offsets)
        sides = torch.from_numpy(j.sides).to(dev())
        diag = cli.device_edges(j.score_attract)
        pr = cli.pair_loss_sigmoid_fwd_bwd(e, scalar(p.t), scalar(p.b), cli.device_edges(p.attract))
        f = cli.maxsim_scores(q, qo, d, do)
        sl = cli.pair_loss_sigmoid_scores_fwd_bwd(f["scores"], scalar(j.score_t), scalar(j.score_b), diag,
                                                  sides=sides)
        g = cli.maxsim_backward(q, qo, d, do, f["argmax"], sl["d_scores"])
    stream.synchronize()
    for r in (pr, f, sl, g):
        assert int(r["device_status"].item()) == 0
    # pooled part, every anchor
    ref = oracle.pair_loss_sigmoid(p.e_rounded, p.t, p.b, p.attract)
    compare_pooled(p, dict(loss=pr["loss"].item(), dt=pr["d_inverse_temperature"].item(),
                           db=pr["d_bias"].item(), de=pr["d_embeddings"].double().cpu().numpy(), status=0), ref)
    # MaxSim scores on sampled pairs, own-document pairs included
    S = f["scores"].double().cpu().numpy()
    rng = np.random.default_rng(2)
    pq, pd = rng.integers(0, m.nq, 2000), rng.integers(0, m.nd, 2000)
    pq[:64] = pd[:64]
    ps, pa, pg = oracle.maxsim_pairs(m.q_offsets, m.q, m.d_offsets, m.d, pq, pd)
    check_scores(S[pq, pd], ps)
    g_arg = f["argmax"].cpu().numpy()
    for k in range(len(pq)):
        t0, t1 = int(m.q_offsets[pq[k]]), int(m.q_offsets[pq[k] + 1])
        check_argmax(g_arg[pd[k], t0:t1], pa[k], pg[k])
    # score-matrix loss over the GPU's S: every output against the oracle
    sref = oracle.pair_loss_sigmoid_scores(S, j.score_t, j.score_b, j.score_attract, sides=j.sides)
    assert_rel(sl["loss"].item(), sref["loss"], LOSS_RTOL, "score loss")
    assert_rel(sl["d_inverse_temperature"].item(), sref["dt"], GRAD_RL2, "score loss dt")
    assert_rel(sl["d_bias"].item(), sref["db"], GRAD_RL2, "score loss db")
    dS = sl["d_scores"].double().cpu().numpy()
    assert rel_l2(dS, sref["dscores"]) <= GRAD_RL2
    # backward rows of 16 queries and 16 documents, from the same dS
    dq, dd = g["d_queries"].double().cpu().numpy(), g["d_documents"].double().cpu().numpy()
    active_q, active_d = np.nonzero(np.any(dS != 0, axis=1))[0], np.nonzero(np.any(dS != 0, axis=0))[0]
    for qi in rng.choice(active_q, 16, replace=False):
        t0, t1 = int(m.q_offsets[qi]), int(m.q_offsets[qi + 1])
        ref_q = maxsim_rows_of_query(m, g_arg, qi, dS)
        assert rel_l2(dq[t0:t1], ref_q) <= GRAD_RL2, f"query {qi}"
    for di in rng.choice(active_d, 16, replace=False):
        r0, r1 = int(m.d_offsets[di]), int(m.d_offsets[di + 1])
        ref_d = maxsim_rows_of_document(m, g_arg, di, dS)
        assert rel_l2(dd[r0:r1], ref_d) <= GRAD_RL2, f"document {di}"
