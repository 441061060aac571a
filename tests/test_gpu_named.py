"""GPU parity of maxsim_scores_named against the float64 oracle.

Named pairs ("Training", `uform_late_interaction_side_t`: a query's tokens score the documents it attracts
and repels): S(q, d) and the argmax of every named pair equal the oracle's; a pair no query names scores 0
and its argmax entries stay valid rows of the document, so the backward runs on the same outputs.
"""

import numpy as np
import pytest
import torch

import oracle
from contrastive_late_interaction_gb300 import synth
from tests.gpu_util import GRAD_RL2, bf16, check_argmax, check_scores, dev, i64, rel_l2, routed_argmax

pytestmark = pytest.mark.gpu


def named_lists(seed, nq, nd, k_lo, k_hi, own=False):
    rng = np.random.default_rng(seed)
    lists = []
    for q in range(nq):
        k = int(rng.integers(k_lo, k_hi + 1))
        docs = set(rng.choice(nd, size=min(k, nd), replace=False).tolist())
        if own:
            docs.add(q % nd)
        lists.append(sorted(docs))
    return lists


def row_mask(m, named):
    """[documents, query rows] view of a [queries, documents] pair mask."""
    q_of_row = np.repeat(np.arange(m.nq), np.diff(m.q_offsets.astype(np.int64)))
    return named[q_of_row].T


def run_named(m, lists):
    import contrastive_late_interaction_gb300 as cli
    pairs = cli.device_edges(synth.edges_from_lists(lists))
    r = cli.maxsim_scores_named(bf16(m.q_bf16), i64(m.q_offsets), bf16(m.d_bf16), i64(m.d_offsets), pairs)
    torch.cuda.synchronize()
    return r


def check_named(m, lists, r, full=True):
    assert int(r["device_status"].item()) == 0
    s = r["scores"].double().cpu().numpy()
    am = r["argmax"].cpu().numpy()
    named = np.zeros((m.nq, m.nd), bool)
    for q, docs in enumerate(lists):
        named[q, docs] = True
    assert np.all(s[~named] == 0.0), "a pair no query names has a score"
    dl = np.diff(m.d_offsets).astype(np.int64)
    assert np.all(am >= 0) and np.all(am < dl[:, None]), "an argmax entry outside its document"
    pq, pd = np.nonzero(named)
    ref_s, ref_arg, ref_gap = oracle.maxsim_pairs(m.q_offsets, m.q, m.d_offsets, m.d, pq, pd)
    check_scores(s[pq, pd], ref_s)
    for k in range(len(pq)):
        t0, t1 = int(m.q_offsets[pq[k]]), int(m.q_offsets[pq[k] + 1])
        check_argmax(am[pd[k], t0:t1], ref_arg[k], ref_gap[k])
    return named


def test_named_ragged():
    m = synth.maxsim_random(21, 60, 90, 128, (4, 140), (1, 300))
    lists = named_lists(1, m.nq, m.nd, 0, 6)
    check_named(m, lists, run_named(m, lists))


def test_named_backward_matches_the_oracle():
    """dS zero off the named pairs (as a named-negatives loss gives): dQ and dD equal the oracle's."""
    import contrastive_late_interaction_gb300 as cli
    m = synth.maxsim_random(22, 40, 50, 72, (3, 60), (5, 150))
    lists = named_lists(2, m.nq, m.nd, 1, 5)
    r = run_named(m, lists)
    named = check_named(m, lists, r)
    ds = np.where(named, m.d_scores, 0.0).astype(np.float32)
    g = cli.maxsim_backward(bf16(m.q_bf16), i64(m.q_offsets), bf16(m.d_bf16), i64(m.d_offsets), r["argmax"],
                            torch.from_numpy(ds).to(dev()))
    torch.cuda.synchronize()
    assert int(g["device_status"].item()) == 0
    _, arg, gap = oracle.maxsim_forward(m.q_offsets, m.q, m.d_offsets, m.d)
    arg = routed_argmax(m, r["argmax"].cpu().numpy(), arg, gap, where=row_mask(m, named))
    dq, dd = oracle.maxsim_backward(m.q_offsets, m.q, m.d_offsets, m.d, arg, ds.astype(np.float64))
    assert rel_l2(g["d_queries"].double().cpu().numpy(), dq) <= GRAD_RL2
    assert rel_l2(g["d_documents"].double().cpu().numpy(), dd) <= GRAD_RL2


def test_named_config5_own_document_and_seven_others():
    """The joint config's MaxSim tapes (2048 x 2048), each query naming its own document and seven others."""
    m = synth.joint_config5().maxsim
    lists = named_lists(3, m.nq, m.nd, 7, 7, own=True)
    check_named(m, lists, run_named(m, lists))


def test_no_pairs_scores_nothing():
    m = synth.maxsim_random(23, 10, 12, 64, (2, 20), (3, 30))
    r = run_named(m, [[] for _ in range(m.nq)])
    assert int(r["device_status"].item()) == 0
    assert torch.all(r["scores"] == 0) and torch.all(r["argmax"] == 0)


def test_a_pair_past_the_documents_is_malformed():
    import contrastive_late_interaction_gb300 as cli
    m = synth.maxsim_random(24, 10, 12, 64, (2, 20), (3, 30))
    lists = [[0, 3]] * m.nq
    lists[4] = [1, 12]
    r = run_named(m, lists)
    assert cli.status_name(int(r["device_status"].item())) == "malformed"


@pytest.mark.parametrize("mean", [False, True])
def test_named_backward_ignores_pairs_not_named(mean):
    """maxsim_backward_named with a dS that is nonzero everywhere: only the named pairs reach dQ and dD."""
    import contrastive_late_interaction_gb300 as cli
    m = synth.maxsim_random(25, 50, 70, 128, (2, 70), (3, 260))
    lists = named_lists(4, m.nq, m.nd, 1, 6)
    pairs = cli.device_edges(synth.edges_from_lists(lists))
    f = cli.maxsim_scores_named(bf16(m.q_bf16), i64(m.q_offsets), bf16(m.d_bf16), i64(m.d_offsets), pairs, mean=mean)
    g = cli.maxsim_backward_named(bf16(m.q_bf16), i64(m.q_offsets), bf16(m.d_bf16), i64(m.d_offsets), f["argmax"],
                                  torch.from_numpy(np.ascontiguousarray(m.d_scores)).to(dev()), pairs, mean=mean)
    torch.cuda.synchronize()
    assert int(f["device_status"].item()) == 0 and int(g["device_status"].item()) == 0
    named = np.zeros((m.nq, m.nd), bool)
    for q, docs in enumerate(lists):
        named[q, docs] = True
    _, arg, gap = oracle.maxsim_forward(m.q_offsets, m.q, m.d_offsets, m.d)
    arg = routed_argmax(m, f["argmax"].cpu().numpy(), arg, gap, where=row_mask(m, named))
    ds = np.where(named, m.d_scores, 0.0)
    dq, dd = oracle.maxsim_backward(m.q_offsets, m.q, m.d_offsets, m.d, arg, ds, mean)
    assert rel_l2(g["d_queries"].double().cpu().numpy(), dq) <= GRAD_RL2
    assert rel_l2(g["d_documents"].double().cpu().numpy(), dd) <= GRAD_RL2
