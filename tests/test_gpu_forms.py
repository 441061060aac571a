"""The balanced and ranked pair-loss forms over a score matrix: CUDA path (C ABI) against the oracle."""

import numpy as np
import pytest
import torch

import oracle
from contrastive_late_interaction_gb300 import synth

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

if torch.cuda.is_available():
    import contrastive_late_interaction_gb300 as cli
    from tests.gpu_util import GRAD_RL2, LOSS_RTOL, assert_rel, rel_l2, scalar


def _run(form, s, t, b, att, rep=None, ign=None, sides=None, named=False, ambient=1.0):
    S = torch.from_numpy(np.ascontiguousarray(s, dtype=np.float32)).cuda()
    r = cli.pair_loss_scores_fwd_bwd(form, S, scalar(t), scalar(b), cli.device_edges(att),
                                     cli.device_edges(rep), cli.device_edges(ign),
                                     sides=None if sides is None else torch.from_numpy(sides).cuda(),
                                     negatives_named=named, ambient_weight=ambient)
    torch.cuda.synchronize()
    assert int(r["device_status"].item()) == 0
    return r


def _compare(form, r, ref):
    assert_rel(r["loss"].item(), ref["loss"], LOSS_RTOL, f"{form} loss")
    assert_rel(r["d_inverse_temperature"].item(), ref["dt"], GRAD_RL2, f"{form} dt")
    if form == "balanced":
        assert_rel(r["d_bias"].item(), ref["db"], GRAD_RL2, f"{form} db")
    else:
        assert r["d_bias"].item() == 0.0
    e = rel_l2(r["d_scores"].double().cpu().numpy(), ref["dscores"])
    assert e <= GRAD_RL2, f"{form} dS rel L2 {e:.3e}"


@pytest.mark.parametrize("form", ["balanced", "ranked"])
@pytest.mark.parametrize("with_sides", [False, True])
def test_forms_small_weighted(form, with_sides):
    rng = np.random.default_rng(11 + with_sides)
    n = 300
    s = rng.normal(scale=2.0, size=(n, n)).astype(np.float32)
    lists = [sorted({i} | set(rng.choice(n, size=int(rng.integers(0, 20)), replace=False).tolist())) for i in range(n)]
    att = synth.edges_from_lists(lists)
    att.weights = rng.uniform(0.3, 2.0, size=att.ids.size).astype(np.float32)
    rep = synth.edges_from_lists([sorted(set(rng.choice(n, size=5, replace=False).tolist()) - set(lists[i]))
                                  for i in range(n)])
    rep.weights = rng.uniform(0.3, 2.0, size=rep.ids.size).astype(np.float32)
    ign = synth.ignore_bernoulli(9, n, 0.03)
    sides = rng.integers(1, 4, size=n).astype(np.uint8) if with_sides else None
    r = _run(form, s, 2.0, -0.5, att, rep, ign, sides, ambient=0.7)
    ref = oracle.pair_loss_scores_form(form, s.astype(np.float64), 2.0, -0.5, att, rep, ign, sides, False, 0.7)
    _compare(form, r, ref)


@pytest.mark.parametrize("form", ["balanced", "ranked"])
def test_forms_joint_shape(form):
    """2048 x 2048 with attract (i, i), ambient negatives and sides 1/3 each (the joint step's shape)."""
    j = synth.joint(0, pooled_count=256, pooled_width=64, items=2048, d_len=(64, 65), q_len=(16, 17))
    s = np.random.default_rng(3).normal(scale=5.0, size=(2048, 2048)).astype(np.float32)
    r = _run(form, s, 1.0, 0.0, j.score_attract, sides=j.sides)
    ref = oracle.pair_loss_scores_form(form, s.astype(np.float64), 1.0, 0.0, j.score_attract, sides=j.sides)
    _compare(form, r, ref)


def test_sigmoid_form_through_the_form_verb_matches_the_sigmoid_verb():
    rng = np.random.default_rng(5)
    n = 128
    s = rng.normal(size=(n, n)).astype(np.float32)
    att = synth.diagonal_edges(n)
    a = _run("sigmoid", s, 1.5, 0.25, att)
    S = torch.from_numpy(s).cuda()
    b = cli.pair_loss_sigmoid_scores_fwd_bwd(S, scalar(1.5), scalar(0.25), cli.device_edges(att))
    torch.cuda.synchronize()
    assert a["loss"].item() == b["loss"].item()
    assert torch.equal(a["d_scores"], b["d_scores"])
