"""Exact ties in the MaxSim forward: the argmax is the lowest document row for every sign of the maximum.

Hard MaxSim ("UForm", section "ColBERT-Style Late-Interaction Rerankers") keeps each query token's single
best document row; among equal scores that row is the lowest one.  The inputs repeat one row of each
document at several positions (every row, in some documents), so every maximum is an exact tie between
bit-identical rows: positive maxima, negative maxima (every score below zero) and zero maxima (the
repeated row orthogonal to every query row).  Document lengths mix runs shorter than a 32-column chunk
(several boundaries per chunk), runs that end inside a chunk, and runs over several 128-row tiles; the
repeated rows fall inside one chunk, across chunks and across tiles, and adjacent documents share their
repeated row.
"""

import numpy as np
import pytest
import torch

import oracle
from contrastive_late_interaction_gb300 import synth

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

if torch.cuda.is_available():
    from tests.gpu_util import GRAD_RL2, check_scores, rel_l2, run_maxsim


@pytest.mark.parametrize("regime", ["positive", "negative", "zero"])
@pytest.mark.parametrize("d_len", [(1, 40), (1, 300)])
@pytest.mark.parametrize("mean", [False, True])
def test_maxsim_exact_ties_take_the_lowest_row(regime, d_len, mean):
    m = synth.maxsim_ties(11, regime, d_len=d_len)
    g = run_maxsim(m, mean=mean)
    assert g["status_f"] == 0 and g["status_b"] == 0
    s, arg, gap = oracle.maxsim_forward(m.q_offsets, m.q, m.d_offsets, m.d, mean)
    check_scores(g["scores"], s)
    tied = gap == 0
    assert np.count_nonzero(tied) > 0.8 * gap.size
    assert np.count_nonzero(arg[tied] > 0) > 0.3 * np.count_nonzero(tied)   # the lowest row is not always row 0
    wrong = np.nonzero(g["argmax"] != arg)
    assert wrong[0].size == 0, (f"{wrong[0].size} argmax entries differ, e.g. document {wrong[0][0]} row "
                                f"{wrong[1][0]}: gpu {g['argmax'][wrong[0][0], wrong[1][0]]} "
                                f"oracle {arg[wrong[0][0], wrong[1][0]]}")
    if regime == "negative":
        assert np.all(s < 0)
    if regime == "zero":
        assert np.all(g["scores"] == 0.0)
    dq, dd = oracle.maxsim_backward(m.q_offsets, m.q, m.d_offsets, m.d, arg, m.d_scores, mean)
    assert rel_l2(g["dq"], dq) <= GRAD_RL2
    assert rel_l2(g["dd"], dd) <= GRAD_RL2


def test_maxsim_fixup_list_overflow_scans_every_maximum():
    """More rows with a non-positive maximum than the fix-up list holds (2^18 entries): the fix-up scans
    every maximum instead, and every argmax is still the oracle's (the lowest row)."""
    m = synth.maxsim_ties(12, "negative", nq=160, nd=60, q_len=(20, 50), d_len=(1, 40))
    entries = int(m.q_offsets[-1]) * m.nd
    assert entries > (1 << 18)
    g = run_maxsim(m)
    assert g["status_f"] == 0 and g["status_b"] == 0
    s, arg, gap = oracle.maxsim_forward(m.q_offsets, m.q, m.d_offsets, m.d)
    check_scores(g["scores"], s)
    assert np.all(s < 0)
    wrong = np.count_nonzero(g["argmax"] != arg)
    assert wrong == 0, f"{wrong} of {arg.size} argmax entries differ"
