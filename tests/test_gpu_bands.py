"""Anchor bands of the pooled loss on the GPU, against the float64 oracle.

A band is one device's rows when the loss is sharded across devices ("UForm", section "Matryoshka-Like
Multi-Scale Embedders": the per-rank embeddings all-gathered into one similarity band, the gradients
reduce-scattered back), read as each rank scoring its own items' rows against every gathered column.
Run on one GPU: each band's results are the oracle's band shares, and bands that partition the rows add
up to the whole call.
"""

import numpy as np
import pytest
import torch

import oracle
from contrastive_late_interaction_gb300 import synth
from tests.gpu_util import GRAD_RL2, LOSS_RTOL, assert_rel, bf16, dev, rel_l2, scalar

pytestmark = pytest.mark.gpu

# A band sum and the whole call round H to bf16 at different points (each direction of a cell apart,
# or both together), so they agree to that rounding, not bit for bit.
SUM_RTOL, SUM_RL2 = 1e-4, 5e-3


def weighted_case(n, width, seed):
    rng = np.random.default_rng(seed)
    p = synth.pooled_bags(seed, n, width, ignore_p=0.02)
    p.attract.weights = rng.uniform(0.2, 2.0, size=p.attract.ids.size).astype(np.float32)
    rep = synth.edges_from_lists([sorted(set(rng.choice(n, size=3, replace=False).tolist()) - {i})
                                  for i in range(n)])
    rep.weights = rng.uniform(0.1, 3.0, size=rep.ids.size).astype(np.float32)
    p.repel = rep
    p.ambient_weight = 0.75
    p.t, p.b = 7.0, -3.0
    return p


def edges(p):
    import contrastive_late_interaction_gb300 as cli
    return (cli.device_edges(p.attract), cli.device_edges(p.repel if p.repel.ids.size else None),
            cli.device_edges(p.ignore if p.ignore.ids.size else None))


def run(p, band=None, groups=None, prefixes=None):
    import contrastive_late_interaction_gb300 as cli
    e = bf16(p.e_bf16)
    kw = dict(negatives_named=p.negatives_named, ambient_weight=p.ambient_weight, band=band)
    if groups is not None:
        g, t, b = groups
        r = cli.pair_loss_sigmoid_groups_fwd_bwd(
            e, torch.from_numpy(np.asarray(g, np.int32)).to(dev()), torch.tensor(np.asarray(t, np.float32),
                                                                                   device=dev()),
            torch.tensor(np.asarray(b, np.float32), device=dev()), *edges(p), **kw)
    elif prefixes is not None:
        r = cli.pair_loss_sigmoid_matryoshka_fwd_bwd(e, prefixes, scalar(p.t), scalar(p.b), *edges(p), **kw)
    else:
        r = cli.pair_loss_sigmoid_fwd_bwd(e, scalar(p.t), scalar(p.b), *edges(p), **kw)
    torch.cuda.synchronize()
    assert int(r["device_status"].item()) == 0
    return dict(loss=float(r["loss"].item()), dt=r["d_inverse_temperature"].double().cpu().numpy(),
                db=r["d_bias"].double().cpu().numpy(), de=r["d_embeddings"].double().cpu().numpy())


def oracle_band(p, band, groups=None):
    g, t, b = groups if groups is not None else (np.zeros(p.count, int), [p.t], [p.b])
    return oracle.pair_loss_sigmoid_groups(p.e_rounded, g, t, b, p.attract, p.repel if p.repel.ids.size else None,
                                           p.ignore if p.ignore.ids.size else None, p.negatives_named,
                                           p.ambient_weight, band=band)


def compare(gpu, ref):
    assert_rel(gpu["loss"], ref["loss"], LOSS_RTOL, "loss")
    assert rel_l2(gpu["dt"], ref["dt"]) <= GRAD_RL2, (gpu["dt"], ref["dt"])
    assert rel_l2(gpu["db"], ref["db"]) <= GRAD_RL2, (gpu["db"], ref["db"])
    e = rel_l2(gpu["de"], ref["de"])
    assert e <= GRAD_RL2, f"dE rel L2 {e:.3e}"


def check_sum(parts, full):
    assert_rel(sum(x["loss"] for x in parts), full["loss"], SUM_RTOL, "loss of the bands")
    assert rel_l2(sum(x["dt"] for x in parts), full["dt"]) <= SUM_RTOL
    assert rel_l2(sum(x["db"] for x in parts), full["db"]) <= SUM_RTOL
    e = rel_l2(sum(x["de"] for x in parts), full["de"])
    assert e <= SUM_RL2, f"dE of the bands, rel L2 {e:.3e}"


BANDS_1000 = [(0, 77), (77, 300), (377, 622), (999, 1)]   # off the 256-row block grid; a one-row band


def test_bands_match_the_oracle_and_add_up():
    p = weighted_case(1000, 200, 5)
    parts = []
    for band in BANDS_1000:
        g = run(p, band)
        compare(g, oracle_band(p, band))
        parts.append(g)
    check_sum(parts, run(p))


def test_band_inside_one_tile_named_negatives():
    p = weighted_case(300, 72, 6)
    p.negatives_named = True
    for band in ((130, 20), (0, 1)):
        compare(run(p, band), oracle_band(p, band))


def test_whole_batch_band_is_the_plain_call():
    p = weighted_case(500, 64, 7)
    a, b = run(p), run(p, (0, 500))
    assert a["loss"] == b["loss"] and np.array_equal(a["dt"], b["dt"]) and np.array_equal(a["db"], b["db"])
    assert rel_l2(b["de"], a["de"]) <= 1e-6


def test_groups_bands_match_the_oracle_and_add_up():
    p = weighted_case(700, 128, 8)
    rng = np.random.default_rng(8)
    groups = (rng.integers(0, 3, size=p.count), [7.0, 3.0, 11.0], [-3.0, -1.0, -6.0])
    parts = []
    for band in ((0, 256), (256, 100), (356, 344)):
        g = run(p, band, groups=groups)
        compare(g, oracle_band(p, band, groups))
        parts.append(g)
    check_sum(parts, run(p, groups=groups))


def test_matryoshka_bands_add_up():
    p = weighted_case(600, 256, 9)
    prefixes = [64, 128, 256]
    full = run(p, prefixes=prefixes)
    parts = [run(p, band, prefixes=prefixes) for band in ((0, 300), (300, 299), (599, 1))]
    check_sum(parts, full)


def test_config2_bands():
    """N = 4096, D = 512 with 1% ignores: each band's L, dt, db against the C oracle's shares of its anchor
    rows, and the bands against the whole call."""
    p = synth.pooled_config2()
    parts = []
    for band in ((0, 1024), (1024, 1500), (2524, 1572)):
        g = run(p, band)
        rows = np.arange(band[0], band[0] + band[1])
        ref = oracle.pair_loss_sigmoid(p.e_rounded, p.t, p.b, p.attract, None, p.ignore, p.negatives_named,
                                       p.ambient_weight, rows=rows, want_de=False)
        assert_rel(g["loss"], ref["loss"], LOSS_RTOL, "loss")
        assert_rel(g["dt"][0], ref["dt"], GRAD_RL2, "dt")
        assert_rel(g["db"][0], ref["db"], GRAD_RL2, "db")
        parts.append(g)
    check_sum(parts, run(p))


# ---------------------------------------------------------------------------
# MaxSim sharded by queries: each device scores its queries against every (gathered) document, keeps its
# dQ rows and reduce-scatters dD.  On one GPU a query band is a sub-tape with offsets rebased to zero.
# ---------------------------------------------------------------------------

def query_band(m, q0, q1):
    r0, r1 = int(m.q_offsets[q0]), int(m.q_offsets[q1])
    return synth.MaxSimInputs(m.width, (m.q_offsets[q0:q1 + 1] - m.q_offsets[q0]).astype(np.uint64),
                              m.q_bf16[r0:r1], m.d_offsets, m.d_bf16, np.ascontiguousarray(m.d_scores[q0:q1]))


@pytest.mark.parametrize("mean", [False, True])
def test_maxsim_query_bands_add_up(mean):
    from tests.gpu_util import run_maxsim
    m = synth.maxsim_random(12, 40, 30, 128, (1, 70), (1, 300))
    full = run_maxsim(m, mean=mean)
    assert full["status_f"] == 0 and full["status_b"] == 0
    dd = np.zeros_like(full["dd"])
    for q0, q1 in ((0, 13), (13, 29), (29, 40)):
        part = run_maxsim(query_band(m, q0, q1), mean=mean)
        assert part["status_f"] == 0 and part["status_b"] == 0
        r0, r1 = int(m.q_offsets[q0]), int(m.q_offsets[q1])
        # a row's scores, maxima and argmax do not depend on the other rows of the call
        assert np.array_equal(part["scores"], full["scores"][q0:q1])
        assert np.array_equal(part["argmax"][:, :r1 - r0], full["argmax"][:, r0:r1])
        assert rel_l2(part["dq"], full["dq"][r0:r1]) <= 1e-6
        dd += part["dd"]
    assert rel_l2(dd, full["dd"]) <= 1e-5
