"""GPU parity of pair_loss_sigmoid_groups_fwd_bwd against the float64 oracle.

Temperature groups ("Training", `uform_contrastive_t`, `temperature_groups`): item i selects a group and a
cell takes its anchor's (inverse temperature, bias).
"""

import numpy as np
import pytest
import torch

import oracle
from contrastive_late_interaction_gb300 import synth
from tests.gpu_util import GRAD_RL2, LOSS_RTOL, assert_rel, bf16, dev, rel_l2, scalar

pytestmark = pytest.mark.gpu


def run(p, groups, t, b, ld=None, ld_de=None):
    import contrastive_late_interaction_gb300 as cli
    e_bits = p.e_bf16
    if ld is not None and ld > p.width:
        e_bits = np.zeros((p.count, ld), dtype=np.uint16)
        e_bits[:, :p.width] = p.e_bf16
    out = {"width": p.width}
    if ld_de is not None:
        out["d_embeddings"] = torch.full((p.count, ld_de), 7.0, device=dev())[:, :p.width]
    r = cli.pair_loss_sigmoid_groups_fwd_bwd(
        bf16(e_bits), torch.from_numpy(np.asarray(groups, np.int32)).to(dev()),
        torch.tensor(np.asarray(t, np.float32), device=dev()), torch.tensor(np.asarray(b, np.float32), device=dev()),
        cli.device_edges(p.attract), cli.device_edges(p.repel if p.repel.ids.size else None),
        cli.device_edges(p.ignore if p.ignore.ids.size else None), negatives_named=p.negatives_named,
        ambient_weight=p.ambient_weight, out=out)
    torch.cuda.synchronize()
    return r


def compare(p, groups, t, b, r):
    ref = oracle.pair_loss_sigmoid_groups(p.e_rounded, groups, t, b, p.attract, p.repel if p.repel.ids.size else None,
                                          p.ignore if p.ignore.ids.size else None, p.negatives_named, p.ambient_weight)
    assert int(r["device_status"].item()) == 0
    assert_rel(r["loss"].item(), ref["loss"], LOSS_RTOL, "loss")
    dt, db = r["d_inverse_temperature"].double().cpu().numpy(), r["d_bias"].double().cpu().numpy()
    assert rel_l2(dt, ref["dt"]) <= GRAD_RL2, (dt, ref["dt"])
    assert rel_l2(db, ref["db"]) <= GRAD_RL2, (db, ref["db"])
    e = rel_l2(r["d_embeddings"].double().cpu().numpy(), ref["de"])
    assert e <= GRAD_RL2, f"dE rel L2 {e:.3e}"
    return ref


def test_groups_tiny():
    """N=256, D=64, bags of two; three groups of different pairs."""
    p = synth.pooled_tiny()
    groups = np.random.default_rng(1).integers(0, 3, size=p.count)
    t, b = [10.0, 5.0, 15.0], [-10.0, -5.0, -12.0]
    compare(p, groups, t, b, run(p, groups, t, b))


def test_groups_ragged_weighted_named():
    """N and D off the tile grid, weighted edges, ignores, named negatives, padded strides, one group that
    no item selects (its gradients are zero)."""
    rng = np.random.default_rng(12)
    n, width = 300, 72
    p = synth.pooled_bags(4, n, width, ignore_p=0.02)
    p.attract.weights = rng.uniform(0.2, 2.0, size=p.attract.ids.size).astype(np.float32)
    rep_lists = [sorted(set(rng.choice(n, size=5, replace=False).tolist()) - {i}) for i in range(n)]
    p.repel = synth.edges_from_lists(rep_lists)
    p.repel.weights = rng.uniform(0.1, 3.0, size=p.repel.ids.size).astype(np.float32)
    p.negatives_named = True
    groups = rng.integers(0, 3, size=n)
    t, b = [7.0, 2.0, -3.0, 9.0], [-3.0, 0.5, 1.0, 4.0]
    r = run(p, groups, t, b, ld=width + 8, ld_de=width + 4)
    compare(p, groups, t, b, r)
    assert r["d_inverse_temperature"][3].item() == 0.0 and r["d_bias"][3].item() == 0.0
    pad = r["d_embeddings"].as_strided((n, 4), (width + 4, 1), width)
    assert torch.all(pad == 7.0), "columns past the width were written"


def test_one_group_is_the_pooled_call():
    import contrastive_late_interaction_gb300 as cli
    p = synth.pooled_bags(6, 500, 128, ignore_p=0.01)
    r = run(p, np.zeros(p.count, int), [p.t], [p.b])
    q = cli.pair_loss_sigmoid_fwd_bwd(bf16(p.e_bf16), scalar(p.t), scalar(p.b), cli.device_edges(p.attract), None,
                                      cli.device_edges(p.ignore))
    torch.cuda.synchronize()
    assert r["loss"].item() == q["loss"].item()
    assert torch.equal(r["d_embeddings"], q["d_embeddings"])


def test_groups_config2():
    """N=4096, D=512 (bags U{1..4}, 1% ignored pairs) with two groups."""
    p = synth.pooled_config2()
    groups = np.random.default_rng(3).integers(0, 2, size=p.count)
    t, b = [10.0, 6.0], [-10.0, -7.0]
    compare(p, groups, t, b, run(p, groups, t, b))


def test_a_group_out_of_range_is_malformed():
    import contrastive_late_interaction_gb300 as cli
    p = synth.pooled_tiny()
    groups = np.zeros(p.count, int)
    groups[17] = 2
    r = run(p, groups, [10.0, 5.0], [-10.0, -5.0])
    st = int(r["device_status"].item())
    assert cli.status_name(st) == "malformed", cli.status_name(st)
