"""GPU parity of pair_loss_sigmoid_matryoshka_fwd_bwd against the float64 oracle.

Matryoshka prefixes under the sigmoid pair loss ("Training", `uform_contrastive_t`,
`matryoshka_dimensions`; "UForm", section "Matryoshka-Like Multi-Scale Embedders"): each listed prefix is
normalised, scored under the SigLIP loss and its gradient sent back through the normalisation.
"""

import numpy as np
import pytest
import torch

import oracle
from contrastive_late_interaction_gb300 import synth
from tests.gpu_util import GRAD_RL2, LOSS_RTOL, assert_rel, bf16, dev, rel_l2, scalar

pytestmark = pytest.mark.gpu


def run(p, prefixes, ld=None, ld_de=None):
    import contrastive_late_interaction_gb300 as cli
    e_bits = p.e_bf16
    if ld is not None and ld > p.width:
        e_bits = np.zeros((p.count, ld), dtype=np.uint16)
        e_bits[:, :p.width] = p.e_bf16
    out = {"width": p.width}
    if ld_de is not None:
        out["d_embeddings"] = torch.full((p.count, ld_de), 7.0, device=dev())[:, :p.width]
    r = cli.pair_loss_sigmoid_matryoshka_fwd_bwd(
        bf16(e_bits), prefixes, scalar(p.t), scalar(p.b), cli.device_edges(p.attract),
        cli.device_edges(p.repel if p.repel.ids.size else None), cli.device_edges(p.ignore if p.ignore.ids.size else None),
        negatives_named=p.negatives_named, ambient_weight=p.ambient_weight, out=out)
    torch.cuda.synchronize()
    return r


def compare(p, prefixes, r):
    ref = oracle.pair_loss_sigmoid_matryoshka(p.e_rounded, prefixes, p.t, p.b, p.attract,
                                              p.repel if p.repel.ids.size else None,
                                              p.ignore if p.ignore.ids.size else None, p.negatives_named,
                                              p.ambient_weight)
    assert int(r["device_status"].item()) == 0
    assert_rel(r["loss"].item(), ref["loss"], LOSS_RTOL, "loss")
    assert_rel(r["d_inverse_temperature"].item(), ref["dt"], GRAD_RL2, "dt")
    assert_rel(r["d_bias"].item(), ref["db"], GRAD_RL2, "db")
    e = rel_l2(r["d_embeddings"].double().cpu().numpy(), ref["de"])
    assert e <= GRAD_RL2, f"dE rel L2 {e:.3e}"
    pl = r["prefix_loss"].double().cpu().numpy()
    for k, per in enumerate(ref["per_prefix"]):
        assert_rel(pl[k], per["loss"], LOSS_RTOL, f"loss of prefix {per['width']}")


def test_matryoshka_tiny():
    """N=256, D=64, bags of two, t=10, b=-10; three prefixes, the full width last."""
    p = synth.pooled_tiny()
    prefixes = [16, 32, 64]
    compare(p, prefixes, run(p, prefixes))


def test_matryoshka_ragged_weighted():
    """N and widths off the tile grid, weighted attract and repel edges, ignores, padded strides; the full
    width is not scored, so dE past the last prefix is zero."""
    rng = np.random.default_rng(11)
    n, width = 300, 72
    p = synth.pooled_bags(9, n, width, ignore_p=0.02)
    p.attract.weights = rng.uniform(0.2, 2.0, size=p.attract.ids.size).astype(np.float32)
    rep_lists = [sorted(set(rng.choice(n, size=3, replace=False).tolist()) - {i}) for i in range(n)]
    p.repel = synth.edges_from_lists(rep_lists)
    p.repel.weights = rng.uniform(0.1, 3.0, size=p.repel.ids.size).astype(np.float32)
    p.ambient_weight = 0.75
    p.t, p.b = 7.0, -3.0
    prefixes = [8, 40, 64]
    r = run(p, prefixes, ld=width + 8, ld_de=width + 4)
    compare(p, prefixes, r)
    assert torch.all(r["d_embeddings"][:, 64:] == 0)
    pad = r["d_embeddings"].as_strided((n, 4), (width + 4, 1), width)
    assert torch.all(pad == 7.0), "columns past the width were written"


def test_matryoshka_config2_prefixes():
    """N=4096, D=512 (bags U{1..4}, 1% ignored pairs) with the prefixes {64, 128, 256, 512}."""
    p = synth.pooled_config2()
    prefixes = [64, 128, 256, 512]
    compare(p, prefixes, run(p, prefixes))
