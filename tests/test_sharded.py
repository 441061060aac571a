"""The sharded pooled step's exchanges on CPU: two gloo ranks, each holding half of the batch's rows,
all-gather E, run a band call for their own anchors, reduce-scatter dE and all-reduce L, dt and db; the
result must be the whole batch's loss ("UForm", section "Matryoshka-Like Multi-Scale Embedders": one
SigLIP loss over the domain, the embeddings all-gathered into one similarity band, the gradients
reduce-scattered back).

No GPU here: the band call is the oracle's dense band formulation (the test injects it; the product path
calls the library's band verb), and the whole batch is checked against the C oracle.
"""

import os
import socket
import sys

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _inputs():
    from contrastive_late_interaction_gb300 import synth
    p = synth.pooled_bags(21, 96, 24, ignore_p=0.05)
    p.t, p.b = 6.0, -2.0
    return p


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import oracle
    from contrastive_late_interaction_gb300 import sharded, synth
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        p = _inputs()
        n = p.count // world
        e = torch.from_numpy(p.e_bf16.view(np.int16).copy()).view(torch.bfloat16)
        local = e[rank * n:(rank + 1) * n].clone()

        def band_call(e_all, begin, count):
            x = e_all.float().double().numpy()
            r = oracle.pair_loss_sigmoid_groups(x, np.zeros(p.count, np.int64), [p.t], [p.b], p.attract, None,
                                                p.ignore, band=(begin, count))
            f64 = dict(dtype=torch.float64)
            return dict(loss=torch.tensor([r["loss"]], **f64),
                        d_inverse_temperature=torch.tensor([r["dt"][0]], **f64),
                        d_bias=torch.tensor([r["db"][0]], **f64), d_embeddings=torch.from_numpy(r["de"]))

        r = sharded.pair_loss_sigmoid_sharded(local, None, None, None, band_call=band_call)
        out[rank] = (float(r["loss"]), float(r["d_inverse_temperature"]), float(r["d_bias"]),
                     r["d_embeddings"].numpy())
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_reproduce_the_whole_batch():
    sys.path.insert(0, ROOT)
    import oracle
    world, port = 2, _free_port()
    manager = mp.Manager()
    out = manager.dict()
    mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
    p = _inputs()
    ref = oracle.pair_loss_sigmoid(p.e_rounded, p.t, p.b, p.attract, ignore=p.ignore)
    de = np.concatenate([out[r][3] for r in range(world)], axis=0)
    for r in range(world):
        loss, dt, db, _ = out[r]
        assert abs(loss - ref["loss"]) <= 1e-12 * abs(ref["loss"])
        assert abs(dt - ref["dt"]) <= 1e-10 * max(abs(ref["dt"]), 1e-30)
        assert abs(db - ref["db"]) <= 1e-10 * max(abs(ref["db"]), 1e-30)
    assert np.max(np.abs(de - ref["de"])) <= 1e-12 * np.max(np.abs(ref["de"]))
