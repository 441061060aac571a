"""The sharded pooled step on one GPU: two processes (gloo ranks), each holding half of the batch's rows on
cuda:0, all-gather E through host memory, run the library's anchor-band call for their own anchors,
reduce-scatter dE and all-reduce L, dt and db; together they must reproduce the whole call, checked
against the float64 oracle ("UForm", section "Matryoshka-Like Multi-Scale Embedders": the embeddings
all-gathered into one similarity band, the gradients reduce-scattered back).  The two ranks' kernels never
wait on each other: every exchange is a host-side gloo collective between whole calls.
"""

import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _inputs(case):
    from contrastive_late_interaction_gb300 import synth
    if case == "ragged":
        p = synth.pooled_bags(22, 1000, 200, ignore_p=0.02)
        p.t, p.b = 7.0, -3.0
        return p
    return synth.pooled_config2()


def _worker(rank, world, port, case, out):
    sys.path.insert(0, ROOT)
    import contrastive_late_interaction_gb300 as cli
    from contrastive_late_interaction_gb300 import sharded
    torch.cuda.set_device(0)
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        p = _inputs(case)
        n = p.count // world
        dev = torch.device("cuda:0")
        e = torch.from_numpy(p.e_bf16.view(np.int16).copy()).view(torch.bfloat16)
        local = e[rank * n:(rank + 1) * n].to(dev)
        t = torch.tensor([p.t], dtype=torch.float32, device=dev)
        b = torch.tensor([p.b], dtype=torch.float32, device=dev)
        r = sharded.pair_loss_sigmoid_sharded(local, t, b, cli.device_edges(p.attract, dev),
                                              ignore=cli.device_edges(p.ignore if p.ignore.ids.size else None, dev))
        torch.cuda.synchronize()
        out[rank] = (float(r["loss"]), float(r["d_inverse_temperature"]), float(r["d_bias"]),
                     r["d_embeddings"].double().cpu().numpy())
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("case", ["ragged", "config2"])
def test_two_ranks_on_one_gpu_reproduce_the_whole_call(case):
    sys.path.insert(0, ROOT)
    import oracle
    from tests.gpu_util import GRAD_RL2, LOSS_RTOL, assert_rel, rel_l2
    world, port = 2, _free_port()
    manager = mp.get_context("spawn").Manager()
    out = manager.dict()
    mp.spawn(_worker, args=(world, port, case, out), nprocs=world, join=True)
    p = _inputs(case)
    ref = oracle.pair_loss_sigmoid(p.e_rounded, p.t, p.b, p.attract,
                                   ignore=p.ignore if p.ignore.ids.size else None)
    for r in range(world):
        loss, dt, db, _ = out[r]
        assert_rel(loss, ref["loss"], LOSS_RTOL, "loss")
        assert_rel(dt, ref["dt"], GRAD_RL2, "dt")
        assert_rel(db, ref["db"], GRAD_RL2, "db")
    de = np.concatenate([out[r][3] for r in range(world)], axis=0)
    assert rel_l2(de, ref["de"]) <= GRAD_RL2
