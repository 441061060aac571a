"""The pooled sigmoid pair loss sharded by anchor rows across the ranks of a torch.distributed group.

"UForm", section "Matryoshka-Like Multi-Scale Embedders": one SigLIP loss spans every device of the
NVLink domain; each rank's embeddings are all-gathered into one similarity band and the gradients are
reduce-scattered back (the collectives are those of section "NVLink-Based Cross-GPU Collaboration").
Read as: rank r owns the items [r n, (r + 1) n) of a batch of N = R n and scores those rows (its
anchors) against every gathered column.  One step is

    1. all-gather E (bf16, N x D) from the ranks' [n x D] shares;
    2. the anchor-band call of `pair_loss_sigmoid_fwd_bwd` with (row_begin, row_count) = (r n, n): that
       band's shares of L, dt, db and of dE over all N rows (still divided by the whole batch's N);
    3. reduce-scatter dE (fp32): rank r receives the sum over ranks of rows [r n, (r + 1) n);
    4. all-reduce (sum) L, dt and db.

The band shares of ranks that partition the rows add up to the whole call, so every rank ends with the
whole batch's L, dt and db and its own rows of the whole batch's dE.  On NCCL the exchanges run on device
tensors; on other backends (gloo) they are staged through host memory.  The relations are those of the
whole batch, as the single-device call takes them (CSR over all N anchors, global item ids); a band call
reads only its own anchors' rows of them.

Only the collectives live here: every loss, gradient and contraction runs in the library's kernels
through the band call.
"""

from __future__ import annotations

import torch
import torch.distributed as dist


def _on_device(group) -> bool:
    return dist.get_backend(group) == "nccl"


def _all_gather_rows(local: torch.Tensor, world: int, group) -> torch.Tensor:
    """[world * n, ...] from every rank's [n, ...] (equal shares), exchanged as bytes."""
    raw = local.contiguous().view(torch.uint8)
    if _on_device(group):
        out = torch.empty((world * raw.shape[0],) + tuple(raw.shape[1:]), dtype=torch.uint8, device=raw.device)
        dist.all_gather_into_tensor(out, raw, group=group)
    else:
        host = raw.cpu()
        parts = [torch.empty_like(host) for _ in range(world)]
        dist.all_gather(parts, host, group=group)
        out = torch.cat(parts, dim=0).to(local.device)
    return out.view(local.dtype).view((world * local.shape[0],) + tuple(local.shape[1:]))


def _reduce_scatter_rows(full: torch.Tensor, world: int, rank: int, group) -> torch.Tensor:
    """This rank's [n, ...] rows of the sum over ranks of [world * n, ...]."""
    n = full.shape[0] // world
    if _on_device(group):
        out = torch.empty((n,) + tuple(full.shape[1:]), dtype=full.dtype, device=full.device)
        dist.reduce_scatter_tensor(out, full.contiguous(), group=group)
        return out
    host = full.contiguous().cpu()
    dist.all_reduce(host, group=group)
    return host[rank * n:(rank + 1) * n].to(full.device)


def _all_reduce_sum(t: torch.Tensor, group) -> torch.Tensor:
    if _on_device(group):
        dist.all_reduce(t, group=group)
        return t
    host = t.cpu()
    dist.all_reduce(host, group=group)
    return host.to(t.device)


def pair_loss_sigmoid_sharded(local_embeddings, inverse_temperature, bias, attract, repel=None, ignore=None,
                              negatives_named=False, ambient_weight=1.0, group=None, band_call=None):
    """One sharded pooled step on this rank.

    local_embeddings: bf16 [n, D], this rank's rows of the batch (every rank the same n).
    inverse_temperature, bias: fp32 device scalars, the same on every rank.
    attract, repel, ignore: device edge sets of the whole batch (see `device_edges`).
    Returns dict(loss, d_inverse_temperature, d_bias, d_embeddings) where the scalars are the whole batch's
    and d_embeddings (fp32 [n, D]) holds this rank's rows of the whole batch's dE.

    `band_call(embeddings, row_begin, row_count)` replaces the library's band call (it must return a dict
    with loss, d_embeddings, d_inverse_temperature, d_bias); by default it is `pair_loss_sigmoid_fwd_bwd`
    with `band=(row_begin, row_count)`.
    """
    world = dist.get_world_size(group)
    rank = dist.get_rank(group)
    n = local_embeddings.shape[0]
    e_all = _all_gather_rows(local_embeddings, world, group)
    if band_call is None:
        from ._binding import check_device_status, pair_loss_sigmoid_fwd_bwd

        def band_call(e, begin, count):
            r = pair_loss_sigmoid_fwd_bwd(e, inverse_temperature, bias, attract, repel, ignore,
                                          negatives_named=negatives_named, ambient_weight=ambient_weight,
                                          band=(begin, count))
            check_device_status(r["device_status"], "pair_loss_sigmoid_fwd_bwd")
            return r
    r = band_call(e_all, rank * n, n)
    de_local = _reduce_scatter_rows(r["d_embeddings"], world, rank, group)
    scalars = torch.cat([r["loss"].reshape(1), r["d_inverse_temperature"].reshape(1), r["d_bias"].reshape(1)])
    scalars = _all_reduce_sum(scalars.to(torch.float64), group)
    return dict(loss=scalars[0], d_inverse_temperature=scalars[1], d_bias=scalars[2], d_embeddings=de_local)
