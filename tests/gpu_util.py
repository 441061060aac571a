"""Helpers shared by the GPU tests: uploading seeded inputs and comparing against the oracle."""

import numpy as np
import torch

import contrastive_late_interaction_gb300 as cli

# Tolerances (the acceptance bar): losses and scores 2e-3 relative, gradients 1e-2 relative L2,
# argmax exact wherever the oracle's top-2 gap exceeds 1e-3.
LOSS_RTOL = 2e-3
SCORE_RTOL = 2e-3
GRAD_RL2 = 1e-2
ARGMAX_GAP = 1e-3


def dev():
    return torch.device("cuda:0")


def bf16(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16).copy()).view(torch.bfloat16).to(dev())


def i64(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.asarray(a, dtype=np.uint64).view(np.int64).copy()).to(dev())


def scalar(x: float) -> torch.Tensor:
    return torch.tensor([float(x)], dtype=torch.float32, device=dev())


def rel_l2(a, b) -> float:
    a, b = np.asarray(a, dtype=np.float64), np.asarray(b, dtype=np.float64)
    den = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / (den if den > 0 else 1.0))


def assert_rel(a, b, rtol, what):
    a, b = float(a), float(b)
    assert abs(a - b) <= rtol * max(abs(b), 1e-30), f"{what}: gpu {a!r} oracle {b!r}"


def near_tie_bound(s_max, abs_dot, width):
    """How far below the maximum a score the forward may pick as its argmax can lie.

    The forward compares scores truncated to keys (the low 5 of 23 mantissa bits replaced), which moves a
    value by less than 2^-18 of itself, so two values within that distance can compare equal; each score is
    also an fp32 accumulation of `width` exact bf16 products, off by at most about width * 2^-24 of the sum
    of the products' magnitudes (`abs_dot`).  Twice each term, for the two scores compared."""
    return 2.0 ** -17 * abs(s_max) + width * 2.0 ** -22 * abs_dot


def routed_argmax(m, gpu_arg, ora_arg, gap, rows=None, where=None):
    """The argmax the reference gradient routes through, [documents, rows] like the tables given.

    Where the oracle's top-2 gap exceeds ARGMAX_GAP the choice is unique and check_argmax has already
    required the GPU to make it.  Elsewhere several rows can be correct: the GPU's choice is kept after
    checking that it lies inside its document and scores within the forward's own near-tie bound
    (`near_tie_bound`) of the oracle's row, so the gradients are compared through the same valid routing.
    `rows` maps the tables' columns to query-tape rows (default: all rows in order); document d's rows
    start at m.d_offsets[d].  `where` (same shape) limits the routing to the entries a gradient reads
    (named pairs)."""
    use = np.array(ora_arg, dtype=np.int64, copy=True)
    gpu_arg = np.asarray(gpu_arg)
    rows = np.arange(use.shape[1]) if rows is None else np.asarray(rows)
    open_choice = (np.asarray(gap) <= ARGMAX_GAP) & (gpu_arg != use)
    todo = np.nonzero(open_choice if where is None else open_choice & where)
    q, dm = (m.q, m.d) if todo[0].size else (None, None)
    for d, c in zip(*todo):
        r0, r1 = int(m.d_offsets[d]), int(m.d_offsets[d + 1])
        jg, jo = int(gpu_arg[d, c]), int(use[d, c])
        assert 0 <= jg < r1 - r0, f"argmax {jg} outside document {d}"
        qt = q[rows[c]]
        s_g = float(qt @ dm[r0 + jg])
        s_o = float(qt @ dm[r0 + jo])
        bound = near_tie_bound(s_o, max(float(np.abs(qt) @ np.abs(dm[r0 + jg])),
                                        float(np.abs(qt) @ np.abs(dm[r0 + jo]))), m.width)
        assert s_o - s_g <= bound, \
            f"argmax {jg} of document {d} scores {s_g!r}, the maximum {s_o!r} (row {jo}) is {s_o - s_g:.3e} above it"
        use[d, c] = jg
    return use.astype(np.int32)


def run_pooled(p, weights=None, ld=None, ld_de=None, repel=None):
    """Runs the pooled loss on the GPU for synth.PooledInputs p.  Returns numpy outputs and the status."""
    e_bits = p.e_bf16
    width = p.width
    if ld is not None and ld > width:
        e_bits = np.zeros((p.count, ld), dtype=np.uint16)
        e_bits[:, :width] = p.e_bf16
    e = bf16(e_bits)
    out = {"width": width}
    if ld_de is not None:
        out["d_embeddings"] = torch.full((p.count, ld_de), 7.0, device=dev())[:, :width]
    r = cli.pair_loss_sigmoid_fwd_bwd(e, scalar(p.t), scalar(p.b), cli.device_edges(p.attract),
                                      cli.device_edges(repel if repel is not None else
                                                       (p.repel if p.repel.ids.size else None)),
                                      cli.device_edges(p.ignore if p.ignore.ids.size else None),
                                      negatives_named=p.negatives_named, ambient_weight=p.ambient_weight, out=out)
    torch.cuda.synchronize()
    status = int(r["device_status"].item())
    return dict(loss=r["loss"].item(), dt=r["d_inverse_temperature"].item(), db=r["d_bias"].item(),
                de=r["d_embeddings"].double().cpu().numpy(), status=status, raw=r)


def maxsim_tensors(m):
    return bf16(m.q_bf16), i64(m.q_offsets), bf16(m.d_bf16), i64(m.d_offsets)


def run_maxsim(m, mean=False, argmax=None):
    q, qo, d, do = maxsim_tensors(m)
    f = cli.maxsim_scores(q, qo, d, do, mean=mean)
    am = f["argmax"] if argmax is None else torch.from_numpy(np.ascontiguousarray(argmax, dtype=np.int32)).to(dev())
    ds = torch.from_numpy(np.ascontiguousarray(m.d_scores, dtype=np.float32)).to(dev())
    g = cli.maxsim_backward(q, qo, d, do, am, ds, mean=mean)
    torch.cuda.synchronize()
    return dict(scores=f["scores"].double().cpu().numpy(), argmax=f["argmax"].cpu().numpy(),
                dq=g["d_queries"].double().cpu().numpy(), dd=g["d_documents"].double().cpu().numpy(),
                status_f=int(f["device_status"].item()), status_b=int(g["device_status"].item()))


def check_scores(gpu, ref, what="scores"):
    err = np.abs(gpu - ref) / np.maximum(np.abs(ref), 1.0)
    assert err.max() <= SCORE_RTOL, f"{what}: max rel err {err.max():.3e}"


def check_argmax(gpu, ref, gap):
    """Exact agreement wherever the oracle's top-2 gap exceeds ARGMAX_GAP, and wherever the gap is zero:
    an exact tie, which both sides break to the lowest document row."""
    sure = (gap > ARGMAX_GAP) | (gap == 0)
    bad = np.count_nonzero(gpu[sure] != ref[sure])
    assert bad == 0, f"{bad} argmax mismatches of {np.count_nonzero(sure)} decided or exactly tied entries"
    return np.count_nonzero(sure)
