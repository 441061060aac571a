"""Float64 CPU oracle of the contrastive scoring path (TEST INFRASTRUCTURE ONLY).

Only `tests/`, `__graft_entry__.smoke()` and `bench.py`'s CPU-baseline leg (and
its `--impl reference` arm) may import this package.  The product path never
does: it shares no code with the CUDA library and is not a fallback for it.

The arithmetic lives in `cli_oracle.c` (plain C, float64); this module builds
it with gcc on first use and marshals numpy arrays through ctypes.

Pins: every function is checked by `tests/test_oracle.py` against closed
forms, brute force, finite differences and invariants; nothing here is
"parity unpinned".
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "cli_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libcli_oracle.so")
_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (float64, no fast-math) into oracle/_build/."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-fno-fast-math",
                        "-o", tmp, _SRC, "-lm"], check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            I64, D, I = ctypes.c_int64, ctypes.c_double, ctypes.c_int
            lib.oracle_sigmoid.argtypes = [D]
            lib.oracle_sigmoid.restype = D
            lib.oracle_softplus.argtypes = [D]
            lib.oracle_softplus.restype = D
            lib.oracle_pair_loss_sigmoid.argtypes = [I64, I64, P, D, D, P, P, P, P, P, P, P, P, I, D,
                                                     I64, P, P, P, P, P, P, I]
            lib.oracle_pair_loss_sigmoid_scores.argtypes = [I64, I64, P, D, D, P, P, P, P, P, P, P, P, P,
                                                            I, D, P, P, P, P]
            lib.oracle_pair_loss_scores_form.argtypes = [I, I64, I64, P, D, D, P, P, P, P, P, P, P, P, P,
                                                         I, D, P, P, P, P]
            lib.oracle_maxsim_pairs.argtypes = [I64, P, P, I64, P, P, I64, I, I64, P, P, P, P, P, P, I]
            lib.oracle_maxsim_forward.argtypes = [I64, P, P, I64, P, P, I64, I, P, P, P, I]
            lib.oracle_maxsim_backward.argtypes = [I64, P, P, I64, P, P, I64, I, P, P, P, P, I]
            lib.oracle_maxsim_grad_query.argtypes = [I64, P, P, I64, P, P, I64, I, I64, P, P]
            lib.oracle_maxsim_grad_doc.argtypes = [I64, P, P, I64, P, P, I64, I, I64, P, P]
            for f in ("oracle_pair_loss_sigmoid", "oracle_pair_loss_sigmoid_scores", "oracle_pair_loss_scores_form",
                      "oracle_maxsim_pairs",
                      "oracle_maxsim_forward", "oracle_maxsim_backward", "oracle_maxsim_grad_query",
                      "oracle_maxsim_grad_doc"):
                getattr(lib, f).restype = I
            _lib = lib
    return _lib


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _f64(a):
    return None if a is None else np.ascontiguousarray(a, dtype=np.float64)


def _u64(a):
    return None if a is None else np.ascontiguousarray(a, dtype=np.uint64)


def _u32(a):
    return None if a is None else np.ascontiguousarray(a, dtype=np.uint32)


def sigmoid(x: float) -> float:
    return _load().oracle_sigmoid(float(x))


def softplus(x: float) -> float:
    return _load().oracle_softplus(float(x))


def _edges(e):
    """(offsets, ids, weights) from an Edges-like object, a tuple, or None."""
    if e is None:
        return None, None, None
    if isinstance(e, tuple):
        off, ids = e[0], e[1]
        w = e[2] if len(e) > 2 else None
    else:
        off, ids, w = e.offsets, e.ids, e.weights
    if off is None:
        return None, None, None
    return _u64(off), _u32(ids if len(ids) else np.zeros(1, np.uint32)), _f64(w)


def pair_loss_sigmoid(e, t, b, attract=None, repel=None, ignore=None, negatives_named=False,
                      ambient_weight=1.0, rows=None, want_de=True, threads=None):
    """Pooled sigmoid pair loss.  Returns dict(loss, dt, db, de, row_loss).

    With `rows`, only those anchors are evaluated: `loss`, `dt`, `db` are their
    shares and `de`/`row_loss` have one entry per listed anchor.
    """
    lib = _load()
    e = _f64(e)
    n, w = e.shape
    ao, ai, aw = _edges(attract)
    ro, ri, rw = _edges(repel)
    io, ii, _ = _edges(ignore)
    sel = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    m = n if sel is None else len(sel)
    de = np.zeros((m, w)) if want_de else None
    row_loss = np.zeros(m)
    out = np.zeros(3)
    rc = lib.oracle_pair_loss_sigmoid(n, w, _ptr(e), float(t), float(b), _ptr(ao), _ptr(ai), _ptr(aw),
                                      _ptr(ro), _ptr(ri), _ptr(rw), _ptr(io), _ptr(ii), int(negatives_named),
                                      float(ambient_weight), m, _ptr(sel), _ptr(out[0:1]), _ptr(de),
                                      _ptr(row_loss), _ptr(out[1:2]), _ptr(out[2:3]),
                                      threads or default_threads())
    assert rc == 0
    return dict(loss=out[0], dt=out[1], db=out[2], de=de, row_loss=row_loss)


def _dense_relations(n, attract, repel, ignore, negatives_named, ambient_weight):
    """(Y, W): Y[i, j] = +1 attract, -1 repel, 0 skipped; W the weight; resolved in the documented order
    ("Training", `uform_relations_view_t`: ignore, then attract, then repel, then the negatives default;
    `uform_negatives_t`: ambient repels at `ambient_weight`, named scores only repel edges).  The diagonal
    is never scored."""
    Y = np.full((n, n), 0 if negatives_named else -1, dtype=np.int8)
    W = np.full((n, n), 0.0 if negatives_named else float(ambient_weight))

    def each(edges):
        off, ids, w = _edges(edges)
        if off is None:
            return
        for i in range(n):
            for k in range(int(off[i]), int(off[i + 1])):
                yield i, int(ids[k]), (1.0 if w is None else float(w[k]))

    for i, j, w in each(repel):
        Y[i, j], W[i, j] = -1, w
    for i, j, w in each(attract):
        Y[i, j], W[i, j] = 1, w
    for i, j, _ in each(ignore):
        Y[i, j], W[i, j] = 0, 0.0
    np.fill_diagonal(Y, 0)
    W[Y == 0] = 0.0
    return Y, W


def pair_loss_sigmoid_groups(e, groups, t, b, attract=None, repel=None, ignore=None, negatives_named=False,
                             ambient_weight=1.0, band=None):
    """Pooled sigmoid pair loss with temperature groups.  Returns dict(loss, dt, db, de) with dt, db one per
    group.

    "Training", `uform_contrastive_t` (`temperature_groups`: learnable (inverse temperature, bias) pairs,
    one per group a step's items select).  Reading: item i selects group g(i), and a cell takes its
    anchor's pair: z_ij = t[g(i)] s_ij + b[g(i)], l_ij = w_ij softplus(-y_ij z_ij), L = (1/N) sum l_ij
    (the SigLIP loss of "UForm", section "Matryoshka-Like Multi-Scale Embedders", per anchor).  Written out
    densely in float64 (a second formulation beside the C oracle, which it equals with one group).

    `band` = (row_begin, row_count) keeps only the cells whose anchor i lies in those rows, still divided
    by N: one device's share when the loss is sharded across devices ("UForm", section "Matryoshka-Like
    Multi-Scale Embedders": one SigLIP loss over the NVLink domain, the per-rank embeddings all-gathered
    into one similarity band and the gradients reduce-scattered back; the collectives are in section
    "NVLink-Based Cross-GPU Collaboration").  Read as: each rank scores its own items' rows against every
    gathered column, so the shares of bands that partition the rows add up to the whole.
    """
    e = _f64(e)
    n = e.shape[0]
    g = np.asarray(groups, dtype=np.int64)
    tv, bv = np.asarray(t, dtype=np.float64), np.asarray(b, dtype=np.float64)
    Y, W = _dense_relations(n, attract, repel, ignore, negatives_named, ambient_weight)
    if band is not None:
        lo, count = int(band[0]), int(band[1])
        outside = np.ones(n, dtype=bool)
        outside[lo:lo + count] = False
        W[outside, :] = 0.0
        Y[outside, :] = 0
    S = e @ e.T
    Z = tv[g][:, None] * S + bv[g][:, None]
    m = -Y * Z                                    # softplus(-y z) and its derivative sigma(-y z)
    sp = np.maximum(m, 0.0) + np.log1p(np.exp(-np.abs(m)))
    sg = np.where(m >= 0, 1.0 / (1.0 + np.exp(-np.abs(m))), np.exp(-np.abs(m)) / (1.0 + np.exp(-np.abs(m))))
    Gz = -W * Y * sg / n                          # dL/dz_ij
    loss = float(np.sum(W * sp) / n)
    dS = tv[g][:, None] * Gz
    de = (dS + dS.T) @ e
    dt = np.bincount(g, weights=np.sum(Gz * S, axis=1), minlength=len(tv))
    db = np.bincount(g, weights=np.sum(Gz, axis=1), minlength=len(tv))
    return dict(loss=loss, dt=dt, db=db, de=de)


def round_bf16(x):
    """Nearest-even rounding of float64 values to bfloat16 (through float32), returned as float64.
    The device scores bf16 copies of the normalised prefixes; the oracle scores the same values."""
    f = np.ascontiguousarray(x, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32).astype(np.float64)


def pair_loss_sigmoid_matryoshka(e, prefixes, t, b, attract=None, repel=None, ignore=None, negatives_named=False,
                                 ambient_weight=1.0, round_prefix=True, threads=None):
    """Matryoshka prefixes under the pooled sigmoid pair loss.  Returns dict(loss, dt, db, de, per_prefix).

    "Training", `uform_contrastive_t` (`matryoshka_dimensions`: ascending prefix widths, every one
    scored) and "UForm", section "Matryoshka-Like Multi-Scale Embedders" (each prefix trained under the
    SigLIP loss on cosine similarities).  Reading: with u_p,i = e_i[:p] / |e_i[:p]|,
        L = sum_p L_sigmoid(u_p),  one (t, b) for every prefix,
    and dE_i[:p] += (g_i - (g_i . u_i) u_i) / |e_i[:p]| with g = dL_p / du_p (the gradient of the
    normalisation).  A prefix of zero norm scores the zero vector and passes no gradient.  The device
    scores bf16 copies of u_p, so with `round_prefix` the oracle rounds u_p the same way before scoring
    and passes the gradient through that rounding unchanged.
    """
    e = _f64(e)
    n, w = e.shape
    de = np.zeros((n, w))
    tot = dict(loss=0.0, dt=0.0, db=0.0)
    per = []
    for p in prefixes:
        x = e[:, :p]
        norm = np.sqrt(np.sum(x * x, axis=1))
        inv = np.divide(1.0, norm, out=np.zeros_like(norm), where=norm > 0)
        u = x * inv[:, None]
        r = pair_loss_sigmoid(round_bf16(u) if round_prefix else u, t, b, attract, repel, ignore, negatives_named,
                              ambient_weight, threads=threads)
        g = r["de"]
        de[:, :p] += (g - np.sum(g * u, axis=1)[:, None] * u) * inv[:, None]
        for k in tot:
            tot[k] += r[k]
        per.append(dict(width=p, loss=r["loss"], dt=r["dt"], db=r["db"]))
    return dict(loss=tot["loss"], dt=tot["dt"], db=tot["db"], de=de, per_prefix=per)


def pair_loss_sigmoid_scores(scores, t, b, attract=None, repel=None, ignore=None, sides=None,
                             negatives_named=False, ambient_weight=1.0):
    """Sigmoid pair loss over a given score matrix [R, C].  Returns dict(loss, dt, db, dscores)."""
    lib = _load()
    s = _f64(scores)
    r, c = s.shape
    ao, ai, aw = _edges(attract)
    ro, ri, rw = _edges(repel)
    io, ii, _ = _edges(ignore)
    sd = None if sides is None else np.ascontiguousarray(sides, dtype=np.uint8)
    ds = np.zeros((r, c))
    out = np.zeros(3)
    rc = lib.oracle_pair_loss_sigmoid_scores(r, c, _ptr(s), float(t), float(b), _ptr(ao), _ptr(ai), _ptr(aw),
                                             _ptr(ro), _ptr(ri), _ptr(rw), _ptr(io), _ptr(ii), _ptr(sd),
                                             int(negatives_named), float(ambient_weight), _ptr(out[0:1]),
                                             _ptr(ds), _ptr(out[1:2]), _ptr(out[2:3]))
    assert rc == 0
    return dict(loss=out[0], dt=out[1], db=out[2], dscores=ds)


FORMS = {"balanced": 1, "ranked": 2}


def pair_loss_scores_form(form, scores, t, b, attract=None, repel=None, ignore=None, sides=None,
                          negatives_named=False, ambient_weight=1.0):
    """The `balanced` or `ranked` pair-loss form over a score matrix [R, C].  Returns dict(loss, dt, db,
    dscores)."""
    lib = _load()
    s = _f64(scores)
    r, c = s.shape
    ao, ai, aw = _edges(attract)
    ro, ri, rw = _edges(repel)
    io, ii, _ = _edges(ignore)
    sd = None if sides is None else np.ascontiguousarray(sides, dtype=np.uint8)
    ds = np.zeros((r, c))
    out = np.zeros(3)
    rc = lib.oracle_pair_loss_scores_form(FORMS[form], r, c, _ptr(s), float(t), float(b), _ptr(ao), _ptr(ai),
                                          _ptr(aw), _ptr(ro), _ptr(ri), _ptr(rw), _ptr(io), _ptr(ii), _ptr(sd),
                                          int(negatives_named), float(ambient_weight), _ptr(out[0:1]), _ptr(ds),
                                          _ptr(out[1:2]), _ptr(out[2:3]))
    assert rc == 0
    return dict(loss=out[0], dt=out[1], db=out[2], dscores=ds)


def maxsim_forward(q_off, q, d_off, d, mean=False, threads=None):
    """All pairs.  Returns (scores [nq, nd], argmax [nd, rows_q] int32, gap [nd, rows_q])."""
    lib = _load()
    q_off, d_off, q, d = _u64(q_off), _u64(d_off), _f64(q), _f64(d)
    nq, nd, w = len(q_off) - 1, len(d_off) - 1, q.shape[1]
    rows_q = int(q_off[-1])
    scores = np.zeros((nq, nd))
    argmax = np.zeros((nd, rows_q), dtype=np.int32)
    gap = np.zeros((nd, rows_q))
    rc = lib.oracle_maxsim_forward(nq, _ptr(q_off), _ptr(q), nd, _ptr(d_off), _ptr(d), w, int(mean),
                                   _ptr(scores), _ptr(argmax), _ptr(gap), threads or default_threads())
    assert rc == 0
    return scores, argmax, gap


def maxsim_pairs(q_off, q, d_off, d, pairs_q, pairs_d, mean=False, threads=None):
    """Listed pairs.  Returns (scores [P], argmax list, gap list) with one |q|-array per pair."""
    lib = _load()
    q_off, d_off, q, d = _u64(q_off), _u64(d_off), _f64(q), _f64(d)
    nq, nd, w = len(q_off) - 1, len(d_off) - 1, q.shape[1]
    pq = np.ascontiguousarray(pairs_q, dtype=np.int64)
    pd = np.ascontiguousarray(pairs_d, dtype=np.int64)
    lens = (q_off[pq + 1] - q_off[pq]).astype(np.int64)
    arg_off = np.zeros(len(pq) + 1, dtype=np.int64)
    arg_off[1:] = np.cumsum(lens)
    score = np.zeros(len(pq))
    argmax = np.zeros(int(arg_off[-1]), dtype=np.int32)
    gap = np.zeros(int(arg_off[-1]))
    rc = lib.oracle_maxsim_pairs(nq, _ptr(q_off), _ptr(q), nd, _ptr(d_off), _ptr(d), w, int(mean), len(pq),
                                 _ptr(pq), _ptr(pd), _ptr(arg_off), _ptr(score), _ptr(argmax), _ptr(gap),
                                 threads or default_threads())
    assert rc == 0
    return (score, [argmax[arg_off[k]:arg_off[k + 1]] for k in range(len(pq))],
            [gap[arg_off[k]:arg_off[k + 1]] for k in range(len(pq))])


def maxsim_backward(q_off, q, d_off, d, argmax, dscores, mean=False, threads=None):
    """Returns (dq [rows_q, W], dd [rows_d, W]) given the oracle's argmax [nd, rows_q]."""
    lib = _load()
    q_off, d_off, q, d = _u64(q_off), _u64(d_off), _f64(q), _f64(d)
    nq, nd, w = len(q_off) - 1, len(d_off) - 1, q.shape[1]
    am = np.ascontiguousarray(argmax, dtype=np.int32)
    ds = _f64(dscores)
    dq = np.zeros((int(q_off[-1]), w))
    dd = np.zeros((int(d_off[-1]), w))
    rc = lib.oracle_maxsim_backward(nq, _ptr(q_off), _ptr(q), nd, _ptr(d_off), _ptr(d), w, int(mean), _ptr(am),
                                    _ptr(ds), _ptr(dq), _ptr(dd), threads or default_threads())
    assert rc == 0
    return dq, dd


def maxsim_grad_query(q_off, q, d_off, d, qi, dscores_row, mean=False):
    """dQ rows of query `qi` (its own argmax computed inside)."""
    lib = _load()
    q_off, d_off, q, d = _u64(q_off), _u64(d_off), _f64(q), _f64(d)
    nq, nd, w = len(q_off) - 1, len(d_off) - 1, q.shape[1]
    out = np.zeros((int(q_off[qi + 1] - q_off[qi]), w))
    rc = lib.oracle_maxsim_grad_query(nq, _ptr(q_off), _ptr(q), nd, _ptr(d_off), _ptr(d), w, int(mean), int(qi),
                                      _ptr(_f64(dscores_row)), _ptr(out))
    assert rc == 0
    return out


def maxsim_grad_doc(q_off, q, d_off, d, di, dscores_col, mean=False):
    """dD rows of document `di` (its own argmax computed inside)."""
    lib = _load()
    q_off, d_off, q, d = _u64(q_off), _u64(d_off), _f64(q), _f64(d)
    nq, nd, w = len(q_off) - 1, len(d_off) - 1, q.shape[1]
    out = np.zeros((int(d_off[di + 1] - d_off[di]), w))
    rc = lib.oracle_maxsim_grad_doc(nq, _ptr(q_off), _ptr(q), nd, _ptr(d_off), _ptr(d), w, int(mean), int(di),
                                    _ptr(_f64(dscores_col)), _ptr(out))
    assert rc == 0
    return out
