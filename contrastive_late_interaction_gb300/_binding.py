"""Thin ctypes binding over the C ABI of include/cli.h (argument marshalling only).

Every function here fills the verb's argument struct from torch tensors that
already live on the GPU, calls the exported C symbol of the same name, and
turns a non-OK status into an exception.  All arithmetic happens in the CUDA
library; if it is missing, importing this module raises.  PyTorch is used only
for device memory and streams.
"""

from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

c_size_t, c_void_p, c_int, c_float = ctypes.c_size_t, ctypes.c_void_p, ctypes.c_int, ctypes.c_float

STATUS_NAMES = ["ok", "invalid-argument", "shape-mismatch", "unsupported", "device", "malformed", "internal"]
CLI_OK, CLI_INVALID_ARGUMENT, CLI_SHAPE_MISMATCH, CLI_UNSUPPORTED, CLI_DEVICE, CLI_MALFORMED, CLI_INTERNAL = range(7)


class CliError(RuntimeError):
    """A non-OK status from the library; `status` is the cli_status_t value."""

    def __init__(self, status: int, where: str):
        self.status = int(status)
        super().__init__(f"{where}: {status_name(status)} ({status})")


class InvalidArgumentError(CliError, ValueError):
    pass


class ShapeMismatchError(CliError, ValueError):
    pass


class UnsupportedError(CliError, NotImplementedError):
    pass


class MalformedError(CliError, ValueError):
    pass


class DeviceError(CliError):
    pass


class InternalError(CliError):
    pass


_ERRORS = {CLI_INVALID_ARGUMENT: InvalidArgumentError, CLI_SHAPE_MISMATCH: ShapeMismatchError,
           CLI_UNSUPPORTED: UnsupportedError, CLI_MALFORMED: MalformedError, CLI_DEVICE: DeviceError,
           CLI_INTERNAL: InternalError}


def raise_for(status: int, where: str):
    if status != CLI_OK:
        raise _ERRORS.get(int(status), CliError)(status, where)


# ----------------------------------------------------------------------------
# structs (field for field as in include/cli.h)
# ----------------------------------------------------------------------------

class Edges(ctypes.Structure):
    _fields_ = [("offsets", c_void_p), ("ids", c_void_p), ("weights", c_void_p), ("edges", c_size_t)]


class Relations(ctypes.Structure):
    _fields_ = [("attract", Edges), ("repel", Edges), ("ignore", Edges), ("negatives_named", c_int),
                ("ambient_weight", c_float)]


class PairLossSigmoidArgs(ctypes.Structure):
    _fields_ = [("count", c_size_t), ("width", c_size_t), ("ld", c_size_t), ("embeddings", c_void_p),
                ("inverse_temperature", c_void_p), ("bias", c_void_p), ("relations", Relations),
                ("loss", c_void_p), ("d_embeddings", c_void_p), ("ld_d_embeddings", c_size_t),
                ("d_inverse_temperature", c_void_p), ("d_bias", c_void_p), ("workspace", c_void_p),
                ("workspace_bytes", c_size_t), ("device_status", c_void_p), ("stream", c_void_p),
                ("row_begin", c_size_t), ("row_count", c_size_t)]


class PairLossGroupsArgs(ctypes.Structure):
    _fields_ = [("base", PairLossSigmoidArgs), ("groups", c_void_p), ("group_count", c_size_t)]


class PairLossMatryoshkaArgs(ctypes.Structure):
    _fields_ = [("base", PairLossSigmoidArgs), ("prefix_widths", c_void_p), ("prefix_count", c_size_t),
                ("prefix_loss", c_void_p)]


MATRYOSHKA_MAX_PREFIXES = 8   # CLI_MATRYOSHKA_MAX_PREFIXES in include/cli.h


class PairLossSigmoidScoresArgs(ctypes.Structure):
    _fields_ = [("rows", c_size_t), ("cols", c_size_t), ("ld", c_size_t), ("scores", c_void_p),
                ("inverse_temperature", c_void_p), ("bias", c_void_p), ("relations", Relations),
                ("sides", c_void_p), ("loss", c_void_p), ("d_scores", c_void_p), ("ld_d_scores", c_size_t),
                ("d_inverse_temperature", c_void_p), ("d_bias", c_void_p), ("workspace", c_void_p),
                ("workspace_bytes", c_size_t), ("device_status", c_void_p), ("stream", c_void_p)]


class PairLossScoresArgs(ctypes.Structure):
    _fields_ = [("form", c_int), ("args", PairLossSigmoidScoresArgs)]


FORMS = {"balanced": 1, "ranked": 2, "sigmoid": 3}


class Tape(ctypes.Structure):
    _fields_ = [("data", c_void_p), ("offsets", c_void_p), ("count", c_size_t), ("rows", c_size_t)]


class MaxSimArgs(ctypes.Structure):
    _fields_ = [("queries", Tape), ("documents", Tape), ("width", c_size_t), ("mean", c_int),
                ("scores", c_void_p), ("ld_scores", c_size_t), ("argmax", c_void_p), ("ld_argmax", c_size_t),
                ("workspace", c_void_p), ("workspace_bytes", c_size_t), ("device_status", c_void_p),
                ("stream", c_void_p)]


class MaxSimNamedArgs(ctypes.Structure):
    _fields_ = [("base", MaxSimArgs), ("pairs", Edges)]


class MaxSimBackwardArgs(ctypes.Structure):
    _fields_ = [("queries", Tape), ("documents", Tape), ("width", c_size_t), ("mean", c_int),
                ("argmax", c_void_p), ("ld_argmax", c_size_t), ("d_scores", c_void_p), ("ld_d_scores", c_size_t),
                ("d_queries", c_void_p), ("d_documents", c_void_p), ("workspace", c_void_p),
                ("workspace_bytes", c_size_t), ("device_status", c_void_p), ("stream", c_void_p)]


class MaxSimBackwardNamedArgs(ctypes.Structure):
    _fields_ = [("base", MaxSimBackwardArgs), ("pairs", Edges)]


EXPORTS = {
    "cli_status_name": (ctypes.c_char_p, [c_int]),
    "pair_loss_sigmoid_fwd_bwd": (c_int, [ctypes.POINTER(PairLossSigmoidArgs)]),
    "pair_loss_sigmoid_workspace_bytes": (c_size_t, [c_size_t, c_size_t, c_size_t]),
    "pair_loss_sigmoid_groups_fwd_bwd": (c_int, [ctypes.POINTER(PairLossGroupsArgs)]),
    "pair_loss_sigmoid_matryoshka_fwd_bwd": (c_int, [ctypes.POINTER(PairLossMatryoshkaArgs)]),
    "pair_loss_sigmoid_matryoshka_workspace_bytes": (c_size_t, [c_size_t, c_size_t, c_size_t]),
    "pair_loss_sigmoid_scores_fwd_bwd": (c_int, [ctypes.POINTER(PairLossSigmoidScoresArgs)]),
    "pair_loss_sigmoid_scores_workspace_bytes": (c_size_t, [c_size_t, c_size_t]),
    "pair_loss_scores_fwd_bwd": (c_int, [ctypes.POINTER(PairLossScoresArgs)]),
    "pair_loss_scores_workspace_bytes": (c_size_t, [c_int, c_size_t, c_size_t]),
    "maxsim_scores": (c_int, [ctypes.POINTER(MaxSimArgs)]),
    "maxsim_workspace_bytes": (c_size_t, [c_size_t, c_size_t, c_size_t, c_size_t, c_size_t]),
    "maxsim_scores_named": (c_int, [ctypes.POINTER(MaxSimNamedArgs)]),
    "maxsim_named_workspace_bytes": (c_size_t, [c_size_t, c_size_t, c_size_t, c_size_t, c_size_t]),
    "maxsim_backward": (c_int, [ctypes.POINTER(MaxSimBackwardArgs)]),
    "maxsim_backward_named": (c_int, [ctypes.POINTER(MaxSimBackwardNamedArgs)]),
    "maxsim_backward_workspace_bytes": (c_size_t, [c_size_t, c_size_t, c_size_t, c_size_t, c_size_t]),
    "maxsim_backward_no_alloc": (c_int, [ctypes.POINTER(MaxSimBackwardArgs)]),
    "cli_selftest_bounded_wait": (c_int, [c_void_p, c_void_p, ctypes.c_uint32, c_void_p]),
}
NO_ALLOC_MAX_QUERY_ROWS = 262144   # CLI_MAXSIM_NO_ALLOC_MAX_QUERY_ROWS in include/cli.h


def _load():
    path = _build.LIB
    if not os.path.exists(path):
        raise ImportError(f"the CUDA library {path} is not built; run __graft_entry__.build() "
                          "(there is no CPU fallback)")
    lib = ctypes.CDLL(path)
    for name, (res, args) in EXPORTS.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


lib = _load()
LIB_PATH = _build.LIB


def status_name(status: int) -> str:
    return lib.cli_status_name(int(status)).decode()


# ----------------------------------------------------------------------------
# marshalling helpers
# ----------------------------------------------------------------------------

def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _check_cuda(t, name, dtype=None):
    if t is None:
        return
    if not t.is_cuda:
        raise InvalidArgumentError(CLI_INVALID_ARGUMENT, f"{name} must be device memory")
    if dtype is not None and t.dtype != dtype:
        raise InvalidArgumentError(CLI_INVALID_ARGUMENT, f"{name} must be {dtype}")


def _edges(e, count):
    """(offsets int64[count+1], ids int32[E], weights float32[E] | None) on the device -> Edges."""
    if e is None:
        return Edges(None, None, None, 0)
    off, ids = e[0], e[1]
    w = e[2] if len(e) > 2 else None
    _check_cuda(off, "offsets", torch.int64)
    _check_cuda(ids, "ids", torch.int32)
    _check_cuda(w, "weights", torch.float32)
    return Edges(_ptr(off), _ptr(ids) if ids.numel() else None, _ptr(w), int(ids.numel()))


def device_edges(edges, device="cuda"):
    """Uploads a host edge set (offsets, ids[, weights] numpy arrays or an object with those fields)."""
    if edges is None:
        return None
    if hasattr(edges, "offsets"):
        off, ids, w = edges.offsets, edges.ids, edges.weights
    else:
        off, ids = edges[0], edges[1]
        w = edges[2] if len(edges) > 2 else None
    import numpy as np
    o = torch.from_numpy(np.asarray(off, dtype=np.uint64).view(np.int64).copy()).to(device)
    i = torch.from_numpy(np.asarray(ids, dtype=np.uint32).view(np.int32).copy()).to(device)
    ww = None if w is None else torch.from_numpy(np.asarray(w, dtype=np.float32).copy()).to(device)
    return (o, i, ww) if ww is not None else (o, i)


def _band(band):
    """The anchor band (row_begin, row_count) of a pooled call; None is every row.  The library checks it."""
    if band is None:
        return dict(row_begin=0, row_count=0)
    begin, count = (int(v) for v in band)
    if begin < 0 or count < 0:
        raise ShapeMismatchError(CLI_SHAPE_MISMATCH, "band must be (row_begin, row_count) >= 0")
    return dict(row_begin=begin, row_count=count)


def _ws(nbytes, device):
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)


def selftest_bounded_wait(limit_us=20000, device_status=None, gave_up=None, stream=None):
    """Runs the failure path of the kernels' bounded waits (one CTA waiting on a barrier nothing arrives
    at, giving up after `limit_us`).  Returns dict(device_status, gave_up) of device int32 tensors; the
    status reads CLI_INTERNAL and gave_up the number of threads (64) once the stream reaches them."""
    dev = torch.device("cuda", torch.cuda.current_device())
    st = device_status if device_status is not None else torch.zeros(1, dtype=torch.int32, device=dev)
    gu = gave_up if gave_up is not None else torch.zeros(1, dtype=torch.int32, device=dev)
    _check_cuda(st, "device_status", torch.int32)
    _check_cuda(gu, "gave_up", torch.int32)
    raise_for(lib.cli_selftest_bounded_wait(_ptr(st), _ptr(gu), int(limit_us), _stream(stream)),
              "cli_selftest_bounded_wait")
    return dict(device_status=st, gave_up=gu)


def check_device_status(status: torch.Tensor, where: str = "device"):
    """Synchronises on the status word and raises if the device reported a fault."""
    raise_for(int(status.item()), where)


# ----------------------------------------------------------------------------
# verbs
# ----------------------------------------------------------------------------

def pair_loss_sigmoid_workspace_bytes(count, width, edges):
    return int(lib.pair_loss_sigmoid_workspace_bytes(count, width, edges))


def pair_loss_sigmoid_fwd_bwd(embeddings, inverse_temperature, bias, attract, repel=None, ignore=None,
                              negatives_named=False, ambient_weight=1.0, out=None, workspace=None,
                              device_status=None, stream=None, band=None):
    """Pooled sigmoid pair loss over bf16 embeddings [N, ld] (first `width` = embeddings.shape[1] columns
    unless `out['width']` narrows it).  Returns dict(loss, d_embeddings, d_inverse_temperature, d_bias,
    device_status) of device tensors; the device status is not synchronised here.  `band` = (row_begin,
    row_count) scores only the anchors in those rows: the results are that band's shares of the whole call's."""
    _check_cuda(embeddings, "embeddings", torch.bfloat16)
    _check_cuda(inverse_temperature, "inverse_temperature", torch.float32)
    _check_cuda(bias, "bias", torch.float32)
    n, ld = embeddings.shape
    width = (out or {}).get("width", ld)
    dev = embeddings.device
    out = dict(out or {})
    loss = out.get("loss") if out.get("loss") is not None else torch.empty(1, device=dev)
    de = out.get("d_embeddings") if out.get("d_embeddings") is not None else torch.empty(n, width, device=dev)
    dt = out.get("d_inverse_temperature") if out.get("d_inverse_temperature") is not None else torch.empty(1, device=dev)
    db = out.get("d_bias") if out.get("d_bias") is not None else torch.empty(1, device=dev)
    st = device_status if device_status is not None else torch.zeros(1, dtype=torch.int32, device=dev)
    A, R, I = _edges(attract, n), _edges(repel, n), _edges(ignore, n)
    total = A.edges + R.edges + I.edges
    need = pair_loss_sigmoid_workspace_bytes(n, width, total)
    ws = workspace if workspace is not None else _ws(need, dev)
    args = PairLossSigmoidArgs(
        count=n, width=width, ld=embeddings.stride(0), embeddings=_ptr(embeddings),
        inverse_temperature=_ptr(inverse_temperature), bias=_ptr(bias),
        relations=Relations(A, R, I, int(bool(negatives_named)), float(ambient_weight)),
        loss=_ptr(loss), d_embeddings=_ptr(de), ld_d_embeddings=de.stride(0),
        d_inverse_temperature=_ptr(dt), d_bias=_ptr(db), workspace=_ptr(ws), workspace_bytes=ws.numel(),
        device_status=_ptr(st), stream=_stream(stream), **_band(band))
    raise_for(lib.pair_loss_sigmoid_fwd_bwd(ctypes.byref(args)), "pair_loss_sigmoid_fwd_bwd")
    return dict(loss=loss, d_embeddings=de, d_inverse_temperature=dt, d_bias=db, device_status=st)


def pair_loss_sigmoid_groups_fwd_bwd(embeddings, groups, inverse_temperature, bias, attract, repel=None, ignore=None,
                                     negatives_named=False, ambient_weight=1.0, out=None, workspace=None,
                                     device_status=None, stream=None, band=None):
    """The pooled sigmoid pair loss with temperature groups: `groups` (int32 [N]) selects each item's pair of
    `inverse_temperature`, `bias` (fp32 [G]) and a cell takes its anchor's.  Returns dict(loss, d_embeddings,
    d_inverse_temperature [G], d_bias [G], device_status) of device tensors."""
    _check_cuda(embeddings, "embeddings", torch.bfloat16)
    _check_cuda(groups, "groups", torch.int32)
    _check_cuda(inverse_temperature, "inverse_temperature", torch.float32)
    _check_cuda(bias, "bias", torch.float32)
    n, ld = embeddings.shape
    g = inverse_temperature.numel()
    if bias.numel() != g or groups.numel() != n:
        raise ShapeMismatchError(CLI_SHAPE_MISMATCH, "groups, inverse_temperature and bias disagree in size")
    width = (out or {}).get("width", ld)
    dev = embeddings.device
    out = dict(out or {})
    loss = out.get("loss") if out.get("loss") is not None else torch.empty(1, device=dev)
    de = out.get("d_embeddings") if out.get("d_embeddings") is not None else torch.empty(n, width, device=dev)
    dt = out.get("d_inverse_temperature") if out.get("d_inverse_temperature") is not None else torch.empty(g, device=dev)
    db = out.get("d_bias") if out.get("d_bias") is not None else torch.empty(g, device=dev)
    st = device_status if device_status is not None else torch.zeros(1, dtype=torch.int32, device=dev)
    A, R, I = _edges(attract, n), _edges(repel, n), _edges(ignore, n)
    total = A.edges + R.edges + I.edges
    need = pair_loss_sigmoid_workspace_bytes(n, width, total)
    ws = workspace if workspace is not None else _ws(need, dev)
    base = PairLossSigmoidArgs(
        count=n, width=width, ld=embeddings.stride(0), embeddings=_ptr(embeddings),
        inverse_temperature=_ptr(inverse_temperature), bias=_ptr(bias),
        relations=Relations(A, R, I, int(bool(negatives_named)), float(ambient_weight)),
        loss=_ptr(loss), d_embeddings=_ptr(de), ld_d_embeddings=de.stride(0),
        d_inverse_temperature=_ptr(dt), d_bias=_ptr(db), workspace=_ptr(ws), workspace_bytes=ws.numel(),
        device_status=_ptr(st), stream=_stream(stream), **_band(band))
    args = PairLossGroupsArgs(base=base, groups=_ptr(groups), group_count=g)
    raise_for(lib.pair_loss_sigmoid_groups_fwd_bwd(ctypes.byref(args)), "pair_loss_sigmoid_groups_fwd_bwd")
    return dict(loss=loss, d_embeddings=de, d_inverse_temperature=dt, d_bias=db, device_status=st)


def pair_loss_sigmoid_matryoshka_workspace_bytes(count, width, edges):
    return int(lib.pair_loss_sigmoid_matryoshka_workspace_bytes(count, width, edges))


def pair_loss_sigmoid_matryoshka_fwd_bwd(embeddings, prefix_widths, inverse_temperature, bias, attract, repel=None,
                                         ignore=None, negatives_named=False, ambient_weight=1.0, out=None,
                                         workspace=None, device_status=None, stream=None, band=None):
    """The pooled sigmoid pair loss summed over the normalised prefixes `prefix_widths` of bf16 embeddings
    [N, ld] (first `width` = embeddings.shape[1] columns unless `out['width']` narrows it).  Returns
    dict(loss, d_embeddings, d_inverse_temperature, d_bias, prefix_loss, device_status) of device tensors."""
    _check_cuda(embeddings, "embeddings", torch.bfloat16)
    _check_cuda(inverse_temperature, "inverse_temperature", torch.float32)
    _check_cuda(bias, "bias", torch.float32)
    n, ld = embeddings.shape
    width = (out or {}).get("width", ld)
    dev = embeddings.device
    out = dict(out or {})
    widths = (c_size_t * len(prefix_widths))(*[int(p) for p in prefix_widths])
    loss = out.get("loss") if out.get("loss") is not None else torch.empty(1, device=dev)
    de = out.get("d_embeddings") if out.get("d_embeddings") is not None else torch.empty(n, width, device=dev)
    dt = out.get("d_inverse_temperature") if out.get("d_inverse_temperature") is not None else torch.empty(1, device=dev)
    db = out.get("d_bias") if out.get("d_bias") is not None else torch.empty(1, device=dev)
    pl = out.get("prefix_loss") if out.get("prefix_loss") is not None else torch.empty(max(1, len(prefix_widths)),
                                                                                         device=dev)
    st = device_status if device_status is not None else torch.zeros(1, dtype=torch.int32, device=dev)
    A, R, I = _edges(attract, n), _edges(repel, n), _edges(ignore, n)
    total = A.edges + R.edges + I.edges
    need = pair_loss_sigmoid_matryoshka_workspace_bytes(n, width, total)
    ws = workspace if workspace is not None else _ws(need, dev)
    base = PairLossSigmoidArgs(
        count=n, width=width, ld=embeddings.stride(0), embeddings=_ptr(embeddings),
        inverse_temperature=_ptr(inverse_temperature), bias=_ptr(bias),
        relations=Relations(A, R, I, int(bool(negatives_named)), float(ambient_weight)),
        loss=_ptr(loss), d_embeddings=_ptr(de), ld_d_embeddings=de.stride(0),
        d_inverse_temperature=_ptr(dt), d_bias=_ptr(db), workspace=_ptr(ws), workspace_bytes=ws.numel(),
        device_status=_ptr(st), stream=_stream(stream), **_band(band))
    args = PairLossMatryoshkaArgs(base=base, prefix_widths=ctypes.cast(widths, c_void_p),
                                  prefix_count=len(prefix_widths), prefix_loss=_ptr(pl))
    raise_for(lib.pair_loss_sigmoid_matryoshka_fwd_bwd(ctypes.byref(args)), "pair_loss_sigmoid_matryoshka_fwd_bwd")
    return dict(loss=loss, d_embeddings=de, d_inverse_temperature=dt, d_bias=db, prefix_loss=pl, device_status=st)


def pair_loss_sigmoid_scores_workspace_bytes(rows, cols):
    return int(lib.pair_loss_sigmoid_scores_workspace_bytes(rows, cols))


def pair_loss_sigmoid_scores_fwd_bwd(scores, inverse_temperature, bias, attract, repel=None, ignore=None,
                                     sides=None, negatives_named=False, ambient_weight=1.0, out=None,
                                     workspace=None, device_status=None, stream=None):
    """Sigmoid pair loss over an fp32 score matrix [rows, cols]."""
    _check_cuda(scores, "scores", torch.float32)
    _check_cuda(sides, "sides", torch.uint8)
    rows, cols = scores.shape
    dev = scores.device
    out = dict(out or {})
    loss = out.get("loss") if out.get("loss") is not None else torch.empty(1, device=dev)
    ds = out.get("d_scores") if out.get("d_scores") is not None else torch.empty(rows, cols, device=dev)
    dt = out.get("d_inverse_temperature") if out.get("d_inverse_temperature") is not None else torch.empty(1, device=dev)
    db = out.get("d_bias") if out.get("d_bias") is not None else torch.empty(1, device=dev)
    st = device_status if device_status is not None else torch.zeros(1, dtype=torch.int32, device=dev)
    ws = workspace if workspace is not None else _ws(pair_loss_sigmoid_scores_workspace_bytes(rows, cols), dev)
    A, R, I = _edges(attract, rows), _edges(repel, rows), _edges(ignore, rows)
    args = PairLossSigmoidScoresArgs(
        rows=rows, cols=cols, ld=scores.stride(0), scores=_ptr(scores), inverse_temperature=_ptr(inverse_temperature),
        bias=_ptr(bias), relations=Relations(A, R, I, int(bool(negatives_named)), float(ambient_weight)),
        sides=_ptr(sides), loss=_ptr(loss), d_scores=_ptr(ds), ld_d_scores=ds.stride(0),
        d_inverse_temperature=_ptr(dt), d_bias=_ptr(db), workspace=_ptr(ws), workspace_bytes=ws.numel(),
        device_status=_ptr(st), stream=_stream(stream))
    raise_for(lib.pair_loss_sigmoid_scores_fwd_bwd(ctypes.byref(args)), "pair_loss_sigmoid_scores_fwd_bwd")
    return dict(loss=loss, d_scores=ds, d_inverse_temperature=dt, d_bias=db, device_status=st)


def pair_loss_scores_workspace_bytes(form, rows, cols):
    return int(lib.pair_loss_scores_workspace_bytes(FORMS[form], rows, cols))


def pair_loss_scores_fwd_bwd(form, scores, inverse_temperature, bias, attract, repel=None, ignore=None, sides=None,
                             negatives_named=False, ambient_weight=1.0, out=None, workspace=None, device_status=None,
                             stream=None):
    """Pair loss of form 'balanced', 'ranked' or 'sigmoid' over an fp32 score matrix [rows, cols]."""
    _check_cuda(scores, "scores", torch.float32)
    _check_cuda(sides, "sides", torch.uint8)
    rows, cols = scores.shape
    dev = scores.device
    out = dict(out or {})
    loss = out.get("loss") if out.get("loss") is not None else torch.empty(1, device=dev)
    ds = out.get("d_scores") if out.get("d_scores") is not None else torch.empty(rows, cols, device=dev)
    dt = out.get("d_inverse_temperature") if out.get("d_inverse_temperature") is not None else torch.empty(1, device=dev)
    db = out.get("d_bias") if out.get("d_bias") is not None else torch.empty(1, device=dev)
    st = device_status if device_status is not None else torch.zeros(1, dtype=torch.int32, device=dev)
    ws = workspace if workspace is not None else _ws(pair_loss_scores_workspace_bytes(form, rows, cols), dev)
    A, R, I = _edges(attract, rows), _edges(repel, rows), _edges(ignore, rows)
    inner = PairLossSigmoidScoresArgs(
        rows=rows, cols=cols, ld=scores.stride(0), scores=_ptr(scores), inverse_temperature=_ptr(inverse_temperature),
        bias=_ptr(bias), relations=Relations(A, R, I, int(bool(negatives_named)), float(ambient_weight)),
        sides=_ptr(sides), loss=_ptr(loss), d_scores=_ptr(ds), ld_d_scores=ds.stride(0),
        d_inverse_temperature=_ptr(dt), d_bias=_ptr(db), workspace=_ptr(ws), workspace_bytes=ws.numel(),
        device_status=_ptr(st), stream=_stream(stream))
    args = PairLossScoresArgs(form=FORMS[form], args=inner)
    raise_for(lib.pair_loss_scores_fwd_bwd(ctypes.byref(args)), "pair_loss_scores_fwd_bwd")
    return dict(loss=loss, d_scores=ds, d_inverse_temperature=dt, d_bias=db, device_status=st)


def _tape(data, offsets):
    _check_cuda(data, "tape data", torch.bfloat16)
    _check_cuda(offsets, "tape offsets", torch.int64)
    return Tape(_ptr(data), _ptr(offsets), offsets.numel() - 1, data.shape[0])


def maxsim_workspace_bytes(nq, nd, rows_q, rows_d, width):
    return int(lib.maxsim_workspace_bytes(nq, nd, rows_q, rows_d, width))


def maxsim_backward_workspace_bytes(nq, nd, rows_q, rows_d, width):
    return int(lib.maxsim_backward_workspace_bytes(nq, nd, rows_q, rows_d, width))


def maxsim_scores(q_data, q_offsets, d_data, d_offsets, mean=False, out=None, workspace=None, device_status=None,
                  stream=None):
    """Hard MaxSim of every query against every document.  Returns dict(scores [nq, nd] fp32,
    argmax [nd, rows_q] int32 (document-major), device_status)."""
    Q, D = _tape(q_data, q_offsets), _tape(d_data, d_offsets)
    width = q_data.shape[1]
    if d_data.shape[1] != width:
        raise ShapeMismatchError(CLI_SHAPE_MISMATCH, "maxsim_scores: query and document widths differ")
    dev = q_data.device
    out = dict(out or {})
    scores = out.get("scores") if out.get("scores") is not None else torch.empty(Q.count, D.count, device=dev)
    argmax = out.get("argmax") if out.get("argmax") is not None else torch.empty(D.count, Q.rows, dtype=torch.int32,
                                                                                  device=dev)
    st = device_status if device_status is not None else torch.zeros(1, dtype=torch.int32, device=dev)
    ws = workspace if workspace is not None else _ws(maxsim_workspace_bytes(Q.count, D.count, Q.rows, D.rows, width),
                                                     dev)
    args = MaxSimArgs(queries=Q, documents=D, width=width, mean=int(bool(mean)), scores=_ptr(scores),
                      ld_scores=scores.stride(0), argmax=_ptr(argmax), ld_argmax=argmax.stride(0),
                      workspace=_ptr(ws), workspace_bytes=ws.numel(), device_status=_ptr(st), stream=_stream(stream))
    raise_for(lib.maxsim_scores(ctypes.byref(args)), "maxsim_scores")
    return dict(scores=scores, argmax=argmax, device_status=st)


def maxsim_named_workspace_bytes(nq, nd, rows_q, rows_d, width):
    return int(lib.maxsim_named_workspace_bytes(nq, nd, rows_q, rows_d, width))


def maxsim_scores_named(q_data, q_offsets, d_data, d_offsets, pairs, mean=False, out=None, workspace=None,
                        device_status=None, stream=None):
    """Hard MaxSim of each query against the documents `pairs` names (a CSR over the queries, as from
    `device_edges`).  Returns dict(scores [nq, nd] fp32, zero for pairs not named, argmax [nd, rows_q] int32,
    a valid row of the document for pairs not named, device_status)."""
    Q, D = _tape(q_data, q_offsets), _tape(d_data, d_offsets)
    width = q_data.shape[1]
    if d_data.shape[1] != width:
        raise ShapeMismatchError(CLI_SHAPE_MISMATCH, "maxsim_scores_named: query and document widths differ")
    dev = q_data.device
    out = dict(out or {})
    scores = out.get("scores") if out.get("scores") is not None else torch.empty(Q.count, D.count, device=dev)
    argmax = out.get("argmax") if out.get("argmax") is not None else torch.empty(D.count, Q.rows, dtype=torch.int32,
                                                                                  device=dev)
    st = device_status if device_status is not None else torch.zeros(1, dtype=torch.int32, device=dev)
    ws = workspace if workspace is not None else _ws(
        maxsim_named_workspace_bytes(Q.count, D.count, Q.rows, D.rows, width), dev)
    base = MaxSimArgs(queries=Q, documents=D, width=width, mean=int(bool(mean)), scores=_ptr(scores),
                      ld_scores=scores.stride(0), argmax=_ptr(argmax), ld_argmax=argmax.stride(0),
                      workspace=_ptr(ws), workspace_bytes=ws.numel(), device_status=_ptr(st), stream=_stream(stream))
    args = MaxSimNamedArgs(base=base, pairs=_edges(pairs, Q.count))
    raise_for(lib.maxsim_scores_named(ctypes.byref(args)), "maxsim_scores_named")
    return dict(scores=scores, argmax=argmax, device_status=st)


def maxsim_backward(q_data, q_offsets, d_data, d_offsets, argmax, d_scores, mean=False, out=None, workspace=None,
                    device_status=None, stream=None):
    """Gradient through the argmax.  Returns dict(d_queries, d_documents, device_status)."""
    Q, D = _tape(q_data, q_offsets), _tape(d_data, d_offsets)
    _check_cuda(argmax, "argmax", torch.int32)
    _check_cuda(d_scores, "d_scores", torch.float32)
    width = q_data.shape[1]
    dev = q_data.device
    out = dict(out or {})
    dq = out.get("d_queries") if out.get("d_queries") is not None else torch.empty(Q.rows, width, device=dev)
    dd = out.get("d_documents") if out.get("d_documents") is not None else torch.empty(D.rows, width, device=dev)
    st = device_status if device_status is not None else torch.zeros(1, dtype=torch.int32, device=dev)
    ws = workspace if workspace is not None else _ws(
        maxsim_backward_workspace_bytes(Q.count, D.count, Q.rows, D.rows, width), dev)
    args = MaxSimBackwardArgs(queries=Q, documents=D, width=width, mean=int(bool(mean)), argmax=_ptr(argmax),
                              ld_argmax=argmax.stride(0), d_scores=_ptr(d_scores), ld_d_scores=d_scores.stride(0),
                              d_queries=_ptr(dq), d_documents=_ptr(dd), workspace=_ptr(ws),
                              workspace_bytes=ws.numel(), device_status=_ptr(st), stream=_stream(stream))
    raise_for(lib.maxsim_backward(ctypes.byref(args)), "maxsim_backward")
    return dict(d_queries=dq, d_documents=dd, device_status=st)


def maxsim_backward_named(q_data, q_offsets, d_data, d_offsets, argmax, d_scores, pairs, mean=False, out=None,
                          device_status=None, stream=None):
    """Gradient through the argmax of the named pairs only (`pairs` as for maxsim_scores_named).  Returns
    dict(d_queries, d_documents, device_status)."""
    Q, D = _tape(q_data, q_offsets), _tape(d_data, d_offsets)
    _check_cuda(argmax, "argmax", torch.int32)
    _check_cuda(d_scores, "d_scores", torch.float32)
    width = q_data.shape[1]
    dev = q_data.device
    out = dict(out or {})
    dq = out.get("d_queries") if out.get("d_queries") is not None else torch.empty(Q.rows, width, device=dev)
    dd = out.get("d_documents") if out.get("d_documents") is not None else torch.empty(D.rows, width, device=dev)
    st = device_status if device_status is not None else torch.zeros(1, dtype=torch.int32, device=dev)
    base = MaxSimBackwardArgs(queries=Q, documents=D, width=width, mean=int(bool(mean)), argmax=_ptr(argmax),
                              ld_argmax=argmax.stride(0), d_scores=_ptr(d_scores), ld_d_scores=d_scores.stride(0),
                              d_queries=_ptr(dq), d_documents=_ptr(dd), workspace=None, workspace_bytes=0,
                              device_status=_ptr(st), stream=_stream(stream))
    args = MaxSimBackwardNamedArgs(base=base, pairs=_edges(pairs, Q.count))
    raise_for(lib.maxsim_backward_named(ctypes.byref(args)), "maxsim_backward_named")
    return dict(d_queries=dq, d_documents=dd, device_status=st)
