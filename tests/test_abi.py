"""The C ABI without a GPU: the library loads, exports every symbol include/cli.h declares, names its
statuses, and refuses bad arguments on the host before touching the device.

Pointers below are fake, well-aligned addresses: every call here must return before any CUDA call,
so nothing ever dereferences them.
"""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def b():
    from contrastive_late_interaction_gb300 import build
    build.build()
    from contrastive_late_interaction_gb300 import _binding
    return _binding


def declared_functions():
    text = open(os.path.join(ROOT, "include", "cli.h")).read()
    return set(re.findall(r"^\s*(?:const\s+char\s*\*|cli_status_t|size_t)\s*([a-z_]+)\s*\(", text, re.M))


def test_every_declared_symbol_is_exported(b):
    names = declared_functions()
    assert {"pair_loss_sigmoid_fwd_bwd", "maxsim_scores", "maxsim_backward", "cli_status_name"} <= names
    lib = ctypes.CDLL(b.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n
    assert names == set(b.EXPORTS)


def test_selftest_host_checks(b):
    f = b.lib.cli_selftest_bounded_wait
    assert f(None, None, 1000, None) == b.CLI_INVALID_ARGUMENT
    assert f(A * 1, None, 0, None) == b.CLI_INVALID_ARGUMENT
    assert f(A * 1, A * 2, 2000001, None) == b.CLI_INVALID_ARGUMENT


def test_status_names(b):
    assert [b.status_name(i) for i in range(7)] == b.STATUS_NAMES
    assert b.status_name(99) == "unknown"


def test_workspace_sizes_are_positive_and_monotone(b):
    small = b.pair_loss_sigmoid_workspace_bytes(256, 64, 256)
    big = b.pair_loss_sigmoid_workspace_bytes(32768, 768, 98304)
    assert 0 < small < big and big % 256 == 0
    assert b.maxsim_workspace_bytes(512, 512, 18432, 270336, 128) >= 512 * 18432 * 4
    assert b.maxsim_backward_workspace_bytes(512, 512, 18432, 270336, 128) >= 18432 * 4


A = 1 << 32  # fake device addresses, 256-byte aligned, far apart


def edges(off, ids, n):
    return b_mod().Edges(off, ids, None, n)


def b_mod():
    from contrastive_late_interaction_gb300 import _binding
    return _binding


def pooled_args(b, **over):
    n, w = 1024, 512
    ws = b.pair_loss_sigmoid_workspace_bytes(n, w, 2048)
    args = dict(count=n, width=w, ld=w, embeddings=A * 1, inverse_temperature=A * 2, bias=A * 3,
                relations=b.Relations(b.Edges(A * 4, A * 5, None, 2048), b.Edges(None, None, None, 0),
                                      b.Edges(None, None, None, 0), 0, 1.0),
                loss=A * 6, d_embeddings=A * 7, ld_d_embeddings=w, d_inverse_temperature=A * 8, d_bias=A * 9,
                workspace=A * 10, workspace_bytes=ws, device_status=A * 11, stream=None)
    args.update(over)
    return b.PairLossSigmoidArgs(**args)


def call_pooled(b, **over):
    return b.lib.pair_loss_sigmoid_fwd_bwd(ctypes.byref(pooled_args(b, **over)))


def test_pooled_host_checks(b):
    assert b.lib.pair_loss_sigmoid_fwd_bwd(None) == b.CLI_INVALID_ARGUMENT
    assert call_pooled(b, embeddings=None) == b.CLI_INVALID_ARGUMENT
    assert call_pooled(b, device_status=None) == b.CLI_INVALID_ARGUMENT
    assert call_pooled(b, count=1) == b.CLI_SHAPE_MISMATCH
    assert call_pooled(b, width=60, ld=64) == b.CLI_SHAPE_MISMATCH
    assert call_pooled(b, ld=500) == b.CLI_SHAPE_MISMATCH
    assert call_pooled(b, width=4104, ld=4104, ld_d_embeddings=4104) == b.CLI_UNSUPPORTED
    assert call_pooled(b, ld_d_embeddings=510) == b.CLI_SHAPE_MISMATCH
    assert call_pooled(b, embeddings=A + 8) == b.CLI_INVALID_ARGUMENT               # not 16-byte aligned
    assert call_pooled(b, workspace_bytes=1024) == b.CLI_INVALID_ARGUMENT          # workspace too small
    # the anchor band must lie inside the batch; (0, 0) is every row
    assert call_pooled(b, row_begin=1000, row_count=25) == b.CLI_SHAPE_MISMATCH
    assert call_pooled(b, row_begin=2**64 - 1, row_count=2) == b.CLI_SHAPE_MISMATCH
    assert call_pooled(b, row_begin=5, row_count=0) == b.CLI_SHAPE_MISMATCH
    assert call_pooled(b, row_begin=1000, row_count=24, workspace_bytes=1024) == b.CLI_INVALID_ARGUMENT
    assert call_pooled(b, row_begin=0, row_count=0, workspace_bytes=1024) == b.CLI_INVALID_ARGUMENT
    # a step naming no attract edge is refused
    no_attract = b.Relations(b.Edges(None, None, None, 0), b.Edges(A * 4, A * 5, None, 7),
                             b.Edges(None, None, None, 0), 0, 1.0)
    assert call_pooled(b, relations=no_attract) == b.CLI_INVALID_ARGUMENT
    bad_ambient = b.Relations(b.Edges(A * 4, A * 5, None, 2048), b.Edges(None, None, None, 0),
                              b.Edges(None, None, None, 0), 0, -1.0)
    assert call_pooled(b, relations=bad_ambient) == b.CLI_INVALID_ARGUMENT
    # outputs overlapping inputs
    assert call_pooled(b, d_embeddings=A * 1 + 4096) == b.CLI_INVALID_ARGUMENT
    assert call_pooled(b, loss=A * 2) == b.CLI_INVALID_ARGUMENT
    assert call_pooled(b, workspace=A * 7) == b.CLI_INVALID_ARGUMENT   # workspace inside another output


def maxsim_args(b, **over):
    rq, rd, nq, nd, w = 4096, 65536, 100, 200, 128
    ws = b.maxsim_workspace_bytes(nq, nd, rq, rd, w)
    args = dict(queries=b.Tape(A * 1, A * 2, nq, rq), documents=b.Tape(A * 3, A * 4, nd, rd), width=w, mean=0,
                scores=A * 5, ld_scores=nd, argmax=A * 6, ld_argmax=rq, workspace=A * 8, workspace_bytes=ws,
                device_status=A * 9, stream=None)
    args.update(over)
    return b.MaxSimArgs(**args)


def test_maxsim_host_checks(b):
    f = lambda **o: b.lib.maxsim_scores(ctypes.byref(maxsim_args(b, **o)))
    assert b.lib.maxsim_scores(None) == b.CLI_INVALID_ARGUMENT
    assert f(width=12) == b.CLI_SHAPE_MISMATCH
    assert f(width=264) == b.CLI_UNSUPPORTED
    assert f(ld_scores=10) == b.CLI_SHAPE_MISMATCH
    assert f(ld_argmax=100) == b.CLI_SHAPE_MISMATCH
    assert f(queries=b.Tape(A * 1, A * 2, 100, 50)) == b.CLI_INVALID_ARGUMENT    # fewer rows than items
    assert f(queries=b.Tape(A * 1 + 2, A * 2, 100, 4096)) == b.CLI_INVALID_ARGUMENT  # misaligned data
    assert f(workspace_bytes=4096) == b.CLI_INVALID_ARGUMENT
    assert f(scores=A * 3 + 64) == b.CLI_INVALID_ARGUMENT       # scores inside the document tape
    assert f(argmax=A * 5) == b.CLI_INVALID_ARGUMENT            # two outputs overlap


def test_maxsim_backward_host_checks(b):
    rq, rd, nq, nd, w = 4096, 65536, 100, 200, 128
    base = dict(queries=b.Tape(A * 1, A * 2, nq, rq), documents=b.Tape(A * 3, A * 4, nd, rd), width=w, mean=0,
                argmax=A * 5, ld_argmax=rq, d_scores=A * 6, ld_d_scores=nd, d_queries=A * 7, d_documents=A * 8,
                workspace=A * 9, workspace_bytes=b.maxsim_backward_workspace_bytes(nq, nd, rq, rd, w),
                device_status=A * 10, stream=None)

    def f(**o):
        a = dict(base)
        a.update(o)
        return b.lib.maxsim_backward(ctypes.byref(b.MaxSimBackwardArgs(**a)))

    assert f(d_queries=None) == b.CLI_INVALID_ARGUMENT
    assert f(ld_d_scores=3) == b.CLI_SHAPE_MISMATCH
    assert f(d_documents=A * 5) == b.CLI_INVALID_ARGUMENT      # output over the argmax input
    assert f(d_queries=A * 7 + 4) == b.CLI_INVALID_ARGUMENT    # misaligned


def test_score_loss_host_checks(b):
    r = c = 64
    base = dict(rows=r, cols=c, ld=c, scores=A * 1, inverse_temperature=A * 2, bias=A * 3,
                relations=b.Relations(b.Edges(A * 4, A * 5, None, 64), b.Edges(None, None, None, 0),
                                      b.Edges(None, None, None, 0), 0, 1.0),
                sides=None, loss=A * 6, d_scores=A * 7, ld_d_scores=c, d_inverse_temperature=A * 8, d_bias=A * 9,
                workspace=A * 10, workspace_bytes=b.pair_loss_sigmoid_scores_workspace_bytes(r, c),
                device_status=A * 11, stream=None)

    def f(**o):
        a = dict(base)
        a.update(o)
        return b.lib.pair_loss_sigmoid_scores_fwd_bwd(ctypes.byref(b.PairLossSigmoidScoresArgs(**a)))

    assert f(rows=0) == b.CLI_SHAPE_MISMATCH
    assert f(ld=10) == b.CLI_SHAPE_MISMATCH
    assert f(cols=32, ld=32, ld_d_scores=32, sides=A * 12) == b.CLI_SHAPE_MISMATCH   # sides need a square matrix
    assert f(d_scores=A * 1) == b.CLI_INVALID_ARGUMENT
    assert f(workspace_bytes=0) == b.CLI_INVALID_ARGUMENT


def test_matryoshka_host_checks(b):
    n, w = 1024, 512
    ws = b.pair_loss_sigmoid_matryoshka_workspace_bytes(n, w, 2048)
    assert ws > b.pair_loss_sigmoid_workspace_bytes(n, w, 2048)

    def f(widths, count=None, prefix_loss=A * 12, **over):
        arr = (ctypes.c_size_t * max(1, len(widths)))(*widths) if widths is not None else None
        args = b.PairLossMatryoshkaArgs(base=pooled_args(b, **{"workspace_bytes": ws, **over}),
                                        prefix_widths=ctypes.cast(arr, ctypes.c_void_p) if arr is not None else None,
                                        prefix_count=len(widths) if count is None else count,
                                        prefix_loss=prefix_loss)
        return b.lib.pair_loss_sigmoid_matryoshka_fwd_bwd(ctypes.byref(args))

    assert b.lib.pair_loss_sigmoid_matryoshka_fwd_bwd(None) == b.CLI_INVALID_ARGUMENT
    assert f(None, count=1) == b.CLI_INVALID_ARGUMENT                     # no prefix list
    assert f([64], count=0) == b.CLI_SHAPE_MISMATCH
    assert f([8 * (k + 1) for k in range(9)]) == b.CLI_SHAPE_MISMATCH    # more than eight prefixes
    assert f([64, 64]) == b.CLI_SHAPE_MISMATCH                           # not strictly ascending
    assert f([128, 64]) == b.CLI_SHAPE_MISMATCH
    assert f([60, 128]) == b.CLI_SHAPE_MISMATCH                          # not a multiple of 8
    assert f([64, 520]) == b.CLI_SHAPE_MISMATCH                          # past the width
    assert f([64], workspace_bytes=b.pair_loss_sigmoid_workspace_bytes(n, w, 2048)) == b.CLI_INVALID_ARGUMENT
    assert f([64], prefix_loss=A * 1) == b.CLI_INVALID_ARGUMENT          # an output inside the embeddings
    assert f([64], embeddings=None) == b.CLI_INVALID_ARGUMENT            # the pooled checks still apply


def test_groups_host_checks(b):
    n, w = 1024, 512

    def f(groups=A * 13, count=3, **over):
        args = b.PairLossGroupsArgs(base=pooled_args(b, **over), groups=groups, group_count=count)
        return b.lib.pair_loss_sigmoid_groups_fwd_bwd(ctypes.byref(args))

    assert b.lib.pair_loss_sigmoid_groups_fwd_bwd(None) == b.CLI_INVALID_ARGUMENT
    assert f(groups=None) == b.CLI_INVALID_ARGUMENT
    assert f(groups=A * 13 + 2) == b.CLI_INVALID_ARGUMENT                # not 4-byte aligned
    assert f(count=0) == b.CLI_SHAPE_MISMATCH
    assert f(groups=A * 7) == b.CLI_INVALID_ARGUMENT                     # an input inside the dE output
    assert f(count=3, d_bias=A * 8 + 8) == b.CLI_INVALID_ARGUMENT        # d_bias [3] overlaps d_inverse_temperature [3]
    assert f(count=3, embeddings=None) == b.CLI_INVALID_ARGUMENT         # the pooled checks still apply


def test_maxsim_named_host_checks(b):
    rq, rd, nq, nd, w = 4096, 65536, 100, 200, 128
    ws = b.maxsim_named_workspace_bytes(nq, nd, rq, rd, w)
    assert ws > b.maxsim_workspace_bytes(nq, nd, rq, rd, w)

    def f(pairs=None, **o):
        pairs = pairs if pairs is not None else b.Edges(A * 10, A * 11, None, 800)
        args = b.MaxSimNamedArgs(base=maxsim_args(b, **{"workspace_bytes": ws, **o}), pairs=pairs)
        return b.lib.maxsim_scores_named(ctypes.byref(args))

    assert b.lib.maxsim_scores_named(None) == b.CLI_INVALID_ARGUMENT
    assert f(pairs=b.Edges(None, None, None, 0)) == b.CLI_INVALID_ARGUMENT          # no pair list
    assert f(pairs=b.Edges(A * 10, None, None, 800)) == b.CLI_INVALID_ARGUMENT      # ids missing
    assert f(workspace_bytes=b.maxsim_workspace_bytes(nq, nd, rq, rd, w)) == b.CLI_INVALID_ARGUMENT
    assert f(pairs=b.Edges(A * 5, A * 11, None, 800)) == b.CLI_INVALID_ARGUMENT     # offsets inside the scores
    assert f(width=12) == b.CLI_SHAPE_MISMATCH                                        # the plain checks still apply


def test_maxsim_backward_named_host_checks(b):
    rq, rd, nq, nd, w = 4096, 65536, 100, 200, 128

    def f(pairs=None, **o):
        pairs = pairs if pairs is not None else b.Edges(A * 10, A * 11, None, 800)
        args = dict(queries=b.Tape(A * 1, A * 2, nq, rq), documents=b.Tape(A * 3, A * 4, nd, rd), width=w, mean=0,
                    argmax=A * 5, ld_argmax=rq, d_scores=A * 6, ld_d_scores=nd, d_queries=A * 7, d_documents=A * 8,
                    workspace=None, workspace_bytes=0, device_status=A * 9, stream=None)
        args.update(o)
        named = b.MaxSimBackwardNamedArgs(base=b.MaxSimBackwardArgs(**args), pairs=pairs)
        return b.lib.maxsim_backward_named(ctypes.byref(named))

    assert b.lib.maxsim_backward_named(None) == b.CLI_INVALID_ARGUMENT
    assert f(pairs=b.Edges(None, None, None, 0)) == b.CLI_INVALID_ARGUMENT
    assert f(d_queries=A * 7 + 4) == b.CLI_INVALID_ARGUMENT                       # misaligned output
    assert f(pairs=b.Edges(A * 7, A * 11, None, 800)) == b.CLI_INVALID_ARGUMENT    # pair offsets inside dQ
    assert f(width=264) == b.CLI_UNSUPPORTED
