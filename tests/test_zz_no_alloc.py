"""maxsim_backward_no_alloc: the MaxSim backward for callers that cannot allocate device memory.

Some callers cannot call cudaMalloc (allocation is not allowed where they run, or their device memory is
all reserved by their own allocator), so they cannot lend a workspace either.  This entry point keeps its
one piece of scratch in a fixed device array inside the library.  The GPU tests call it through the C ABI
twice in a row, with different query tapes (and with queries and documents no pair reaches), and check
each result against maxsim_backward (which takes a lent workspace), element for element.  This file is
collected last on purpose.
"""

import ctypes

import numpy as np
import pytest
import torch

from contrastive_late_interaction_gb300 import synth

DD_ROUNDING = 1e-6   # dD of the two entry points: the same sums, bucket entries possibly in another order


def _args(b, q, qo, d, do, am, ds, dq, dd, st, stream, mean=0):
    return b.MaxSimBackwardArgs(
        queries=b.Tape(q.data_ptr(), qo.data_ptr(), qo.numel() - 1, q.shape[0]),
        documents=b.Tape(d.data_ptr(), do.data_ptr(), do.numel() - 1, d.shape[0]),
        width=q.shape[1], mean=mean, argmax=am.data_ptr(), ld_argmax=am.stride(0), d_scores=ds.data_ptr(),
        ld_d_scores=ds.stride(0), d_queries=dq.data_ptr(), d_documents=dd.data_ptr(), workspace=None,
        workspace_bytes=0, device_status=st.data_ptr(), stream=stream)


def test_no_alloc_rejects_query_tapes_beyond_its_scratch():
    from contrastive_late_interaction_gb300 import build
    build.build()
    from contrastive_late_interaction_gb300 import _binding as b
    A = 1 << 32
    rows = b.NO_ALLOC_MAX_QUERY_ROWS + 1
    a = b.MaxSimBackwardArgs(queries=b.Tape(A, 2 * A, 10, rows), documents=b.Tape(3 * A, 4 * A, 10, 100), width=128,
                             mean=0, argmax=5 * A, ld_argmax=rows, d_scores=6 * A, ld_d_scores=10, d_queries=7 * A,
                             d_documents=8 * A, workspace=None, workspace_bytes=0, device_status=9 * A, stream=None)
    assert b.lib.maxsim_backward_no_alloc(ctypes.byref(a)) == b.CLI_UNSUPPORTED


@pytest.mark.gpu
@pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")
def test_no_alloc_matches_the_workspace_entry_point_on_two_calls():
    """Both entry points run the same kernels.  dQ sums each row's terms in document order, so it is equal
    element for element; dD sums each document row's bucket in the order its entries were scattered (slot
    claims by shared-memory atomics, which may differ between runs), so it is equal to rounding: relative
    L2 at most 1e-6, far inside the gradient tolerance."""
    import contrastive_late_interaction_gb300 as cli
    from contrastive_late_interaction_gb300 import _binding as b
    from tests.gpu_util import bf16, i64, rel_l2
    stream = torch.cuda.current_stream()
    for seed, nq, nd, ql, dl in ((11, 70, 40, (3, 60), (5, 300)), (12, 33, 57, (1, 9), (2, 80))):
        m = synth.maxsim_random(seed, nq, nd, 128, ql, dl)
        q, qo, d, do = bf16(m.q_bf16), i64(m.q_offsets), bf16(m.d_bf16), i64(m.d_offsets)
        f = cli.maxsim_scores(q, qo, d, do)
        ds = torch.from_numpy(m.d_scores).cuda()
        ref = cli.maxsim_backward(q, qo, d, do, f["argmax"], ds)
        dq = torch.full_like(ref["d_queries"], 123.0)
        dd = torch.full_like(ref["d_documents"], 123.0)
        st = torch.full((1,), 77, dtype=torch.int32, device="cuda")
        args = _args(b, q, qo, d, do, f["argmax"], ds, dq, dd, st, ctypes.c_void_p(stream.cuda_stream))
        assert b.lib.maxsim_backward_no_alloc(ctypes.byref(args)) == b.CLI_OK
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        assert int(ref["device_status"].item()) == 0
        assert torch.equal(dq, ref["d_queries"])
        assert rel_l2(dd.double().cpu().numpy(), ref["d_documents"].double().cpu().numpy()) <= DD_ROUNDING


@pytest.mark.gpu
@pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")
@pytest.mark.parametrize("mean", [0, 1])
def test_no_alloc_writes_zeros_for_queries_and_documents_no_pair_reaches(mean):
    """dS with whole rows (queries) and columns (documents) zero: the workspace entry point skips them by
    its activity flags, this one (no flags: it has no workspace for them) computes their rows as sums of
    zero terms.  The outputs start as 123.0; every row must be overwritten, the skipped ones with zeros;
    dQ agrees element for element and dD to rounding, as above."""
    import contrastive_late_interaction_gb300 as cli
    from contrastive_late_interaction_gb300 import _binding as b
    from tests.gpu_util import bf16, i64, rel_l2
    stream = torch.cuda.current_stream()
    m = synth.maxsim_random(13, 60, 45, 128, (2, 40), (3, 200))
    dsn = np.array(m.d_scores, dtype=np.float32)
    rng = np.random.default_rng(14)
    dead_q, dead_d = rng.random(m.nq) < 0.3, rng.random(m.nd) < 0.3
    dsn[dead_q, :] = 0.0
    dsn[:, dead_d] = 0.0
    q, qo, d, do = bf16(m.q_bf16), i64(m.q_offsets), bf16(m.d_bf16), i64(m.d_offsets)
    f = cli.maxsim_scores(q, qo, d, do, mean=bool(mean))
    ds = torch.from_numpy(dsn).cuda()
    ref = cli.maxsim_backward(q, qo, d, do, f["argmax"], ds, mean=bool(mean))
    for _ in range(2):
        dq = torch.full_like(ref["d_queries"], 123.0)
        dd = torch.full_like(ref["d_documents"], 123.0)
        st = torch.full((1,), 77, dtype=torch.int32, device="cuda")
        args = _args(b, q, qo, d, do, f["argmax"], ds, dq, dd, st, ctypes.c_void_p(stream.cuda_stream), mean)
        assert b.lib.maxsim_backward_no_alloc(ctypes.byref(args)) == b.CLI_OK
        torch.cuda.synchronize()
        assert int(st.item()) == 0 and int(ref["device_status"].item()) == 0
        assert torch.equal(dq, ref["d_queries"])
        assert rel_l2(dd.double().cpu().numpy(), ref["d_documents"].double().cpu().numpy()) <= DD_ROUNDING
        rq = torch.from_numpy(np.repeat(dead_q, np.diff(m.q_offsets.astype(np.int64)))).cuda()
        rd = torch.from_numpy(np.repeat(dead_d, np.diff(m.d_offsets.astype(np.int64)))).cuda()
        assert bool(torch.all(dq[rq] == 0)) and bool(torch.all(dd[rd] == 0))
