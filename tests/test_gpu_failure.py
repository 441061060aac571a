"""Failure detection on the GPU without a fault.

Every wait of the tensor-core kernels is bounded: a wait that runs out writes CLI_INTERNAL to the device
status, the CTA's other waiters give up, and the kernel returns.  `cli_selftest_bounded_wait` makes one
such wait run out (a barrier nothing arrives at, a 20 ms limit); the status must say so, every waiting
thread must have given up, and the next call on the stream must run normally.
"""

import time

import numpy as np
import pytest
import torch

import oracle
from contrastive_late_interaction_gb300 import synth
from tests.gpu_util import check_scores, run_maxsim

pytestmark = pytest.mark.gpu


def test_a_wait_that_runs_out_reports_and_the_context_stays_usable():
    import contrastive_late_interaction_gb300 as cli
    from contrastive_late_interaction_gb300._binding import CLI_INTERNAL
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    r = cli.selftest_bounded_wait(limit_us=20000)
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert int(r["device_status"].item()) == CLI_INTERNAL
    assert int(r["gave_up"].item()) == 64
    assert 0.02 <= elapsed < 5.0, elapsed
    m = synth.maxsim_tiny()
    g = run_maxsim(m)
    assert g["status_f"] == 0 and g["status_b"] == 0
    s, _, _ = oracle.maxsim_forward(m.q_offsets, m.q, m.d_offsets, m.d)
    check_scores(g["scores"], s)
