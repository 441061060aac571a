"""Writes config1_oracle.json: the float64 oracle's outputs on the tiny configuration (seed 0).

Run from the repository root:  python tests/golden/make_golden.py

The stored values come from `oracle/` alone (the inputs from the seeded generators in
`contrastive_late_interaction_gb300/synth.py`, which hold none of the method's arithmetic).  They pin the
oracle against later edits of its own arithmetic: `tests/test_golden.py` recomputes them and compares.
A change to this file goes with a commit message that names the passage, or the reading of it, that
justifies the new values.
"""
import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from contrastive_late_interaction_gb300 import synth  # noqa: E402

# dE rows and MaxSim query rows / document rows stored in full (the rest enter through sums).
POOLED_ROWS = (0, 1, 2, 127, 255)
MAXSIM_Q_ROWS = (0, 7, 64, 127)
MAXSIM_D_ROWS = (0, 31, 256, 511)


def compute():
    p = synth.pooled_tiny()
    r = oracle.pair_loss_sigmoid(p.e_rounded, p.t, p.b, p.attract)
    de = np.asarray(r["de"], dtype=np.float64)
    m = synth.maxsim_tiny()
    out = {"pooled": {"loss": float(r["loss"]), "dt": float(r["dt"]), "db": float(r["db"]),
                      "de_sum": float(de.sum()), "de_sum_sq": float((de * de).sum()),
                      "de_rows": {str(i): de[i].tolist() for i in POOLED_ROWS}},
           "maxsim": {}}
    for mean in (False, True):
        s, arg, _ = oracle.maxsim_forward(m.q_offsets, m.q, m.d_offsets, m.d, mean)
        dq, dd = oracle.maxsim_backward(m.q_offsets, m.q, m.d_offsets, m.d, arg, m.d_scores, mean)
        part = out["maxsim"]["mean" if mean else "sum"] = {
            "scores": np.asarray(s, dtype=np.float64).tolist(),
            "dq_sum_sq": float((dq * dq).sum()), "dd_sum_sq": float((dd * dd).sum()),
            "dq_rows": {str(i): dq[i].tolist() for i in MAXSIM_Q_ROWS},
            "dd_rows": {str(i): dd[i].tolist() for i in MAXSIM_D_ROWS}}
        if not mean:   # the argmax is the same with the mean (1/|q| scales a query's scores only)
            part["argmax"] = np.asarray(arg).astype(int).tolist()
    return out


if __name__ == "__main__":
    with open(os.path.join(HERE, "config1_oracle.json"), "w") as f:
        json.dump(compute(), f, separators=(",", ":"))
        f.write("\n")
