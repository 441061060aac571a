#!/usr/bin/env python
"""Benchmark of the in-batch contrastive scoring path on GB300.

One step = the whole hot path over one synthetic batch shaped like the joint
step: the pooled sigmoid pair loss forward+backward (N=16384, D=512, bags of
1-4, ambient repel, t=10, b=-10), hard MaxSim forward over 2048 x 2048 items
(D=128, query runs U{16..48} copied from their documents' runs U{64..512}),
the sigmoid loss over the MaxSim score matrix (t=1, b=0, attract (i,i), sides
1/3 each) and the MaxSim backward -- four C-ABI calls on one stream.

Prints one JSON line (rank 0).  `value` is the whole job's algorithmic
TFLOP/s (3N^2D for the pooled loss, 2*D*rowsQ*rowsD + 4*D*rowsQ*docs for
MaxSim), summed over ranks with the slowest rank's time; the pooled pairs/s
and the MaxSim TFLOP/s are under `parts`.  `--impl reference` times the
float64 CPU oracle on bounded samples of the same workload instead.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = "sigmoid pair-loss pairs/s & MaxSim TFLOP/s fwd+bwd, % of GB300 BF16 TC peak"
L2_FLUSH_BYTES = 256 << 20


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=["joint", "pooled2", "maxsim3", "pooled4", "matryoshka5", "groups5", "named5"], default="joint")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="CPU work budget of the oracle baseline")
    ap.add_argument("--no-extra-parts", action="store_true",
                    help="with the joint workload, skip the separately timed config-4 pooled and config-3 MaxSim calls")
    return ap.parse_args()


# ---------------------------------------------------------------------------
# workload description and algorithmic work
# ---------------------------------------------------------------------------

def make_workload(name: str, seed: int):
    from contrastive_late_interaction_gb300 import synth
    if name == "joint":
        j = synth.joint_config5(seed)
        return dict(pooled=j.pooled, maxsim=j.maxsim, joint=j, prefixes=None)
    if name == "pooled2":
        return dict(pooled=synth.pooled_config2(seed), maxsim=None, joint=None, prefixes=None)
    if name == "pooled4":
        return dict(pooled=synth.pooled_config4(seed), maxsim=None, joint=None, prefixes=None)
    if name == "maxsim3":
        return dict(pooled=None, maxsim=synth.maxsim_config3(seed), joint=None, prefixes=None)
    if name == "matryoshka5":
        # the joint step's pooled batch scored at the nested prefixes {64, 128, 256, 512}
        return dict(pooled=synth.joint_config5(seed).pooled, maxsim=None, joint=None, prefixes=[64, 128, 256, 512])
    if name == "named5":
        # the joint step's MaxSim tapes, each query naming its own document and seven others
        j = synth.joint_config5(seed)
        att, rep = synth.named_documents(seed, j.maxsim.nq, j.maxsim.nd, 7)
        return dict(pooled=None, maxsim=j.maxsim, joint=None, prefixes=None, named=(att, rep))
    if name == "groups5":
        # the joint step's pooled batch with four temperature groups drawn uniformly per item
        p = synth.joint_config5(seed).pooled
        g = synth.uniform_int(seed, synth.STREAM_GROUPS, p.count, 0, 3).astype(np.int32)
        return dict(pooled=p, maxsim=None, joint=None, prefixes=None,
                    groups=(g, np.array([10.0, 8.0, 12.0, 6.0], np.float32), np.array([-10.0, -8.0, -12.0, -6.0], np.float32)))
    raise ValueError(name)


def pooled_flops(p, prefixes=None):
    """3 N^2 D per scored width (S by symmetry plus the two gradient contractions)."""
    return sum(3.0 * p.count * p.count * w for w in (prefixes or [p.width]))


def _named_pairs(m, named):
    """(query, document) index arrays of the named pairs."""
    q = np.concatenate([np.repeat(np.arange(m.nq), np.diff(e.offsets).astype(np.int64)) for e in named])
    d = np.concatenate([e.ids.astype(np.int64) for e in named])
    return q, d


def maxsim_fwd_flops(m, named=None):
    """2 D |q| |d| per scored (query, document) pair: every pair, or the named ones."""
    if named is None:
        return 2.0 * m.width * float(m.q_offsets[-1]) * float(m.d_offsets[-1])
    q, d = _named_pairs(m, named)
    return float(np.sum(2.0 * m.width * np.diff(m.q_offsets)[q].astype(np.float64) *
                        np.diff(m.d_offsets)[d].astype(np.float64)))


def maxsim_bwd_flops(m, named=None):
    """4 D |q| per scored pair (one gathered row each for dQ and dD, times c)."""
    if named is None:
        return 4.0 * m.width * float(m.q_offsets[-1]) * m.nd
    q, _ = _named_pairs(m, named)
    return float(np.sum(4.0 * m.width * np.diff(m.q_offsets)[q].astype(np.float64)))


def describe(name, w):
    cfg = {"workload": {"joint": "joint contrastive step (config 5)", "pooled2": "pooled sigmoid loss (config 2)",
                        "pooled4": "large pooled sigmoid loss (config 4)",
                        "maxsim3": "MaxSim fwd+bwd (config 3)",
                        "matryoshka5": "Matryoshka prefixes of the pooled sigmoid loss (config 5 pooled batch)",
                        "groups5": "pooled sigmoid loss with four temperature groups (config 5 pooled batch)",
                        "named5": "MaxSim fwd+bwd over named pairs (config 5 tapes, own document + 7 named)"}[name]}
    p, m = w["pooled"], w["maxsim"]
    if p is not None:
        cfg["pooled"] = {"N": p.count, "D": p.width, "t": p.t, "b": p.b,
                         "attract_edges": int(p.attract.ids.size), "ignore_edges": int(p.ignore.ids.size),
                         "negatives": "named" if p.negatives_named else "ambient"}
        if w.get("prefixes"):
            cfg["pooled"]["prefixes"] = list(w["prefixes"])
        if w.get("groups"):
            cfg["pooled"]["groups"] = {"count": int(len(w["groups"][1])), "t": w["groups"][1].tolist(),
                                       "b": w["groups"][2].tolist(), "selection": "uniform per item"}
    if m is not None:
        cfg["maxsim"] = {"queries": m.nq, "documents": m.nd, "D": m.width, "query_rows": int(m.q_offsets[-1]),
                         "document_rows": int(m.d_offsets[-1]), "form": "mean" if m.mean else "sum"}
        if w.get("named"):
            cfg["maxsim"]["named_pairs"] = int(w["named"][0].ids.size + w["named"][1].ids.size)
            cfg["score_loss"] = {"t": 1.0, "b": 0.0, "attract": "own document", "repel": "7 named documents",
                                 "negatives": "named"}
    if w["joint"] is not None:
        cfg["score_loss"] = {"t": w["joint"].score_t, "b": w["joint"].score_b, "attract": "(i, i)",
                             "sides": "query/document/both, 1/3 each"}
    return cfg


# ---------------------------------------------------------------------------
# GPU step through the C ABI
# ---------------------------------------------------------------------------

class Step:
    """Device buffers of one workload and the step that runs the four C-ABI calls on one stream."""

    def __init__(self, w, device, stream):
        import torch
        import contrastive_late_interaction_gb300 as cli
        self.cli, self.torch, self.stream, self.dev = cli, torch, stream, device
        self.w = w
        self.p, self.m, self.j = w["pooled"], w["maxsim"], w["joint"]
        self.prefixes = w.get("prefixes")
        self.groups = w.get("groups")
        self.named = w.get("named")
        self.host = {}      # pinned host copies for the end-to-end measurement
        self.dev_in = {}
        with torch.cuda.stream(stream):
            self._setup()

    def _pin(self, name, arr, dtype=None):
        torch = self.torch
        a = np.ascontiguousarray(arr)
        t = torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else
                             (a.view(np.int64) if a.dtype == np.uint64 else
                              (a.view(np.int32) if a.dtype == np.uint32 else a))).pin_memory()
        if dtype is not None:
            t = t.view(dtype)
        self.host[name] = t
        d = torch.empty_like(t, device=self.dev)
        d.copy_(t, non_blocking=True)
        self.dev_in[name] = d
        return d

    def _setup(self):
        torch, cli = self.torch, self.cli
        f32 = dict(dtype=torch.float32, device=self.dev)
        if self.p is not None:
            p = self.p
            self.e = self._pin("e", p.e_bf16, torch.bfloat16)
            if self.groups:
                self.grp = self._pin("groups", self.groups[0])
                self.t = self._pin("t", self.groups[1])
                self.b = self._pin("b", self.groups[2])
            else:
                self.t = self._pin("t", np.array([p.t], np.float32))
                self.b = self._pin("b", np.array([p.b], np.float32))
            self.att = (self._pin("att_off", p.attract.offsets), self._pin("att_ids", p.attract.ids))
            self.ign = ((self._pin("ign_off", p.ignore.offsets), self._pin("ign_ids", p.ignore.ids))
                        if p.ignore.ids.size else None)
            edges = int(p.attract.ids.size + p.ignore.ids.size)
            sizer = (cli.pair_loss_sigmoid_matryoshka_workspace_bytes if self.prefixes else
                     cli.pair_loss_sigmoid_workspace_bytes)
            self.p_ws = torch.empty(sizer(p.count, p.width, edges), dtype=torch.uint8, device=self.dev)
            ng = len(self.groups[1]) if self.groups else 1
            self.p_out = dict(loss=torch.empty(1, **f32), d_embeddings=torch.empty(p.count, p.width, **f32),
                              d_inverse_temperature=torch.empty(ng, **f32), d_bias=torch.empty(ng, **f32))
            if self.prefixes:
                self.p_out["prefix_loss"] = torch.empty(len(self.prefixes), **f32)
            self.p_st = torch.zeros(1, dtype=torch.int32, device=self.dev)
        if self.m is not None:
            m = self.m
            rq, rd = int(m.q_offsets[-1]), int(m.d_offsets[-1])
            self.q = self._pin("q", m.q_bf16, torch.bfloat16)
            self.qo = self._pin("qo", m.q_offsets)
            self.d = self._pin("d", m.d_bf16, torch.bfloat16)
            self.do = self._pin("do", m.d_offsets)
            self.f_ws = torch.empty(cli.maxsim_workspace_bytes(m.nq, m.nd, rq, rd, m.width), dtype=torch.uint8,
                                    device=self.dev)
            self.b_ws = torch.empty(cli.maxsim_backward_workspace_bytes(m.nq, m.nd, rq, rd, m.width),
                                    dtype=torch.uint8, device=self.dev)
            self.f_out = dict(scores=torch.empty(m.nq, m.nd, **f32),
                              argmax=torch.empty(m.nd, rq, dtype=torch.int32, device=self.dev))
            self.b_out = dict(d_queries=torch.empty(rq, m.width, **f32), d_documents=torch.empty(rd, m.width, **f32))
            self.f_st = torch.zeros(1, dtype=torch.int32, device=self.dev)
            self.b_st = torch.zeros(1, dtype=torch.int32, device=self.dev)
            if self.j is not None:
                j = self.j
                self.sides = self._pin("sides", j.sides)
                self.diag = (self._pin("diag_off", j.score_attract.offsets), self._pin("diag_ids", j.score_attract.ids))
                self.st_ = self._pin("st", np.array([j.score_t], np.float32))
                self.sb_ = self._pin("sb", np.array([j.score_b], np.float32))
                self.s_ws = torch.empty(cli.pair_loss_sigmoid_scores_workspace_bytes(m.nq, m.nd), dtype=torch.uint8,
                                        device=self.dev)
                self.s_out = dict(loss=torch.empty(1, **f32), d_scores=torch.empty(m.nq, m.nd, **f32),
                                  d_inverse_temperature=torch.empty(1, **f32), d_bias=torch.empty(1, **f32))
                self.s_st = torch.zeros(1, dtype=torch.int32, device=self.dev)
            elif self.named:
                att, rep = self.named
                lists = [sorted(att.ids[att.offsets[q]:att.offsets[q + 1]].tolist() +
                                rep.ids[rep.offsets[q]:rep.offsets[q + 1]].tolist()) for q in range(m.nq)]
                from contrastive_late_interaction_gb300 import synth
                pairs = synth.edges_from_lists(lists)
                self.pairs = (self._pin("pair_off", pairs.offsets), self._pin("pair_ids", pairs.ids))
                self.n_att = (self._pin("natt_off", att.offsets), self._pin("natt_ids", att.ids))
                self.n_rep = (self._pin("nrep_off", rep.offsets), self._pin("nrep_ids", rep.ids))
                self.st_ = self._pin("st", np.array([1.0], np.float32))
                self.sb_ = self._pin("sb", np.array([0.0], np.float32))
                self.f_ws = torch.empty(cli.maxsim_named_workspace_bytes(m.nq, m.nd, rq, rd, m.width),
                                        dtype=torch.uint8, device=self.dev)
                self.s_ws = torch.empty(cli.pair_loss_sigmoid_scores_workspace_bytes(m.nq, m.nd), dtype=torch.uint8,
                                        device=self.dev)
                self.s_out = dict(loss=torch.empty(1, **f32), d_scores=torch.empty(m.nq, m.nd, **f32),
                                  d_inverse_temperature=torch.empty(1, **f32), d_bias=torch.empty(1, **f32))
                self.s_st = torch.zeros(1, dtype=torch.int32, device=self.dev)
            else:
                self.ds = self._pin("ds", m.d_scores)

    def launches_per_step(self):
        """Kernels of this library one step launches (mirrors the launch code of csrc/)."""
        n = 0
        if self.p is not None:
            sets = 1 + (1 if self.ign is not None else 0)
            n += sets                                     # edge validation, one per edge set given
            n += 1 + sets + 1 + 1 + 1                     # in-degree, a scan per set, fill, sort, merge
            if self.groups:
                n += 1 + 3                                # group validation, fused block kernel, final reduction
            elif self.prefixes:                           # per prefix: normalise, fused, 2 reductions, gradient
                n += 5 * len(self.prefixes) + 1           # and the sum over prefixes
            else:
                n += 3                                    # fused block kernel, two-level final reduction
        if self.m is not None:
            n += 2 + 1 + 1 + 1 + 1                        # 2 tape validations, schedule, forward, query sums, fix-up
            if not self.named:
                n += 2 + 1 + 1 + 1 + 1                    # 2 tape validations, activity flags and row->query map,
                                                          # active-document list, dQ, dD
            if self.named:
                n += 2 + 1 + 1                            # 2 tape validations, pair validation, named backward
                n += 1 + 1 + 1                            # pair validation, item marks, compaction
                n += 2 + 1 + 1                            # 2 edge validations, score loss, final reduction
            if self.j is not None:
                n += 1 + 1 + 1                            # edge validation, score loss, final reduction
        return n

    def run(self, events=None):
        """One step.  events: optional dict name -> (start, end) CUDA events recorded around each call."""
        cli = self.cli

        def rec(name, k):
            if events is not None:
                events[name][k].record(self.stream)

        with self.torch.cuda.stream(self.stream):
            if self.p is not None:
                rec("pooled", 0)
                if self.groups:
                    cli.pair_loss_sigmoid_groups_fwd_bwd(self.e, self.grp, self.t, self.b, self.att, None, self.ign,
                                                         out=self.p_out, workspace=self.p_ws, device_status=self.p_st,
                                                         stream=self.stream)
                elif self.prefixes:
                    cli.pair_loss_sigmoid_matryoshka_fwd_bwd(self.e, self.prefixes, self.t, self.b, self.att, None,
                                                             self.ign, out=self.p_out, workspace=self.p_ws,
                                                             device_status=self.p_st, stream=self.stream)
                else:
                    cli.pair_loss_sigmoid_fwd_bwd(self.e, self.t, self.b, self.att, None, self.ign, out=self.p_out,
                                                  workspace=self.p_ws, device_status=self.p_st, stream=self.stream)
                rec("pooled", 1)
            if self.m is not None:
                rec("maxsim_fwd", 0)
                if self.named:
                    f = cli.maxsim_scores_named(self.q, self.qo, self.d, self.do, self.pairs, out=self.f_out,
                                                workspace=self.f_ws, device_status=self.f_st, stream=self.stream)
                else:
                    f = cli.maxsim_scores(self.q, self.qo, self.d, self.do, out=self.f_out, workspace=self.f_ws,
                                          device_status=self.f_st, stream=self.stream)
                rec("maxsim_fwd", 1)
                if self.named:
                    rec("score_loss", 0)
                    s = cli.pair_loss_sigmoid_scores_fwd_bwd(f["scores"], self.st_, self.sb_, self.n_att, self.n_rep,
                                                             negatives_named=True, out=self.s_out, workspace=self.s_ws,
                                                             device_status=self.s_st, stream=self.stream)
                    rec("score_loss", 1)
                    ds = s["d_scores"]
                elif self.j is not None:
                    rec("score_loss", 0)
                    s = cli.pair_loss_sigmoid_scores_fwd_bwd(f["scores"], self.st_, self.sb_, self.diag,
                                                             sides=self.sides, out=self.s_out, workspace=self.s_ws,
                                                             device_status=self.s_st, stream=self.stream)
                    rec("score_loss", 1)
                    ds = s["d_scores"]
                else:
                    ds = self.ds
                rec("maxsim_bwd", 0)
                if self.named:
                    cli.maxsim_backward_named(self.q, self.qo, self.d, self.do, f["argmax"], ds, self.pairs,
                                              out=self.b_out, device_status=self.b_st, stream=self.stream)
                else:
                    cli.maxsim_backward(self.q, self.qo, self.d, self.do, f["argmax"], ds, out=self.b_out,
                                        workspace=self.b_ws, device_status=self.b_st, stream=self.stream)
                rec("maxsim_bwd", 1)

    def upload(self, stream=None):
        """Host -> device copies of every input of a step (pinned memory; the step's stream, or `stream`)."""
        with self.torch.cuda.stream(stream if stream is not None else self.stream):
            for k, h in self.host.items():
                self.dev_in[k].copy_(h, non_blocking=True)
        return sum(h.numel() * h.element_size() for h in self.host.values())

    def results(self):
        """The step's results a caller reads back: the losses and their scalar gradients, dE, the MaxSim
        score matrix, dQ and dD (the argmax and dS are intermediates the backward consumes on the device)."""
        outs = []
        if self.p is not None:
            outs += [self.p_out["loss"], self.p_out["d_inverse_temperature"], self.p_out["d_bias"],
                     self.p_out["d_embeddings"]]
        if self.m is not None:
            outs += [self.f_out["scores"], self.b_out["d_queries"], self.b_out["d_documents"]]
        if self.j is not None or self.named:
            outs += [self.s_out["loss"], self.s_out["d_inverse_temperature"], self.s_out["d_bias"]]
        return outs

    def active_pairs(self):
        """(query row, document) pairs whose c = dS[q, d] is nonzero, read from the step's dS on the device
        (every pair without a score loss and with the random dS)."""
        m = self.m
        if self.j is not None or self.named:
            ds = self.s_out["d_scores"]
        else:
            ds = self.ds
        nz = (ds != 0).sum(dim=1).double().cpu().numpy()
        ql = np.diff(m.q_offsets.astype(np.int64)).astype(np.float64)
        return float(np.sum(nz * ql))

    def statuses(self):
        st = []
        for name in ("p_st", "f_st", "s_st", "b_st"):
            if hasattr(self, name):
                st.append(int(getattr(self, name).item()))
        return st


# ---------------------------------------------------------------------------
# clocks
# ---------------------------------------------------------------------------

class ClockSampler:
    """nvidia-smi sampling every 50 ms on a reader thread that stamps each line on arrival.  Entering
    waits (up to 5 s) for the first line, so the sampler is running before the timed region starts;
    mark() brackets the region, and summary() keeps the lines that arrived inside it (plus one
    interval), or the nearest line after it if none did."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    INTERVAL_S = 0.05

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.stamped = []
        self.lines = []
        self.t0 = self.t1 = None
        self.thread = None

    def _read(self):
        for ln in self.proc.stdout:
            if ln.strip():
                self.stamped.append((time.monotonic(), ln))

    def __enter__(self):
        import threading
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", str(int(self.INTERVAL_S * 1000))],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return self
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        deadline = time.monotonic() + 5.0
        while not self.stamped and time.monotonic() < deadline and self.proc.poll() is None:
            time.sleep(0.01)
        return self

    def mark(self, start: bool):
        if start:
            self.t0 = time.monotonic()
        else:
            self.t1 = time.monotonic()
            time.sleep(2 * self.INTERVAL_S)   # let the last in-region sample arrive

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.proc.wait()
            if self.thread is not None:
                self.thread.join(timeout=5)
        lines = list(self.stamped)
        if self.t0 is not None and self.t1 is not None:
            inside = [ln for t, ln in lines if self.t0 <= t <= self.t1 + self.INTERVAL_S]
            if not inside:
                after = [ln for t, ln in lines if t >= self.t0]
                inside = after[:1]
            lines = [(0.0, ln) for ln in inside]
        self.lines = [ln for _, ln in lines]

    def summary(self):
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
                power.append(float(f[3]))
            except ValueError:
                continue
            for nm, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm), "power_w_max": max(power)}


# ---------------------------------------------------------------------------
# peaks, committed ncu traffic
# ---------------------------------------------------------------------------

def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d.get("bf16_tflops", 1900.0), d.get("bf16_tflops_sustained", 1700.0), d.get("hbm_gbs", 6800.0), "measured"
    return 1900.0, 1700.0, 6800.0, "fallback"


# Committed DRAM-traffic records: file under profiles/ -> the kernel sources its counters were taken on.
TRAFFIC_RECORDS = {
    "maxsim": ("maxsim_forward_traffic.json", ("maxsim.cu", "cli_device.cuh", "compact.cuh")),
    "pooled": ("pooled_fused_traffic.json", ("pair_loss.cu", "cli_device.cuh")),
}


def kernel_source_hash(files=TRAFFIC_RECORDS["maxsim"][1]):
    h = hashlib.sha256()
    for name in files:
        with open(os.path.join(ROOT, "contrastive_late_interaction_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def committed_traffic(workload, kind="maxsim"):
    """DRAM bytes per launch of the roofline kernel (the MaxSim forward tile kernel, or the pooled fused block
    kernel) from the committed ncu summary, if it was taken on the current kernel source; else None."""
    record, files = TRAFFIC_RECORDS[kind]
    path = os.path.join(ROOT, "profiles", record)
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    if d.get("source_hash") != kernel_source_hash(files):
        return None
    return d.get("per_launch_bytes", {}).get(workload)


# ---------------------------------------------------------------------------
# CPU oracle baseline (bounded sample)
# ---------------------------------------------------------------------------

def oracle_sample(w, budget_s: float, threads: int):
    """Times the float64 oracle on a bounded sample of the workload: the first R anchors of the pooled loss
    (each anchor's row is 3*N*D algorithmic flops) and P (query, document) pairs of MaxSim (2*D*|q|*|d|
    each, plus the backward share 4*D*|q| per pair).  Returns (flops, seconds, description)."""
    import oracle
    oracle.build()
    p, m = w["pooled"], w["maxsim"]
    parts = (p is not None) + (m is not None)
    flops = secs = 0.0
    desc = []
    if p is not None:
        pre = w.get("prefixes")
        if pre:   # the oracle's normalised, bf16-rounded prefixes, as its Matryoshka function scores them
            ee = []
            for q in pre:
                x = p.e_rounded[:, :q]
                ee.append(oracle.round_bf16(x / np.linalg.norm(x, axis=1, keepdims=True)))
        else:
            ee = [p.e_rounded]
        r = 8
        while True:
            rows = np.arange(r)
            t0 = time.perf_counter()
            for e in ee:
                if w.get("groups"):   # each sampled anchor row with its group's pair
                    g, tv, bv = w["groups"]
                    for q in range(len(tv)):
                        sel = rows[g[rows] == q]
                        if sel.size:
                            oracle.pair_loss_sigmoid(e, float(tv[q]), float(bv[q]), p.attract,
                                                     ignore=p.ignore if p.ignore.ids.size else None, rows=sel,
                                                     threads=threads)
                else:
                    oracle.pair_loss_sigmoid(e, p.t, p.b, p.attract, ignore=p.ignore if p.ignore.ids.size else None,
                                             rows=rows, threads=threads)
            dt = time.perf_counter() - t0
            if dt > budget_s / parts / 4 or r >= p.count:
                break
            r = min(p.count, max(r * 2, int(r * (budget_s / parts) / max(dt, 1e-3) / 2)))
        flops += sum(3.0 * p.count * e.shape[1] * r for e in ee)
        secs += dt
        desc.append(f"pooled: {r} of {p.count} anchors" + (f" at each of the prefixes {pre}" if pre else ""))
    if m is not None:
        rng = np.random.default_rng(0)
        k = 16
        q, d = m.q, m.d
        while True:
            if w.get("named"):   # a sample of the named pairs
                nq_all, nd_all = _named_pairs(m, w["named"])
                pick = rng.integers(0, nq_all.size, k)
                pq, pd = nq_all[pick], nd_all[pick]
            else:
                pq, pd = rng.integers(0, m.nq, k), rng.integers(0, m.nd, k)
            t0 = time.perf_counter()
            oracle.maxsim_pairs(m.q_offsets, q, m.d_offsets, d, pq, pd, threads=threads)
            dt = time.perf_counter() - t0
            if dt > budget_s / parts / 4 or k >= 1 << 22:
                break
            k = max(k * 2, int(k * (budget_s / parts) / max(dt, 1e-3) / 2))
        ql = (m.q_offsets[pq + 1] - m.q_offsets[pq]).astype(np.float64)
        dl = (m.d_offsets[pd + 1] - m.d_offsets[pd]).astype(np.float64)
        flops += float(np.sum(2.0 * m.width * ql * dl + 4.0 * m.width * ql))
        secs += dt
        desc.append(f"MaxSim: {k} random (query, document) pairs of {m.nq}x{m.nd}" +
                    (" among the named ones" if w.get("named") else ""))
    return flops, secs, "; ".join(desc)


# ---------------------------------------------------------------------------
# main
# ---------------------------------------------------------------------------

def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    pg = None
    if world > 1:
        import torch.distributed as dist
        import torch
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend=backend)
        pg = dist
    return world, rank, local, pg


def max_over_ranks(pg, value, device):
    """The slowest rank's value (every rank gets it); `pg` is torch.distributed or None."""
    if pg is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def aggregate(pg, world, flops_per_rank, ms_local, device):
    """Weak scaling: every rank runs its own batch of `flops_per_rank`; the job's time is the slowest
    rank's, and its throughput is all ranks' work over that time.  Returns (ms, TFLOP/s)."""
    ms = max_over_ranks(pg, ms_local, device)
    return ms, world * flops_per_rank / (ms * 1e-3) / 1e12


def run_reference(args, world, rank):
    if rank != 0:
        return 0
    threads = os.cpu_count() or 1
    w = make_workload(args.workload, 0)
    budget = max(2.0, min(30.0, 150.0 / max(1, args.steps + args.warmup)))
    times, flops_list = [], []
    desc = ""
    for i in range(args.warmup + args.steps):
        fl, sec, desc = oracle_sample(w, budget, threads)
        if i >= args.warmup:
            times.append(sec)
            flops_list.append(fl)
    value = sum(flops_list) / sum(times) / 1e12
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * sum(times) / len(times),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": describe(args.workload, w),
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle", "sample": desc},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def step_names(step):
    """The per-call event names of a step, in launch order."""
    names = []
    if step.p is not None:
        names.append("pooled")
    if step.m is not None:
        names.append("maxsim_fwd")
        if step.j is not None or step.named is not None:
            names.append("score_loss")
        names.append("maxsim_bwd")
    return names


def timed_region(step, stream, flush, steps, device_index, pg=None):
    """K steps on the step's stream, the L2 flushed between them (outside the per-step events), bracketed by a
    barrier and a device synchronisation on both sides, with nvidia-smi clocks sampled inside.  Returns
    (per-step ms, {call: per-step ms}, clock summary, wall seconds)."""
    import torch
    names = step_names(step)
    ev = [{n: (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for n in names}
          for _ in range(steps)]
    st_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    if pg is not None:
        pg.barrier()
    torch.cuda.synchronize()
    with ClockSampler(device_index) as clocks:
        clocks.mark(True)
        wall0 = time.perf_counter()
        for k in range(steps):
            with torch.cuda.stream(stream):
                flush.fill_(k & 0xFF)
                st_ev[k][0].record(stream)
                step.run(ev[k])
                st_ev[k][1].record(stream)
        torch.cuda.synchronize()
        wall = time.perf_counter() - wall0
        clocks.mark(False)
    if pg is not None:
        pg.barrier()
    step_ms = [a.elapsed_time(b) for a, b in st_ev]
    part_ms = {n: [ev[k][n][0].elapsed_time(ev[k][n][1]) for k in range(steps)] for n in names}
    return step_ms, part_ms, clocks.summary(), wall


def warm(step, stream, warmup):
    for _ in range(max(3, warmup)):
        step.run()
    stream.synchronize()
    bad = [s for s in step.statuses() if s != 0]
    if bad:
        raise SystemExit(f"device status {bad} after warm-up")


def part_lines(step, w, part_ms, burst, sustained):
    """The per-call numbers of a timed region: pooled pairs/s and TFLOP/s, MaxSim fwd+bwd TFLOP/s, each as a
    fraction of the burst bf16 peak (the calls run at full clock in a short timed region; the sustained
    peak's fraction is given beside it)."""
    p, m = step.p, step.m
    pre = w.get("prefixes")
    parts = {}
    if p is not None:
        pm = statistics.mean(part_ms["pooled"])
        tf = pooled_flops(p, pre) / (pm * 1e-3) / 1e12
        parts["pair_loss"] = {"ms": pm, "pairs_per_s": len(pre or [0]) * p.count * (p.count - 1) / (pm * 1e-3),
                              "tflops": tf, "frac_of_peak": tf / burst, "frac_of_sustained_peak": tf / sustained,
                              "N": p.count, "D": p.width}
    if m is not None:
        fm, bm = statistics.mean(part_ms["maxsim_fwd"]), statistics.mean(part_ms["maxsim_bwd"])
        fwd, bwd = maxsim_fwd_flops(m, w.get("named")), maxsim_bwd_flops(m, w.get("named"))
        tf = (fwd + bwd) / ((fm + bm) * 1e-3) / 1e12
        active = step.active_pairs()
        parts["maxsim"] = {"fwd_ms": fm, "bwd_ms": bm, "tflops_fwd_bwd": tf, "frac_of_peak": tf / burst,
                           "frac_of_sustained_peak": tf / sustained, "fwd_tflops": fwd / (fm * 1e-3) / 1e12,
                           "bwd_active_pairs": active,
                           # one bf16 row gathered per active (query row, document) pair for each of dQ and dD
                           "bwd_gathered_bytes": active * 4.0 * m.width,
                           "bwd_gathered_gb_per_s": active * 4.0 * m.width / (bm * 1e-3) / 1e9}
        if "score_loss" in part_ms:
            parts["score_loss"] = {"ms": statistics.mean(part_ms["score_loss"])}
    return parts


def extra_part(name, seed, device, stream, flush, args, burst, sustained):
    """A separately timed workload of the default run (the largest pooled config, the config-3 MaxSim), under
    the same timing rules as the main line; returns its per-call numbers and its clocks."""
    import torch
    w = make_workload(name, seed)
    step = Step(w, device, stream)
    warm(step, stream, args.warmup)
    step_ms, part_ms, clk, _ = timed_region(step, stream, flush, args.steps, device.index or 0)
    out = part_lines(step, w, part_ms, burst, sustained)
    out = out.get("pair_loss") or out.get("maxsim")
    out.update({"workload": describe(name, w)["workload"], "ms_per_step": statistics.mean(step_ms), "clocks": clk,
                "traffic": committed_traffic(name, "pooled" if w["pooled"] is not None else "maxsim")})
    del step
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return out


def e2e_serial(step, stream, steps, pg, device):
    """Per step on one stream: the inputs in, the step, the results out.  Returns (ms per step, bytes in,
    bytes out)."""
    import torch
    outs_host = [torch.empty(d.shape, dtype=d.dtype).pin_memory() for d in step.results()]
    for _ in range(2):
        step.upload()
        step.run()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if pg is not None:
        pg.barrier()
    h2d = d2h = 0
    t0 = time.perf_counter()
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(steps):
            h2d = step.upload()
            step.run()
            for h, d in zip(outs_host, step.results()):
                h.copy_(d, non_blocking=True)
            d2h = sum(h.numel() * h.element_size() for h in outs_host)
        e1.record(stream)
    stream.synchronize()
    ms = max(e0.elapsed_time(e1), (time.perf_counter() - t0) * 1e3) / steps
    return max_over_ranks(pg, ms, device), h2d, d2h


def e2e_pipelined(steps2, stream, steps, pg, device):
    """Steps alternate between two device buffer sets: step k's inputs go in on one copy stream once step
    k - 2 (the last user of its set) has finished, the step runs on `stream` once they are in and step
    k - 2's results are out, and its results come back on a second copy stream, so the copies of one step
    overlap the compute of the next.  Every step still copies all of its inputs in and all of its results
    out inside the timed region.  Returns (ms per step, bytes in, bytes out)."""
    import torch
    h2d_s, d2h_s = torch.cuda.Stream(device=device), torch.cuda.Stream(device=device)
    outs_host = [[torch.empty(d.shape, dtype=d.dtype).pin_memory() for d in st.results()] for st in steps2]
    ev = lambda: torch.cuda.Event()
    copied_in = [ev(), ev()]
    computed = [ev(), ev()]
    copied_out = [ev(), ev()]
    sizes = {}

    def one(k):
        i = k % 2
        st = steps2[i]
        if k >= 2:
            h2d_s.wait_event(computed[i])
        sizes["in"] = st.upload(h2d_s)
        copied_in[i].record(h2d_s)
        stream.wait_event(copied_in[i])
        if k >= 2:
            stream.wait_event(copied_out[i])
        st.run()
        computed[i].record(stream)
        d2h_s.wait_event(computed[i])
        with torch.cuda.stream(d2h_s):
            for h, d in zip(outs_host[i], st.results()):
                h.copy_(d, non_blocking=True)
        copied_out[i].record(d2h_s)
        sizes["out"] = sum(h.numel() * h.element_size() for h in outs_host[i])

    for k in range(4):
        one(k)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if pg is not None:
        pg.barrier()
    t0 = time.perf_counter()
    e0.record(h2d_s)
    stream.wait_event(e0)
    d2h_s.wait_event(e0)
    for k in range(steps):
        one(k + 4)
    stream.wait_event(copied_out[(steps + 3) % 2])
    stream.wait_event(copied_out[(steps + 2) % 2])
    e1.record(stream)
    torch.cuda.synchronize()
    ms = max(e0.elapsed_time(e1), (time.perf_counter() - t0) * 1e3) / steps
    return max_over_ranks(pg, ms, device), sizes["in"], sizes["out"]


def main():
    args = parse_args()
    if args.impl == "reference":
        # The oracle runs on rank 0's host cores only; other ranks exit at once, without a process group.
        world = int(os.environ.get("WORLD_SIZE", "1"))
        rank = int(os.environ.get("RANK", "0"))
        return run_reference(args, world, rank)
    world, rank, local, pg = dist_setup(args)
    import torch
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    stream = torch.cuda.Stream(device=device)
    w = make_workload(args.workload, rank)   # weak scaling: every rank its own batch
    step = Step(w, device, stream)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
    warm(step, stream, args.warmup)

    # --- timed region: K steps, L2 flushed between steps (outside the per-step events) ---
    step_ms, part_ms, clocks, wall = timed_region(step, stream, flush, args.steps, local, pg)
    p, m = step.p, step.m
    pre = w.get("prefixes")
    flops = (pooled_flops(p, pre) if p is not None else 0.0) + \
            ((maxsim_fwd_flops(m, w.get("named")) + maxsim_bwd_flops(m, w.get("named"))) if m is not None else 0.0)
    ms, value = aggregate(pg, world, flops, statistics.mean(step_ms), device)
    burst, sustained, hbm, peak_src = peaks()
    parts = part_lines(step, w, part_ms, burst, sustained)

    # roofline: the dominant kernel (by time) of the step, against the burst peak (a short timed region at
    # full clock); the sustained peak's fraction beside it
    if m is not None:
        fm = statistics.mean(part_ms["maxsim_fwd"])
        achieved = maxsim_fwd_flops(m, w.get("named")) / (fm * 1e-3) / 1e12
        roofline = {"kernel": "maxsim forward (maxsim_scores call: forward tile kernel + its schedule, tape "
                              "checks and query sums)",
                    "bound": "tensor", "achieved": achieved, "peak": burst, "unit": "TFLOP/s",
                    "frac": achieved / burst, "peak_source": f"{peak_src} bf16 burst",
                    "frac_of_sustained_peak": achieved / sustained,
                    "traffic": committed_traffic(args.workload),
                    "algorithmic_per_launch": maxsim_fwd_flops(m, w.get("named"))}
    else:
        pm = statistics.mean(part_ms["pooled"])
        achieved = pooled_flops(p, pre) / (pm * 1e-3) / 1e12
        call = ("pair_loss_sigmoid_groups_fwd_bwd" if w.get("groups") else
                "pair_loss_sigmoid_matryoshka_fwd_bwd" if pre else "pair_loss_sigmoid_fwd_bwd")
        roofline = {"kernel": f"pooled fused block kernel ({call} call)", "bound": "tensor",
                    "achieved": achieved, "peak": burst, "unit": "TFLOP/s", "frac": achieved / burst,
                    "peak_source": f"{peak_src} bf16 burst", "frac_of_sustained_peak": achieved / sustained,
                    "traffic": committed_traffic(args.workload, "pooled"),
                    "algorithmic_per_launch": pooled_flops(p, pre)}

    # end to end through the C ABI with host buffers: every input copied in from pinned host memory and every
    # result (losses, dE, scores, dQ, dD) copied back, each step
    e2e = None
    if not args.no_e2e:
        serial_ms, _, _ = e2e_serial(step, stream, args.steps, pg, device)
        step2 = Step(w, device, stream)   # the second device buffer set of the pipelined copies
        e2e_ms, h2d, d2h = e2e_pipelined((step, step2), stream, args.steps, pg, device)
        bad2 = [s for s in step2.statuses() if s != 0]
        if bad2:
            raise SystemExit(f"device status {bad2}")
        del step2
        torch.cuda.empty_cache()
        e2e = {"value": world * flops / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s", "ms_per_step": e2e_ms,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "copies": "step k+1's inputs copied in and step k's results copied out on two copy streams while "
                         "step k+1 computes (two device buffer sets)",
               "serial_ms_per_step": serial_ms,
               "serial_value": world * flops / (serial_ms * 1e-3) / 1e12}

    bad = [s for s in step.statuses() if s != 0]
    if bad:
        raise SystemExit(f"device status {bad}")
    launches = step.launches_per_step() * args.steps

    # the largest pooled config and the config-3 MaxSim, timed on their own (rank 0, single GPU)
    if args.workload == "joint" and not args.no_extra_parts and world == 1:
        del step
        torch.cuda.empty_cache()
        parts["pooled_config4"] = extra_part("pooled4", rank, device, stream, flush, args, burst, sustained)
        parts["maxsim_config3"] = extra_part("maxsim3", rank, device, stream, flush, args, burst, sustained)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        threads = os.cpu_count() or 1
        fl, sec, desc = oracle_sample(w, args.cpu_seconds, threads)
        cpu = {"value": fl / sec / 1e12, "unit": "TFLOP/s", "cores": threads, "kind": "oracle", "sample": desc}

    if rank == 0:
        cfg = describe(args.workload, w)
        cfg["parallelism"] = f"replicas x{world} (independent batches)" if world > 1 else "single GPU"
        cfg["l2"] = "flushed between timed steps (256 MiB write outside the step events)"
        line = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
                "warmup": max(3, args.warmup), "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "bf16", "data": "synthetic", "config": cfg, "parts": parts,
                "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": launches,
                "clocks": clocks, "wall_s_timed": wall}
        print(json.dumps(line), flush=True)
    if pg is not None:
        pg.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
