"""Benchmark of the DFlash2 draft-block head on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload NAME]
                    [--no-records] [--no-cpu-baseline]

One step = one pass of the whole head over one draft batch of the workload:
conv_prepare -> conv_finish (one sublayer's conv pair) -> draft_head (unary
logits, top-K and hidden projection, the selector walk and the teacher-forced
scores in one call).  The timed steps replay those calls captured as two CUDA
graphs; the end-to-end leg makes the calls directly with host buffers.  Inputs are
seeded synthetic tensors (see workloads/), resident in HBM before timing; the
step streams the whole LM head (1.25 GB for the default batch-1 workload, larger
than the 129 MB L2), so no separate L2 flush is needed for the default workload;
other workloads flush L2 with a 256 MB write between steps.

Prints one JSON line (rank 0).  The headline is the batch-1 workload; a default run
then appends a "workloads" object with one record each for the batched, stress and
training-packed conv workloads (timing, roofline, cpu baseline, parity, e2e,
clocks).  Each workload's "parity" block compares the timed step's outputs with the
oracle on the first requests, the same slice its cpu baseline times.  Under
torchrun each rank runs an independent replica on its own GPU (the head shards by
requests with no exchange: "weak" scaling); the time is the max over ranks.
--impl reference times the CPU oracle on the host cores on the same workload instead.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)
sys.path.insert(0, os.path.join(ROOT, "tests"))

import workloads as W  # noqa: E402

METRIC = "draft positions/s (topK+selector walk) and conv GB/s, % of HBM/TC roofline"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


# The dominant kernel per workload, the committed ncu summary of it, and the
# sources whose hash the summary records.
PROFILES = {
    "batch1": ("head_skinny_kernel_batch1.md", ["head_tc.cu", "topk_warp.cuh", "tc_ptx.cuh", "common.cuh"]),
    "batched": ("gemm_wide_topk_batched.md", ["gemm_tc.cu", "tc_pair.cuh", "tc_ptx.cuh", "common.cuh"]),
    "stress": ("gemm_wide_topk_stress.md", ["gemm_tc.cu", "tc_pair.cuh", "tc_ptx.cuh", "common.cuh"]),
    "conv": ("conv_prepare_tc_conv.md", ["conv_tc.cu", "tc_pair.cuh", "tc_ptx.cuh", "common.cuh"]),
    "conv_finish": ("conv_apply_bulk_conv.md", ["conv.cu", "tc_ptx.cuh", "common.cuh"]),
}


def head_traffic(workload="batch1"):
    """DRAM traffic per launch of the workload's dominant kernel from the committed
    ncu summary, or None when there is none or the kernel's sources changed since."""
    import hashlib
    import re
    if workload not in PROFILES:
        return None, "no capture for this workload"
    fname, sources = PROFILES[workload]
    path = os.path.join(ROOT, "profiles", fname)
    try:
        text = open(path).read()
        h = hashlib.sha256()
        for f in sources:
            with open(os.path.join(ROOT, "dflash2_draft_block_gb300", "csrc", f), "rb") as fh:
                h.update(fh.read())
        sha = re.search(r"source_sha256_16 = ([0-9a-f]{16})", text).group(1)
        traffic = int(re.search(r"traffic_bytes_per_launch = (\d+)", text).group(1))
    except (OSError, AttributeError, ValueError):
        return None, "no capture"
    if h.hexdigest()[:16] != sha:
        return None, "kernel changed since the capture"
    return traffic, "profiles/" + fname


def slowest_rank_ms(ms, dist, device):
    """Max of a per-rank time over all ranks (the job is as slow as its slowest
    replica); unchanged when not distributed."""
    if dist is None:
        return ms
    import torch
    t = torch.tensor([float(ms)], device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank, world, ms):
    """Whole-job rate: every rank processed units_per_rank in the (max) time ms."""
    return units_per_rank * world / (ms * 1e-3)


def head_bytes(w):
    """Algorithmic bytes of unary_topk: W_lm + W_H + h read once, ids/vals/G written."""
    return (w.V * w.D * 2 + w.r * w.D * 2 + w.P * w.D * 2 + w.P * w.K * 8 + w.P * w.r * 4)


def draft_bytes(w):
    """Algorithmic bytes of the draft head: the head's, plus the walk's gathered rows
    (per request the anchor's and every predecessor candidate's A row, every
    candidate's B row) and the teacher-forced scores' (per row one A row and K B
    rows), the path and the scores written."""
    T = w.B - 1
    walk = w.R * ((1 + (T - 1) * w.K) + T * w.K) * w.r * 2 + w.R * T * 8
    pair = w.P * (1 + w.K) * w.r * 2 + w.P * w.K * 4
    return head_bytes(w) + walk + pair


def conv_bytes(w, which):
    C, P, G = w.C, w.P, w.G
    act = 2 if w.act == "bf16" else 4
    if which == "prepare":  # x read, y written, W_proj read, dyn_out written, base read
        return P * C * act * 2 + 2 * w.taps * G * C * 2 + P * w.taps * G * 4 + 2 * w.taps * C * 4
    return P * C * act * 2 + P * w.taps * G * 4 + 2 * w.taps * C * 4  # finish


def lattice_bytes(w):
    """Algorithmic bytes of selector_lattice: per request the anchor's A row and the K
    predecessor candidates' A rows of every slot after the first, the K successor
    B rows of every slot, G and the unary values of the drafted rows, and the table
    written."""
    T = w.B - 1
    rows = w.R * ((1 + (T - 1) * w.K) + T * w.K)
    return (rows * w.r * 2 + w.R * T * (w.r * 4 + w.K * 8) + w.R * T * w.K * w.K * 4)


def lattice_flops(w):
    T = w.B - 1
    return 2.0 * w.R * (w.K + (T - 1) * w.K * w.K) * w.r


def time_per_call(step, torch, n):
    """Per-call breakdown from separate loops with an event between consecutive calls
    (outside the timed region): the step's three calls, then the draft head's three
    separate equivalents."""
    out = []
    for runner, ncalls in ((step.run, 3), (step.run_separate, 3)):
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(ncalls + 1)] for _ in range(n)]
        for s in range(n):
            if runner is step.run:
                runner(evs[s])
            else:
                step.run(None)
                runner(evs[s])
            if step.flush is not None:
                step.flush.zero_()
        torch.cuda.synchronize()
        per_call = np.zeros(ncalls)
        for s in range(n):
            for i in range(ncalls):
                per_call[i] += evs[s][i].elapsed_time(evs[s][i + 1])
        out += (per_call / n * 1e3).tolist()
    return out


def graph_time_us(torch, call, iters=20, reps=5):
    """GPU time per call of a short call: `iters` calls captured in one CUDA graph and
    the graph replayed, so the host's per-call cost (Python, argument checks) does
    not show.  Returns (microseconds per call, how it was timed); falls back to a
    plain loop, which then measures host-bound submission, if capture fails."""
    call()
    torch.cuda.synchronize()
    try:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for _ in range(iters):
                call()
        g.replay()
        torch.cuda.synchronize()
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        ev[0].record()
        for _ in range(reps):
            g.replay()
        ev[1].record()
        torch.cuda.synchronize()
        return ev[0].elapsed_time(ev[1]) / (reps * iters) * 1e3, "graph"
    except RuntimeError:
        torch.cuda.synchronize()
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        ev[0].record()
        for _ in range(iters):
            call()
        ev[1].record()
        torch.cuda.synchronize()
        return ev[0].elapsed_time(ev[1]) / iters * 1e3, "loop"


def time_next_rows(step, torch, df2, iters=20):
    """Per-call times of the lattice schedule on the step's own candidates: the table,
    then the greedy and the sampling walk over it; then the draft head with capped
    logits (multiplier 1, softcap 30); then the conv finish fused with the next
    prepare (residual = the step's x), and the same as its separate calls with the
    residual added by torch; then the selector's K-way cross-entropy on the step's
    teacher-forced scores.  None of it is part of the timed step."""
    w = step.w
    lat = torch.empty((w.R, w.B - 1, w.K, w.K), dtype=torch.float32, device=step.ids.device)
    gen = torch.Generator(device=step.ids.device)
    gen.manual_seed(w.seed)
    u = torch.rand((w.R, w.B - 1), generator=gen, device=step.ids.device)
    path = torch.empty((w.R, w.B - 1), dtype=torch.int32, device=step.ids.device)
    sc = torch.empty((w.R, w.B - 1), dtype=torch.float32, device=step.ids.device)
    h, y_next, dyn_next = torch.empty_like(step.z), torch.empty_like(step.z), torch.empty_like(step.dyn)
    ws_conv = step.ws_conv
    # the selector loss's ground truth: a candidate of the row for three rows in four
    # (a column chosen by the row index), a random token (mostly not a candidate) else
    rows = torch.arange(w.P, device=step.ids.device)
    pick = step.ids[rows, (rows * 7) % w.K]
    other = torch.randint(0, w.V, (w.P,), generator=gen, device=step.ids.device, dtype=torch.int32)
    targets = torch.where(rows % 4 == 3, other, pick).to(torch.int32).contiguous()
    ce_out = (torch.empty((w.P,), dtype=torch.float32, device=step.ids.device),
              torch.empty((w.P,), dtype=torch.int32, device=step.ids.device))

    def finish_add_prepare():
        hs = df2.conv_finish(step.z, w.B, w.taps, w.g, step.dyn, step.base, out=h)
        hs.add_(step.x)
        df2.conv_prepare(hs, w.B, w.taps, w.g, step.W_proj, step.base, workspace=ws_conv, out=(y_next, dyn_next))

    calls = [
        lambda: df2.selector_lattice(step.anchors, step.ids, step.vals, step.Gt, step.A, step.Bc, w.B, out=lat),
        lambda: df2.lattice_walk(lat, step.ids, w.B, w.V, out=(path, sc)),
        lambda: df2.lattice_walk(lat, step.ids, w.B, w.V, uniforms=u, temperature=1.0, out=(path, sc)),
        lambda: df2.draft_head(step.h, step.W_lm, w.K, step.W_H, step.A, step.Bc, step.anchors, w.B, step.pred,
                               output_multiplier=1.0, final_logit_softcapping=30.0, workspace=step.ws_draft,
                               out=(step.ids, step.vals, step.Gt, step.path, step.pscore, step.scores)),
        lambda: df2.conv_finish_prepare(step.z, w.B, w.taps, w.g, step.dyn, step.base, step.W_proj, step.base,
                                        step.x, workspace=ws_conv, out=(h, y_next, dyn_next)),
        finish_add_prepare,
        lambda: df2.selector_ce(step.scores, step.ids, targets, w.V, out=ce_out),
    ]
    out, how = [], set()
    for c in calls:
        us, kind = graph_time_us(torch, c, iters)
        out.append(us)
        how.add(kind)
    return out, "+".join(sorted(how))


def config_of(w):
    return {"workload": f"{w.name}: V={w.V} D={w.D} r={w.r} K={w.K} block={w.B} requests={w.R} "
                        f"(P={w.P} positions) conv taps={w.taps} group={w.g}",
            "positions_per_step": w.P, "drafted_positions_per_step": w.R * (w.B - 1),
            "l2": ("inputs larger than L2: the 1.25+ GB LM head is streamed every step"
                   if w.V * w.D * 2 > 256 << 20 else "L2 flushed between steps (256 MB write)")}


# ------------------------------------------------------------------ clocks --

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.dev = device_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", str(self.dev)], stdout=subprocess.PIPE,
                stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *a):
        self.out = ""
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self):
        rows = [l.split(",") for l in (self.out or "").strip().splitlines() if l.count(",") >= 8]
        if not rows:
            try:
                one = subprocess.run(["nvidia-smi", f"--query-gpu={self.FIELDS}",
                                      "--format=csv,noheader,nounits", "-i", str(self.dev)],
                                     capture_output=True, text=True, timeout=10).stdout
                rows = [l.split(",") for l in one.strip().splitlines() if l.count(",") >= 8]
            except (OSError, subprocess.TimeoutExpired):
                rows = []
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        sm = []
        smax = None
        for r in rows:
            r = [x.strip() for x in r]
            try:
                sm.append(float(r[1]))
                smax = float(r[2])
            except ValueError:
                pass
            for n, v in zip(names, r[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(rows)}


# -------------------------------------------------------------- GPU arm --

class Step:
    """Device-resident inputs/outputs of one workload and the five calls."""

    def __init__(self, w, device, torch, df2, inp=None, conv=None):
        self.w, self.torch, self.df2 = w, torch, df2
        inp = W.head_inputs(w) if inp is None else inp
        conv = W.conv_inputs(w) if conv is None else conv

        def bf(a):
            return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(device).view(torch.bfloat16)

        def dv(a):
            return torch.from_numpy(np.ascontiguousarray(a)).to(device)

        self.host = {"h": inp["h"], "x": conv["x"], "z": conv["z"], "anchors": inp["anchors"],
                     "pred": inp["pred"]}
        self.h, self.W_lm, self.W_H = bf(inp["h"]), bf(inp["W_lm"]), bf(inp["W_H"])
        self.A, self.Bc = bf(inp["A"]), bf(inp["Bc"])
        self.anchors, self.pred = dv(inp["anchors"]), dv(inp["pred"])
        act = bf if w.act == "bf16" else dv
        self.x, self.z = act(conv["x"]), act(conv["z"])
        self.W_proj, self.base = bf(conv["W_proj"]), dv(conv["base"])
        P, K, r, G = w.P, w.K, w.r, w.G
        e = torch.empty
        self.ids = e((P, K), dtype=torch.int32, device=device)
        self.vals = e((P, K), dtype=torch.float32, device=device)
        self.Gt = e((P, r), dtype=torch.float32, device=device)
        self.path = e((w.R, w.B - 1), dtype=torch.int32, device=device)
        self.pscore = e((w.R, w.B - 1), dtype=torch.float32, device=device)
        self.scores = e((P, K), dtype=torch.float32, device=device)
        self.y = torch.empty_like(self.x)
        self.y2 = torch.empty_like(self.z)
        self.dyn = e((P, w.taps, G), dtype=torch.float32, device=device)
        self.ws_draft = e(max(1, df2.draft_head_workspace_size(w.R, w.B, w.D, w.V, K, r)), dtype=torch.uint8,
                          device=device)
        self.ws_head = e(max(1, df2.unary_topk_workspace_size(P, w.D, w.V, K, r)), dtype=torch.uint8,
                         device=device)
        dt = df2.DF2_DTYPE_BF16 if w.act == "bf16" else df2.DF2_DTYPE_F32
        self.ws_conv = e(max(1, df2.conv_prepare_workspace_size(P, w.C, w.taps, w.g, dt)),
                         dtype=torch.uint8, device=device)
        self.torch = torch
        self.flush = None
        if w.V * w.D * 2 <= 256 << 20:
            self.flush = e(256 << 20, dtype=torch.uint8, device=device)

    def run(self, events=None):
        """One step: conv_prepare, conv_finish, then the fused draft head (unary
        top-K + H, greedy walk, teacher-forced scores).  events: None, four events
        (one between consecutive calls), or a pair (recorded around the draft head)."""
        d, w = self.df2, self.w
        ev = events or [None] * 4
        if len(ev) == 2:
            ev = [None, None, ev[0], ev[1]]
        self._rec(ev[0])
        d.conv_prepare(self.x, w.B, w.taps, w.g, self.W_proj, self.base, workspace=self.ws_conv,
                       out=(self.y, self.dyn))
        self._rec(ev[1])
        d.conv_finish(self.z, w.B, w.taps, w.g, self.dyn, self.base, out=self.y2)
        self._rec(ev[2])
        d.draft_head(self.h, self.W_lm, w.K, self.W_H, self.A, self.Bc, self.anchors, w.B, self.pred,
                     workspace=self.ws_draft,
                     out=(self.ids, self.vals, self.Gt, self.path, self.pscore, self.scores))
        self._rec(ev[3])

    IO_IN = ("h", "x", "z", "anchors", "pred")
    IO_OUT = ("ids", "vals", "Gt", "path", "pscore", "scores", "y", "y2", "dyn")

    def buffers(self):
        """The step's per-step inputs and outputs (weights and workspaces are shared)."""
        return {k: getattr(self, k) for k in self.IO_IN + self.IO_OUT}

    def new_buffers(self):
        return {k: self.torch.empty_like(v) for k, v in self.buffers().items()}

    def use(self, bufs):
        for k, v in bufs.items():
            setattr(self, k, v)

    def capture(self):
        """The step as two CUDA graphs -- the conv calls, then the draft head call --
        so that replaying them launches the same kernels without the host's per-call
        work between them.  Returns None when capture is not possible here."""
        torch = self.torch
        try:
            g_conv, g_head = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
            d, w = self.df2, self.w
            with torch.cuda.graph(g_conv):
                d.conv_prepare(self.x, w.B, w.taps, w.g, self.W_proj, self.base, workspace=self.ws_conv,
                               out=(self.y, self.dyn))
                d.conv_finish(self.z, w.B, w.taps, w.g, self.dyn, self.base, out=self.y2)
            with torch.cuda.graph(g_head):
                d.draft_head(self.h, self.W_lm, w.K, self.W_H, self.A, self.Bc, self.anchors, w.B, self.pred,
                             workspace=self.ws_draft,
                             out=(self.ids, self.vals, self.Gt, self.path, self.pscore, self.scores))
            torch.cuda.synchronize()
            return g_conv, g_head
        except RuntimeError:
            torch.cuda.synchronize()
            return None

    def run_separate(self, events):
        """The draft head as its three separate calls, an event between each (for the
        per-call breakdown)."""
        d, w = self.df2, self.w
        self._rec(events[0])
        d.unary_topk(self.h, self.W_lm, w.K, self.W_H, workspace=self.ws_head,
                     out=(self.ids, self.vals, self.Gt))
        self._rec(events[1])
        d.selector_walk(self.anchors, self.ids, self.vals, self.Gt, self.A, self.Bc, w.B,
                        out=(self.path, self.pscore))
        self._rec(events[2])
        d.selector_pair_scores(self.pred, self.ids, self.vals, self.Gt, self.A, self.Bc,
                               out=self.scores)
        self._rec(events[3])

    @staticmethod
    def _rec(e):
        if e is not None:
            e.record()

    def outputs(self):
        return [self.ids, self.vals, self.path, self.pscore, self.scores, self.y, self.y2, self.dyn]

    def host_outputs(self):
        """The step's outputs on the host, named as the parity comparators expect
        (bf16 tensors as uint16 bit patterns)."""
        torch = self.torch
        torch.cuda.synchronize()

        def h(t):
            if t.dtype == torch.bfloat16:
                return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
            return t.cpu().numpy()
        return {"ids": h(self.ids), "vals": h(self.vals), "G": h(self.Gt), "path": h(self.path),
                "pscore": h(self.pscore), "scores": h(self.scores), "y": h(self.y), "dyn": h(self.dyn),
                "y2": h(self.y2)}


def count_launches(step, torch, df2):
    """Kernels one step launches, from the library's own launch counter."""
    torch.cuda.synchronize()
    before = df2.kernels_launched()
    step.run()
    torch.cuda.synchronize()
    return df2.kernels_launched() - before


NOMINAL = {"hbm_gbs": 8000.0, "bf16_tflops": 2250.0}


def fractions(roof, peaks_src):
    """frac against the measured peak (the roofline denominator) and against the
    nominal figure (8 TB/s HBM, 2.25 PFLOP/s dense bf16)."""
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["peak_source"] = peaks_src
    nominal = NOMINAL["hbm_gbs"] if roof["bound"] == "hbm" else NOMINAL["bf16_tflops"]
    roof["frac_of_nominal"] = roof["achieved"] / nominal
    roof["nominal_peak"] = nominal
    return roof


def soak(fn, torch, seconds, chunk):
    """Runs fn back to back for about `seconds` (untimed), so that the clock samples
    taken over it and the timed region that follows see the GPU under this load."""
    t_end = time.perf_counter() + seconds
    n = 0
    while time.perf_counter() < t_end:
        for _ in range(chunk):
            fn()
        torch.cuda.synchronize()
        n += chunk
    return n


def with_clock_product(clocks, ms):
    if clocks.get("sm_mhz"):
        clocks["ms_per_step_x_sm_mhz"] = ms * clocks["sm_mhz"]
    clocks["window"] = ("nvidia-smi every 100 ms over a 1 s soak of the same step directly before the "
                        "timed region, and over the timed region")
    return clocks


def gpu_arm(args, w, rank, world, torch, df2, dist, device, inp=None, conv=None, steps=None, warmup=None):
    """The draft-block step of a head workload on this rank's GPU; returns the JSON
    record (rank 0) and the step (for the parity comparison)."""
    steps = args.steps if steps is None else steps
    warmup = args.warmup if warmup is None else warmup
    local = device.index
    step = Step(w, device, torch, df2, inp, conv)
    for _ in range(warmup):
        step.run()
        if step.flush is not None:
            step.flush.zero_()
    torch.cuda.synchronize()
    n_launch = count_launches(step, torch, df2)
    graphs = step.capture()
    if graphs is not None:
        for _ in range(warmup):
            graphs[0].replay()
            graphs[1].replay()
        torch.cuda.synchronize()

    def one_step():
        if graphs is not None:
            graphs[0].replay()
            graphs[1].replay()
        else:
            step.run()
        if step.flush is not None:
            step.flush.zero_()

    # ---- device-resident timing (W warm-up done above).  Each step replays the
    # conv graph and the draft-head graph (or, where capture is not possible, makes
    # the calls).  Only the head call is bracketed by events: every event between
    # kernels drains the launch pipeline, so more of them would inflate the step.
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    flush_ms = 0.0
    chunk = 64 if w.P <= 32 else 8
    with ClockSampler(local) as clk:
        soak(one_step, torch, 1.0, chunk)
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()
        launched0 = df2.kernels_launched()
        t0.record()
        for s in range(steps):
            if graphs is not None:
                graphs[0].replay()
                evs[s][0].record()
                graphs[1].replay()
                evs[s][1].record()
            else:
                step.run(evs[s])
            if step.flush is not None:
                step.flush.zero_()
        t1.record()
        torch.cuda.synchronize()
    # a graph replay launches the captured kernels without passing through the
    # library, whose counter therefore counts them per step
    timed_launches = (n_launch * steps if graphs is not None
                      else df2.kernels_launched() - launched0)
    if dist is not None:
        dist.barrier()
    total_ms = t0.elapsed_time(t1)
    head_us_live = sum(evs[s][0].elapsed_time(evs[s][1]) for s in range(steps)) / steps * 1e3
    if step.flush is not None:
        # the flush runs between timed steps; its time is subtracted
        fe = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        fe[0].record()
        for _ in range(5):
            step.flush.zero_()
        fe[1].record()
        torch.cuda.synchronize()
        flush_ms = fe[0].elapsed_time(fe[1]) / 5 * steps
    step_ms = slowest_rank_ms((total_ms - flush_ms) / steps, dist, device)
    per_call_us = time_per_call(step, torch, min(steps, 50))
    next_us, next_how = time_next_rows(step, torch, df2)

    # ---- end to end through the public API with host buffers.  Every step copies its
    # inputs in from pinned host memory and its results out, with two steps in
    # flight as a server runs them: step i+1's inputs go in and step i-1's results
    # come out on copy streams while step i's kernels run; events keep each buffer
    # set from being overwritten while a kernel or a copy still uses it.
    out_names = [k for k in Step.IO_OUT if k != "Gt"]
    pinned_in = {k: torch.from_numpy(np.ascontiguousarray(v.view(np.int16) if v.dtype == np.uint16 else v))
                 .pin_memory() for k, v in step.host.items()}
    sets = [step.buffers(), step.new_buffers()]
    pinned_out = [{k: torch.empty(sets[0][k].shape, dtype=sets[0][k].dtype).pin_memory() for k in out_names}
                  for _ in range(2)]
    h2d = sum(v.numel() * v.element_size() for v in pinned_in.values())
    d2h = sum(sets[0][k].numel() * sets[0][k].element_size() for k in out_names)
    main_s = torch.cuda.current_stream()
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def copy_in(i):
        s = i % 2
        s_in.wait_event(ev_done[s])  # step i-2's kernels have finished with set s
        with torch.cuda.stream(s_in):
            for k, v in pinned_in.items():
                sets[s][k].view(torch.uint8).reshape(-1).copy_(v.view(torch.uint8).reshape(-1), non_blocking=True)
        ev_in[s].record(s_in)

    def compute(i):
        s = i % 2
        main_s.wait_event(ev_in[s])
        main_s.wait_event(ev_out[s])  # step i-2's results in set s have been read out
        step.use(sets[s])
        step.run()
        ev_done[s].record(main_s)
        if step.flush is not None:
            step.flush.zero_()

    def copy_out(i):
        s = i % 2
        s_out.wait_event(ev_done[s])
        with torch.cuda.stream(s_out):
            for k in out_names:
                pinned_out[s][k].copy_(sets[s][k], non_blocking=True)
        ev_out[s].record(s_out)

    def e2e_steps(n):
        for s in range(2):
            ev_done[s].record(main_s)
            ev_out[s].record(main_s)
        copy_in(0)
        for i in range(n):
            if i + 1 < n:
                copy_in(i + 1)
            compute(i)
            copy_out(i)
        for s in range(2):
            main_s.wait_event(ev_out[s])

    e2e_steps(max(1, warmup))
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    e2e_steps(steps)
    e1.record()
    torch.cuda.synchronize()
    step.use(sets[0])
    e2e_ms = slowest_rank_ms((e0.elapsed_time(e1) - flush_ms) / steps, dist, device)

    clocks = with_clock_product(clk.summary(), step_ms)
    out = None
    if rank == 0:
        peaks, src = load_peaks()
        hb = draft_bytes(w)
        head_us = head_us_live
        traffic, traffic_src = head_traffic(w.name)
        sms = torch.cuda.get_device_properties(device).multi_processor_count
        tail = ("draft_tail_kernel (fold, walk, teacher-forced scores)" if w.P <= sms
                else "top-K merge, walk and teacher-forced kernels")
        if w.P <= 32:
            # few positions: the head streams the LM head from HBM
            roof = {"kernel": "dflash2_draft_head call: head_skinny_kernel + " + tail, "bound": "hbm",
                    "achieved": hb / (head_us * 1e-6) / 1e9, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                    "algorithmic_bytes": hb}
        else:
            # many positions: the logits GEMM (plus G) is tensor-core bound
            flops = 2.0 * w.P * w.D * (w.V + w.r)
            pk = peaks.get("bf16_tflops_sustained", peaks.get("bf16_tflops"))
            roof = {"kernel": "dflash2_draft_head call: gemm_wide_kernel (top-K, G) + " + tail,
                    "bound": "tensor", "achieved": flops / (head_us * 1e-6) / 1e12, "peak": pk,
                    "unit": "TFLOP/s", "algorithmic_flops": flops}
        fractions(roof, src)
        if w.P <= 32:
            roof["target"] = {"rule": ">= 0.70 of the HBM roofline for the batch-1 LM head + top-K + walk, "
                                      "taken at the nominal 8 TB/s", "frac": roof["frac_of_nominal"],
                              "met": roof["frac_of_nominal"] >= 0.70}
        roof["traffic"] = traffic
        roof["traffic_source"] = traffic_src
        roof["traffic_note"] = "DRAM bytes per launch of the head kernel (ncu); the other kernels of the call move < 1%"
        out = {
            "metric": METRIC,
            "value": job_throughput(w.P, world, step_ms),
            "unit": "positions/s",
            "n_gpus": world,
            "steps": steps,
            "warmup": warmup,
            "ms_per_step": step_ms,
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "bf16",
            "data": "synthetic (seeded; shapes and scales of the workload, no dataset or checkpoint)",
            "config": config_of(w),
            "drafted_positions_per_s": job_throughput(w.R * (w.B - 1), world, step_ms),
            "per_call_us": dict(zip(["conv_prepare", "conv_finish", "draft_head", "unary_topk",
                                     "selector_walk", "selector_pair_scores"], per_call_us)),
            "per_call_note": "per_call_us from separate loops with events between calls (the last three "
                             "are the draft head's separate equivalents); roofline.achieved from the "
                             "draft head call's events inside the timed region",
            "draft_head_us_timed": head_us_live,
            "conv_gbs": {"prepare": conv_bytes(w, "prepare") / (per_call_us[0] * 1e-6) / 1e9,
                         "finish": conv_bytes(w, "finish") / (per_call_us[1] * 1e-6) / 1e9},
            "roofline": roof,
            "next_rows": {
                "note": "the lattice schedule, the capped-logit draft head, the fused conv finish -> prepare and the selector CE, timed on "
                        "the step's inputs outside the timed step",
                "timed_by": next_how + " (graph: the calls captured in a CUDA graph and replayed, GPU time only)",
                "selector_lattice_us": next_us[0],
                "lattice_walk_greedy_us": next_us[1],
                "lattice_walk_sampling_us": next_us[2],
                "draft_head_softcap_us": next_us[3],
                "conv_finish_prepare_us": next_us[4],
                "conv_finish_add_prepare_separate_us": next_us[5],
                "selector_ce_us": next_us[6],
                "lattice_gbs": lattice_bytes(w) / (next_us[0] * 1e-6) / 1e9,
                "lattice_tflops": lattice_flops(w) / (next_us[0] * 1e-6) / 1e12,
            },
            "e2e": {"value": job_throughput(w.P, world, e2e_ms), "unit": "positions/s",
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                    "pipelining": "two steps in flight: step i+1's inputs in and step i-1's results out "
                                  "overlap step i's calls"},
            "gpu_launches": timed_launches,
            "execution": ("each step replays two CUDA graphs captured from the public calls (conv prepare + "
                          "finish; draft head)" if graphs is not None else "eager calls"),
            "kernels_per_step": n_launch,
            "clocks": clocks,
        }
    return out, step


# ------------------------------------------------------------- conv arm --

def conv_config(w):
    return {"workload": f"{w.name}: training-packed conv, {w.R} blocks of {w.B} rows (P={w.P} positions), "
                        f"C={w.C}, taps={w.taps}, group={w.g} (G={w.G}), projection {w.C} -> {2 * w.taps * w.G}",
            "positions_per_step": w.P,
            "l2": "inputs larger than L2: x and z are 168 MB each; W_proj (13 MB) stays resident like any weight"}


class ConvStep:
    """The training-packed conv workload's device buffers and its step."""

    def __init__(self, w, device, torch, df2, conv):
        self.w, self.torch = w, torch
        bf = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(device).view(torch.bfloat16)
        self.x, self.z = bf(conv["x"]), bf(conv["z"])
        self.W_proj, self.base = bf(conv["W_proj"]), torch.from_numpy(conv["base"]).to(device)
        self.y, self.y2 = torch.empty_like(self.x), torch.empty_like(self.z)
        self.dyn = torch.empty((w.P, w.taps, w.G), dtype=torch.float32, device=device)
        self.ws = torch.empty(max(1, df2.conv_prepare_workspace_size(w.P, w.C, w.taps, w.g)), dtype=torch.uint8,
                              device=device)
        self.df2 = df2

    def run(self, ev=None):
        w, df2 = self.w, self.df2
        if ev is not None:
            ev[0].record()
        df2.conv_prepare(self.x, w.B, w.taps, w.g, self.W_proj, self.base, workspace=self.ws,
                         out=(self.y, self.dyn))
        if ev is not None:
            ev[1].record()
        df2.conv_finish(self.z, w.B, w.taps, w.g, self.dyn, self.base, out=self.y2)
        if ev is not None:
            ev[2].record()

    def host_outputs(self):
        torch = self.torch
        torch.cuda.synchronize()
        bits = lambda t: t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
        return {"y": bits(self.y), "dyn": self.dyn.cpu().numpy(), "y2": bits(self.y2)}


def conv_arm(args, w, rank, world, torch, df2, dist, device, conv, steps=None, warmup=None):
    """The training-packed conv workload: one step is conv_prepare then conv_finish
    over all P rows.  Events around each call give the live per-call durations: the
    prepare call against the tensor peak (its projection is the contraction), the
    finish call against HBM."""
    steps = args.steps if steps is None else steps
    warmup = args.warmup if warmup is None else warmup
    local = device.index
    cs = ConvStep(w, device, torch, df2, conv)
    x, z, y, y2, dyn = cs.x, cs.z, cs.y, cs.y2, cs.dyn
    for _ in range(warmup):
        cs.run()
    torch.cuda.synchronize()
    before = df2.kernels_launched()
    cs.run()
    torch.cuda.synchronize()
    n_launch = df2.kernels_launched() - before
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        soak(cs.run, torch, 1.0, 8)
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()
        launched0 = df2.kernels_launched()
        t0.record()
        for s in range(steps):
            cs.run(evs[s])
        t1.record()
        torch.cuda.synchronize()
    timed_launches = df2.kernels_launched() - launched0
    step_ms = slowest_rank_ms(t0.elapsed_time(t1) / steps, dist, device)
    prep_us = sum(e[0].elapsed_time(e[1]) for e in evs) / steps * 1e3
    fin_us = sum(e[1].elapsed_time(e[2]) for e in evs) / steps * 1e3

    # end to end: x and z in from pinned host memory, y, dyn_out and the finish output back
    pin = lambda t: torch.empty(t.shape, dtype=t.dtype).pin_memory()
    hx, hz = pin(x), pin(z)
    hx.copy_(x)
    hz.copy_(z)
    outs = [y, dyn, y2]
    houts = [pin(o) for o in outs]

    def e2e_step():
        x.copy_(hx, non_blocking=True)
        z.copy_(hz, non_blocking=True)
        cs.run()
        for o, ho in zip(outs, houts):
            ho.copy_(o, non_blocking=True)

    for _ in range(max(1, warmup)):
        e2e_step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        e2e_step()
    e1.record()
    torch.cuda.synchronize()
    e2e_ms = slowest_rank_ms(e0.elapsed_time(e1) / steps, dist, device)
    h2d = (x.numel() + z.numel()) * 2
    d2h = sum(o.numel() * o.element_size() for o in outs)
    clocks = with_clock_product(clk.summary(), step_ms)
    out = None
    if rank == 0:
        peaks, src = load_peaks()
        flops = 2.0 * w.P * w.C * (2 * w.taps * w.G)
        pk = peaks.get("bf16_tflops_sustained", peaks.get("bf16_tflops"))
        roof = {"kernel": "dflash2_conv_prepare call: conv_prepare_tc_kernel (the projection on the tensor cores, "
                          "dyn_out and the conv apply in its epilogue; one launch)", "bound": "tensor",
                "achieved": flops / (prep_us * 1e-6) / 1e12, "peak": pk, "unit": "TFLOP/s",
                "algorithmic_flops": flops,
                "traffic_note": "the kernel also applies the conv (x read again, y written), so its MMA rate is "
                                "below the contraction's own; traffic is the kernel's DRAM bytes per launch (ncu)"}
        fractions(roof, src)
        roof["traffic"], roof["traffic_source"] = head_traffic(w.name)
        fb = conv_bytes(w, "finish")
        roof_fin = {"kernel": "dflash2_conv_finish call: conv_apply_bulk_kernel", "bound": "hbm",
                    "achieved": fb / (fin_us * 1e-6) / 1e9, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                    "algorithmic_bytes": fb}
        fractions(roof_fin, src)
        roof_fin["traffic"], roof_fin["traffic_source"] = head_traffic("conv_finish")
        out = {
            "metric": METRIC, "value": job_throughput(w.P, world, step_ms), "unit": "positions/s",
            "n_gpus": world, "steps": steps, "warmup": warmup, "ms_per_step": step_ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded; shapes and scales of the workload, no dataset or checkpoint)",
            "config": conv_config(w),
            "per_call_us": {"conv_prepare": prep_us, "conv_finish": fin_us},
            "conv_gbs": {"prepare": conv_bytes(w, "prepare") / (prep_us * 1e-6) / 1e9,
                         "finish": fb / (fin_us * 1e-6) / 1e9},
            "roofline": roof, "roofline_finish": roof_fin,
            "e2e": {"value": job_throughput(w.P, world, e2e_ms), "unit": "positions/s",
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms},
            "gpu_launches": timed_launches, "kernels_per_step": n_launch, "execution": "eager calls",
            "clocks": clocks,
        }
    return out, cs


# ------------------------------------------------------------ oracle arm --

def oracle_requests(w):
    """Requests (anchor blocks for the conv workload) in the oracle's bounded
    sample: the first ones, about 8 LM-head rows of work per step, or 16 conv blocks."""
    if w.conv_only:
        return min(w.R, 16)
    rows_budget = 8
    return max(1, min(w.R, rows_budget // w.B if w.B <= rows_budget else 1))


def first_requests(w, inp, conv, n):
    """The workload's inputs cut to its first n requests (rows 0 .. n*B)."""
    rows = n * w.B
    ws = w.scaled(R=n)
    hi = None
    if inp is not None:
        hi = dict(inp)
        hi["h"] = np.ascontiguousarray(inp["h"][:rows])
        hi["pred"] = np.ascontiguousarray(inp["pred"][:rows])
        hi["anchors"] = np.ascontiguousarray(inp["anchors"][:n])
    ci = dict(conv)
    ci["x"] = np.ascontiguousarray(conv["x"][:rows])
    ci["z"] = np.ascontiguousarray(conv["z"][:rows])
    return ws, hi, ci


def oracle_step(orc, w, inp, conv):
    """The whole step on the CPU oracle for one draft batch (all P rows of w):
    conv prepare and finish, unary top-K with G, the walk and the teacher-forced
    scores.  Returns the outputs by name."""
    y, dyn = orc.conv_prepare(conv["x"], w.B, w.taps, w.g, conv["W_proj"], conv["base"])
    y2 = orc.conv_finish(conv["z"], w.B, w.taps, w.g, dyn, conv["base"])
    out = {"y": y, "dyn": dyn, "y2": y2}
    if w.conv_only:
        return out
    ids, vals, _, G = orc.unary_topk(inp["h"], inp["W_lm"], w.K, W_H=inp["W_H"])
    path, pscore, _, _ = orc.selector_walk(inp["anchors"], ids, vals, G, inp["A"], inp["Bc"], w.B)
    scores, _ = orc.pair_scores(inp["pred"], ids, vals, G, inp["A"], inp["Bc"])
    out.update(ids=ids, vals=vals, G=G, path=path, pscore=pscore, scores=scores)
    return out


def sample_text(w, n):
    if w.conv_only:
        return (f"{n} of {w.R} anchor blocks ({n * w.B} positions) per step: conv prepare (projection "
                f"{w.C} -> {2 * w.taps * w.G} in fp64) and conv finish on them")
    return (f"{n} of {w.R} requests ({n * w.B} positions) per step: the full step on them "
            f"(conv pair, {n * w.B} x {w.V} logits, full-sort top-{w.K}, walk, teacher-forced scores)")


def cpu_baseline(w, inp, conv, steps, warmup, one_thread_steps=1):
    """The oracle, as it stands, timed on the host cores on the workload's first
    requests: at every OpenMP thread (nproc) and, for one step, at one thread."""
    import oracle
    orc = oracle.default()
    n = oracle_requests(w)
    ws, hi, ci = first_requests(w, inp, conv, n)
    for _ in range(warmup):
        oracle_step(orc, ws, hi, ci)
    t = time.perf_counter()
    for _ in range(steps):
        oracle_step(orc, ws, hi, ci)
    dt = (time.perf_counter() - t) / max(1, steps)
    cores = orc.num_threads()
    rec = {"value": ws.P / dt, "unit": "positions/s", "cores": cores, "kind": "oracle",
           "sample": sample_text(w, n), "ms_per_step": dt * 1e3}
    if one_thread_steps:
        orc.set_num_threads(1)
        try:
            t = time.perf_counter()
            for _ in range(one_thread_steps):
                oracle_step(orc, ws, hi, ci)
            d1 = (time.perf_counter() - t) / one_thread_steps
        finally:
            orc.set_num_threads(cores)
        rec["one_thread"] = {"value": ws.P / d1, "unit": "positions/s", "cores": 1, "ms_per_step": d1 * 1e3,
                             "steps": one_thread_steps}
    return rec


def parity_block(w, inp, conv, gpu_out):
    """The timed step's outputs against the oracle on the same first requests the
    cpu baseline runs: compared / flagged / mismatched positions and every float
    and bf16 output within the tolerances (tests/parity.py)."""
    import oracle
    from parity import compare_chain
    orc = oracle.default()
    n = oracle_requests(w)
    s = compare_chain(orc, w, inp, gpu_out, range(n), conv=conv, check=False)
    s["sample"] = sample_text(w, n)
    s["rules"] = ("ids exact outside oracle margins < 1e-3 (flagged); mismatches flagged and <= 0.1% of "
                  "compared; floats within 2e-3 of max(|ref|, row rms); bf16 within that or one step")
    return s


def reference_arm(args, w):
    """--impl reference: the CPU oracle timed on the host cores on bounded samples of
    the workload (the pages hold no runnable implementation of the method)."""
    inp = None if w.conv_only else W.head_inputs(w)
    conv = W.conv_inputs(w)
    cpu = cpu_baseline(w, inp, conv, args.steps, max(0, args.warmup), one_thread_steps=0)
    value = cpu["value"]
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": "positions/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": cpu["ms_per_step"], "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": conv_config(w) if w.conv_only else config_of(w),
            "cpu_baseline": {k: cpu[k] for k in ("value", "unit", "cores", "kind", "sample")},
            "e2e": {"value": value, "unit": "positions/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


# The records that follow the headline in a default run: the other full-size
# workloads, each with its own timing, roofline, cpu baseline, parity and clocks.
RECORD_STEPS = {"batched": 200, "stress": 60, "conv": 500, "batch1": 2000}


def run_workload(args, w, rank, world, torch, df2, dist, device, steps, warmup, cpu_ok):
    inp = None if w.conv_only else W.head_inputs(w)
    conv = W.conv_inputs(w)
    cpu = cpu_baseline(w, inp, conv, steps=2, warmup=0) if cpu_ok else None
    if w.conv_only:
        out, st = conv_arm(args, w, rank, world, torch, df2, dist, device, conv, steps, warmup)
    else:
        out, st = gpu_arm(args, w, rank, world, torch, df2, dist, device, inp, conv, steps, warmup)
    if rank == 0:
        out["cpu_baseline"] = cpu
        if cpu_ok:
            out["parity"] = parity_block(w, inp, conv, st.host_outputs())
    del st
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    # default: 2000 device steps for the headline (about half a second timed); 5
    # steps for the reference arm, whose every step is a bounded CPU sample
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="batch1", choices=[c.name for c in W.CONFIGS])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-records", action="store_true",
                    help="only the headline workload (by default batch1 is followed by batched, stress, conv)")
    args = ap.parse_args()
    steps_given = args.steps is not None
    if args.steps is None:
        args.steps = 5 if args.impl == "reference" else RECORD_STEPS.get(args.workload, 200)
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    w = W.BY_NAME[args.workload]

    if args.impl == "reference":
        if rank != 0:
            return
        print(json.dumps(reference_arm(args, w)), flush=True)
        return

    import torch
    import dflash2_draft_block_gb300 as df2
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)
    cpu_ok = rank == 0 and world == 1 and not args.no_cpu_baseline
    out = run_workload(args, w, rank, world, torch, df2, dist, device, args.steps, args.warmup, cpu_ok)
    records = [] if (args.no_records or w.name != "batch1") else ["batched", "stress", "conv"]
    if records and rank == 0:
        out["workloads"] = {}
    for name in records:
        wr = W.BY_NAME[name]
        steps = args.steps if steps_given else RECORD_STEPS[name]
        rec = run_workload(args, wr, rank, world, torch, df2, dist, device, steps, args.warmup, cpu_ok)
        if rank == 0:
            for k in ("metric", "n_gpus", "higher_is_better", "scaling", "vs_baseline", "data"):
                rec.pop(k, None)
            out["workloads"][name] = rec
    if dist is not None:
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(out), flush=True)


if __name__ == "__main__":
    main()
