"""Comparators between the CUDA path and the oracle, with the flagged-margin rules.

Rules (the same for every test):
- token ids (top-K lists and walk paths) must equal the oracle's exactly, except
  where the oracle's own decision margin is below MARGIN (K-th vs (K+1)-th
  logit for top-K, best vs second score for the walk; also adjacent in-list
  values for the order inside a top-K list).  Such positions are *flagged*;
  every mismatch must be flagged, and mismatches must stay below 0.1% of the
  positions compared.
- float outputs: |gpu - oracle| <= FTOL * max(|oracle|, rms(oracle row)), the
  row-rms floor keeping near-zero entries from blowing up a relative error.
- bf16 outputs: the float rule, or at most one bf16 step apart (two fp32 sums in
  different orders may round to neighbouring bf16 values).
"""
from __future__ import annotations

import dataclasses

import numpy as np

MARGIN = 1e-3
FTOL = 2e-3
MAX_MISMATCH_FRAC = 1e-3


@dataclasses.dataclass
class Report:
    compared: int = 0
    flagged: int = 0
    mismatched: int = 0
    unexplained: list = dataclasses.field(default_factory=list)

    def check(self, what=""):
        assert not self.unexplained, f"{what}: unflagged mismatches {self.unexplained[:5]}"
        if self.compared:
            assert self.mismatched <= max(0, MAX_MISMATCH_FRAC * self.compared) or self.mismatched == 0, (
                f"{what}: {self.mismatched}/{self.compared} mismatched positions")


def close(gpu, ref, ftol=FTOL, what=""):
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    assert gpu.shape == ref.shape, (what, gpu.shape, ref.shape)
    if ref.size == 0:
        return
    r2 = ref.reshape(ref.shape[0], -1) if ref.ndim > 1 else ref.reshape(1, -1)
    g2 = gpu.reshape(r2.shape)
    rms = np.sqrt(np.mean(r2 * r2, axis=1, keepdims=True))
    bound = ftol * np.maximum(np.abs(r2), rms) + 1e-30
    bad = ~(np.abs(g2 - r2) <= bound)
    assert not bad.any(), (f"{what}: {bad.sum()} of {bad.size} values outside tolerance; first "
                           f"{np.argwhere(bad)[:3].tolist()} gpu={g2[bad][:3]} ref={r2[bad][:3]}")


def close_bf16(gpu_bits, ref_bits, ftol=FTOL, what=""):
    from workloads import bf16_bits_to_f32
    g = np.asarray(gpu_bits).astype(np.int32)
    r = np.asarray(ref_bits).astype(np.int32)
    # bf16 bit patterns of finite numbers are ordered per sign; one step apart ==
    # |bits difference| <= 1 with equal signs
    same_sign = (g >> 15) == (r >> 15)
    one_step = same_sign & (np.abs(g - r) <= 1)
    gf = bf16_bits_to_f32(np.asarray(gpu_bits)).astype(np.float64)
    rf = bf16_bits_to_f32(np.asarray(ref_bits)).astype(np.float64)
    r2 = rf.reshape(rf.shape[0], -1)
    rms = np.sqrt(np.mean(r2 * r2, axis=1, keepdims=True))
    bound = ftol * np.maximum(np.abs(r2), rms)
    ok = one_step.reshape(r2.shape) | (np.abs(gf.reshape(r2.shape) - r2) <= bound)
    assert ok.all(), f"{what}: {(~ok).sum()} bf16 values outside tolerance"


def compare_topk(gpu_ids, gpu_vals, ref_ids, ref_vals, ref_margin, what="topk") -> Report:
    gpu_ids, ref_ids = np.asarray(gpu_ids), np.asarray(ref_ids)
    gpu_vals, ref_vals = np.asarray(gpu_vals), np.asarray(ref_vals)
    rep = Report()
    P, K = ref_ids.shape
    for p in range(P):
        rep.compared += 1
        rv = ref_vals[p].astype(np.float64)
        near_order = np.any(np.abs(np.diff(rv)) < MARGIN) if K > 1 else False
        boundary = ref_margin[p] < MARGIN
        if boundary or near_order:
            rep.flagged += 1
        if np.array_equal(gpu_ids[p], ref_ids[p]):
            continue
        rep.mismatched += 1
        gs, rs = set(gpu_ids[p].tolist()), set(ref_ids[p].tolist())
        explained = True
        # ids that both lists hold must sit at positions whose oracle values are
        # within MARGIN of each other
        pos_ref = {int(i): j for j, i in enumerate(ref_ids[p])}
        for j, i in enumerate(gpu_ids[p].tolist()):
            if i in pos_ref and pos_ref[i] != j:
                if abs(rv[pos_ref[i]] - rv[min(j, K - 1)]) >= MARGIN:
                    explained = False
        if gs != rs:
            # a set change is allowed only at a flagged K/K+1 boundary, and only
            # for ids whose values sit within MARGIN of the oracle's K-th value
            if not boundary:
                explained = False
            for j, i in enumerate(gpu_ids[p].tolist()):
                if i not in rs and abs(float(gpu_vals[p][j]) - rv[-1]) >= MARGIN:
                    explained = False
        if not explained:
            rep.unexplained.append((what, p, gpu_ids[p][:8].tolist(), ref_ids[p][:8].tolist()))
    return rep


def compare_topk_values(gpu_ids, gpu_vals, ref_ids, ref_vals, what="topk vals"):
    """Values compared where the ids agree position by position."""
    gpu_ids, ref_ids = np.asarray(gpu_ids), np.asarray(ref_ids)
    same = gpu_ids == ref_ids
    g = np.where(same, gpu_vals, ref_vals)
    close(g, ref_vals, what=what)


def compare_walk(gpu_path, gpu_score, ref_path, ref_score, ref_margin, what="walk") -> Report:
    """Position by position up to the first divergence; a divergence must sit at
    a flagged position (later positions then have other predecessors and are
    checked by check_path_valid instead)."""
    rep = Report()
    R, T = ref_path.shape
    for q in range(R):
        for t in range(T):
            rep.compared += 1
            if ref_margin[q, t] < MARGIN:
                rep.flagged += 1
            if gpu_path[q, t] == ref_path[q, t]:
                ref = float(ref_score[q, t])
                if not abs(float(gpu_score[q, t]) - ref) <= FTOL * max(abs(ref), 1.0):
                    rep.unexplained.append((what, "score", q, t, float(gpu_score[q, t]), ref))
                continue
            rep.mismatched += 1
            if not ref_margin[q, t] < MARGIN:
                rep.unexplained.append((what, "path", q, t, int(gpu_path[q, t]), int(ref_path[q, t])))
            break
    return rep


def check_path_valid(orc, gpu_path, anchors, ids, vals, G, A, Bc, block):
    """The GPU path is a greedy path under the oracle's scores: replayed through the
    oracle's teacher-forced scorer, each chosen token is the oracle's best choice or
    within MARGIN of it."""
    R = anchors.shape[0]
    pred = np.concatenate([anchors[:, None], anchors[:, None], gpu_path[:, :-1]], axis=1)
    pred = np.ascontiguousarray(pred.reshape(-1).astype(np.int32))
    scores, _ = orc.pair_scores(pred, ids, vals, G, A, Bc)
    K = ids.shape[-1]
    scores = scores.reshape(R, block, K)
    idsr = ids.reshape(R, block, K)
    bad = []
    for q in range(R):
        for t in range(1, block):
            chosen = int(gpu_path[q, t - 1])
            js = np.nonzero(idsr[q, t] == chosen)[0]
            if js.size == 0:
                bad.append((q, t, "not a candidate"))
                continue
            if scores[q, t, js[0]] < scores[q, t].max() - MARGIN:
                bad.append((q, t, float(scores[q, t, js[0]]), float(scores[q, t].max())))
    assert not bad, f"GPU path not greedy under oracle scores: {bad[:5]}"
