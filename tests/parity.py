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


def compare_topk(gpu_ids, gpu_vals, ref_ids, ref_vals, ref_margin, what="topk", logit_of=None) -> Report:
    """Row by row under the flagged-margin rule.  ``logit_of(p, ids)``, when given,
    returns the oracle's logits of those ids in row p: an id the GPU keeps and the
    oracle does not must then have an oracle logit within MARGIN of the oracle's K-th
    value (a real near-tie) and a GPU value within the float rule of that logit.
    Without it, the GPU's own value for such an id is taken."""
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
            foreign = [(j, i) for j, i in enumerate(gpu_ids[p].tolist()) if i not in rs]
            if logit_of is not None and foreign:
                true = np.asarray(logit_of(p, [i for _, i in foreign]), np.float64)
                rms = float(np.sqrt(np.mean(rv * rv)))
                for (j, _), u in zip(foreign, true):
                    if not abs(u - rv[-1]) < MARGIN:
                        explained = False
                    if not abs(float(gpu_vals[p][j]) - u) <= FTOL * max(abs(u), rms) + 1e-30:
                        explained = False
            else:
                for j, _ in foreign:
                    if abs(float(gpu_vals[p][j]) - rv[-1]) >= MARGIN:
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
        # the float rule's floor: the rms of the request's path scores
        row = np.asarray(ref_score[q], np.float64)
        rms = float(np.sqrt(np.mean(row * row))) if T else 0.0
        for t in range(T):
            rep.compared += 1
            if ref_margin[q, t] < MARGIN:
                rep.flagged += 1
            if gpu_path[q, t] == ref_path[q, t]:
                ref = float(ref_score[q, t])
                if not abs(float(gpu_score[q, t]) - ref) <= FTOL * max(abs(ref), rms) + 1e-30:
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


# ------------------------------------------------------- one whole draft batch --

def request_rows(requests, block):
    """Row indices of whole requests (anchor blocks) in a [R*B, ...] tensor."""
    requests = np.asarray(requests, np.int64)
    return (requests[:, None] * block + np.arange(block)[None, :]).reshape(-1)


def oracle_rows_topk(orc, w, inp, rows):
    """The oracle's top-K and G on the given rows: (rows, ids, vals, margin, G)."""
    rows = np.asarray(rows, np.int64)
    oi, ov, om, oG = orc.unary_topk(np.ascontiguousarray(inp["h"][rows]), inp["W_lm"], w.K, W_H=inp["W_H"])
    return rows, oi, ov, om, oG


def chain_rows(w, requests, extra_rows=()):
    req = np.asarray(sorted(set(int(q) for q in requests)), np.int64)
    return np.asarray(sorted(set(request_rows(req, w.B).tolist()) | set(int(e) for e in extra_rows)), np.int64)


def compare_chain(orc, w, inp, gpu, requests, extra_rows=(), conv=None, check=True, ref_topk=None):
    """The GPU outputs of one draft batch against the oracle's chain.

    ``gpu`` holds full-size host arrays: ids/vals [P,K], G [P,r], path/pscore
    [R,B-1], optionally scores [P,K] (teacher-forced) and, with ``conv``, y/dyn/y2.
    Whole ``requests`` are compared through every step; ``extra_rows`` are single
    rows compared for the top-K and G only.

    Top-K: the oracle on the same rows (compare_topk's flagged-margin rule, with the
    oracle's logit of every token only the GPU kept).  Walk: the oracle's walk over
    its own candidate lists where a request's lists equal the GPU's; where a flagged
    near-tie changed a list, over the GPU's candidate ids with the oracle's logits of
    them (the walk is then judged on the candidates it was given), and in both cases
    the GPU path must be greedy under the oracle's scores of those lists.  No GPU
    value is an input of the oracle: its G, logits and scores are its own.  Teacher-forced
    scores: the oracle's scorer on the same lists.  Conv: the oracle on the
    requests' anchor blocks (the conv never reads across a block), finish on the
    oracle's own correction.

    ``ref_topk`` may pass in oracle_rows_topk(...) of exactly these rows (the
    expensive part), to compare several GPU runs against one oracle pass.

    Returns a summary dict whose "failures" lists every rule broken; with
    ``check`` the call asserts that there are none."""
    B = w.B
    failures = []

    def rule(fn, *a, **k):
        try:
            fn(*a, **k)
        except AssertionError as e:
            failures.append(str(e)[:300])

    req = np.asarray(sorted(set(int(q) for q in requests)), np.int64)
    rrows = request_rows(req, B)
    summary = {"requests_compared": int(req.size)}
    if not w.conv_only:
        K = w.K
        rows = chain_rows(w, req, extra_rows)
        gi, gv, gG = gpu["ids"], gpu["vals"], gpu["G"]
        if ref_topk is None:
            ref_topk = oracle_rows_topk(orc, w, inp, rows)
        assert np.array_equal(ref_topk[0], rows), "ref_topk was computed on other rows"
        _, oi, ov, om, oG = ref_topk
        def logit_of(k, ids):
            # the oracle's logits of single ids in compared row k
            h_row = np.ascontiguousarray(inp["h"][rows[k]][None, :])
            return orc.logits(h_row, np.ascontiguousarray(inp["W_lm"][np.asarray(ids, np.int64)]))[0]

        topk = compare_topk(gi[rows], gv[rows], oi, ov, om, w.name, logit_of=logit_of)
        summary["topk"] = {"compared": topk.compared, "flagged": topk.flagged, "mismatched": topk.mismatched,
                           "unexplained": len(topk.unexplained)}
        rule(topk.check, w.name + " topk")
        rule(compare_topk_values, gi[rows], gv[rows], oi, ov, w.name + " vals")
        # the largest deviation of a kept logit from the oracle's, relative to
        # max(|logit|, 1), where the ids agree
        same = gi[rows] == oi
        if same.any():
            err = np.abs(gv[rows].astype(np.float64) - ov) / np.maximum(np.abs(ov.astype(np.float64)), 1.0)
            summary["topk"]["max_val_rel_err"] = float(err[same].max())
        rule(close, gG[rows], oG, what=w.name + " G")
        if req.size:
            # the lists the oracle's walk and scorer run on: the oracle's own where
            # the request's lists match the GPU's, the GPU's ids otherwise (a flagged
            # near-tie changed them), always with the oracle's logits of those ids
            # and the oracle's G, so no GPU value enters the oracle
            at = {int(p): k for k, p in enumerate(rows)}
            k_of = np.asarray([at[int(p)] for p in rrows])
            same_req = np.all((gi[rrows] == oi[k_of]).reshape(req.size, -1), axis=1)
            same_rows = np.repeat(same_req, B)[:, None]
            c_ids = np.ascontiguousarray(np.where(same_rows, oi[k_of], gi[rrows]), np.int32)
            c_vals = np.array(ov[k_of], np.float32)
            for n in np.nonzero(~same_rows[:, 0])[0]:
                c_vals[n] = logit_of(k_of[n], c_ids[n])
            c_vals = np.ascontiguousarray(c_vals)
            c_G = np.ascontiguousarray(oG[k_of], np.float32)
            anchors = np.ascontiguousarray(inp["anchors"][req])
            op, os_, omg, st = orc.selector_walk(anchors, c_ids, c_vals, c_G, inp["A"], inp["Bc"], B)
            gpath = np.ascontiguousarray(gpu["path"][req])
            walk = compare_walk(gpath, gpu["pscore"][req], op, os_, omg, w.name + " walk")
            summary["walk"] = {"compared": walk.compared, "flagged": walk.flagged, "mismatched": walk.mismatched,
                               "unexplained": len(walk.unexplained),
                               "requests_on_gpu_lists": int((~same_req).sum())}
            if st != 0:
                failures.append(f"oracle walk status {st}")
            rule(walk.check, w.name + " walk")
            rule(check_path_valid, orc, gpath, anchors, c_ids, c_vals, c_G, inp["A"], inp["Bc"], B)
            if gpu.get("scores") is not None:
                osc, st = orc.pair_scores(np.ascontiguousarray(inp["pred"][rrows]), c_ids, c_vals, c_G,
                                          inp["A"], inp["Bc"])
                summary["teacher_forced_rows"] = int(rrows.size)
                if st != 0:
                    failures.append(f"oracle teacher-forced status {st}")
                rule(close, gpu["scores"][rrows], osc, what=w.name + " teacher-forced scores")
    if conv is not None and gpu.get("y") is not None and req.size:
        x, z = np.ascontiguousarray(conv["x"][rrows]), np.ascontiguousarray(conv["z"][rrows])
        oy, od = orc.conv_prepare(x, B, w.taps, w.g, conv["W_proj"], conv["base"])
        oy2 = orc.conv_finish(z, B, w.taps, w.g, od, conv["base"])
        summary["conv_rows"] = int(rrows.size)
        rule(close, gpu["dyn"][rrows], od, what=w.name + " dyn_out")
        cmp = close_bf16 if x.dtype == np.uint16 else close
        rule(cmp, gpu["y"][rrows], oy, what=w.name + " conv y")
        rule(cmp, gpu["y2"][rrows], oy2, what=w.name + " conv finish")
    summary["failures"] = failures
    summary["ok"] = not failures
    if check:
        assert not failures, failures
    return summary
