"""Pins for the CPU oracle: checks against what the pages and the mathematics fix.

Each ``pin_*`` function takes an ``oracle.Oracle`` and raises ``AssertionError``
when the oracle disagrees with a closed form, a stated invariant, a hand-worked
golden case or brute force.  None of them re-types the oracle's own loops: they
use exact small-integer arithmetic, special cases whose answer is known without
running the method, and properties that characterise the unique answer.

``tests/test_oracle_pins.py`` runs every pin on the oracle; ``tests/test_oracle_mutants.py``
plants plausible mistakes in copies of the oracle source and checks that each one
fails at least one pin.
"""
from __future__ import annotations

import json
import math
import os
import zlib

import numpy as np

from workloads import bf16_bits_to_f32, f32_to_bf16_bits

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def bf(a):
    """Exact-in-bf16 floats -> bf16 bits (asserts exactness)."""
    a = np.asarray(a, np.float32)
    b = f32_to_bf16_bits(a)
    assert np.array_equal(bf16_bits_to_f32(b), a), "fixture value not exact in bf16"
    return b


def _rng(tag):
    return np.random.default_rng(zlib.crc32(tag.encode()))


# ------------------------------------------------------------- logits (o1) --

def pin_logits_one_hot(o):
    """h = e_d selects column d of W_lm exactly: U[v] = W_lm[v, d]."""
    rng = _rng("one_hot")
    V, D = 37, 24
    W = f32_to_bf16_bits(rng.standard_normal((V, D)).astype(np.float32))
    h = np.zeros((D, D), np.float32)
    np.fill_diagonal(h, 1.0)
    U = o.logits(bf(h), W)
    assert np.array_equal(U, bf16_bits_to_f32(W).T)


def pin_logits_permutation(o):
    """W_lm a permuted identity: U[p, v] = h[p, perm[v]] exactly."""
    rng = _rng("perm")
    D = 16
    perm = rng.permutation(D)
    W = np.zeros((D, D), np.float32)
    W[np.arange(D), perm] = 1.0
    h = f32_to_bf16_bits(rng.standard_normal((3, D)).astype(np.float32))
    U = o.logits(h, bf(W))
    assert np.array_equal(U, bf16_bits_to_f32(h)[:, perm])


def pin_logits_integer_exact(o):
    """Small-integer operands: every sum is an exact integer (brute force with Python ints)."""
    rng = _rng("int")
    P, V, D = 3, 11, 29
    h = rng.integers(-8, 9, size=(P, D))
    W = rng.integers(-8, 9, size=(V, D))
    U = o.logits(bf(h), bf(W))
    for p in range(P):
        for v in range(V):
            exact = sum(int(h[p, d]) * int(W[v, d]) for d in range(D))
            assert U[p, v] == exact, (p, v, U[p, v], exact)


def pin_logits_within_rounding(o):
    """Random bf16 operands, D = 4096: the result is within one fp32 ulp of the
    exactly rounded sum (products of bf16 values are exact; math.fsum sums exactly)."""
    rng = _rng("fsum")
    D = 4096
    h = f32_to_bf16_bits(rng.standard_normal((2, D)).astype(np.float32))
    W = f32_to_bf16_bits((rng.standard_normal((5, D)) * 0.02).astype(np.float32))
    U = o.logits(h, W)
    hf, Wf = bf16_bits_to_f32(h).astype(np.float64), bf16_bits_to_f32(W).astype(np.float64)
    for p in range(2):
        for v in range(5):
            exact = np.float32(math.fsum(hf[p] * Wf[v]))
            assert abs(float(U[p, v]) - float(exact)) <= float(np.spacing(np.abs(exact))), (U[p, v], exact)


# -------------------------------------------------------------- top-K (o2) --

def pin_topk_golden(o):
    g = _golden("topk_ties.json")
    h, W = bf(g["h"]), bf(g["W_lm"])
    for case in g["cases"]:
        ids, vals, margin, _ = o.unary_topk(h, W, case["K"])
        assert ids[0].tolist() == case["ids"], (ids, case)
        assert vals[0].tolist() == case["vals"]
        want = math.inf if case["margin"] == "inf" else case["margin"]
        assert margin[0] == want


def _check_topk_properties(U, ids, vals, margin, K):
    """The unique top-K: distinct ids; every kept (value, id) ranks above every
    dropped one; listed in rank order; vals are the kept logits; margin is the gap
    between the K-th kept and the best dropped value."""
    V = U.shape[0]
    assert len(set(ids.tolist())) == K and ids.min() >= 0 and ids.max() < V
    assert np.array_equal(vals, U[ids])
    keys = [(-float(U[i]), int(i)) for i in ids]
    assert keys == sorted(keys)
    kept = set(ids.tolist())
    worst = keys[-1]
    dropped = [(-float(U[i]), i) for i in range(V) if i not in kept]
    assert all(worst < d for d in dropped)
    if dropped:
        assert margin == float(vals[-1]) - max(-d[0] for d in dropped)
    else:
        assert margin == math.inf


def pin_topk_brute_force(o):
    """Tiny vocabularies with many exact ties (small-integer logits, duplicate rows)."""
    rng = _rng("topk")
    for V, D, K in [(12, 3, 5), (40, 4, 7), (64, 2, 64), (9, 1, 1), (33, 5, 32)]:
        h = rng.integers(-2, 3, size=(4, D))
        W = rng.integers(-2, 3, size=(V, D))
        W[V // 2] = W[1]  # exact duplicate rows
        U = h @ W.T  # small integers: exact, independent of the oracle
        ids, vals, margin, _ = o.unary_topk(bf(h), bf(W), K)
        for p in range(4):
            _check_topk_properties(U[p].astype(np.float32), ids[p], vals[p], margin[p], K)


def pin_topk_k_equals_v(o):
    rng = _rng("kv")
    V, D = 50, 8
    h = f32_to_bf16_bits(rng.standard_normal((2, D)).astype(np.float32))
    W = f32_to_bf16_bits(rng.standard_normal((V, D)).astype(np.float32))
    ids, vals, margin, _ = o.unary_topk(h, W, V)
    for p in range(2):
        assert sorted(ids[p].tolist()) == list(range(V))
        assert margin[p] == math.inf
        assert np.all(np.diff(vals[p]) <= 0)


def pin_topk_hidden_projection(o):
    """G = H(h): with W_H = I (r = D) G equals h; with integer operands it is exact."""
    rng = _rng("G")
    D = 12
    h = rng.integers(-4, 5, size=(3, D))
    WH = rng.integers(-3, 4, size=(5, D))
    W = rng.integers(-3, 4, size=(7, D))
    _, _, _, G = o.unary_topk(bf(h), bf(W), 2, W_H=bf(WH))
    assert np.array_equal(G, (h @ WH.T).astype(np.float32))
    _, _, _, G2 = o.unary_topk(bf(h), bf(W), 2, W_H=bf(np.eye(D)))
    assert np.array_equal(G2, h.astype(np.float32))


# ------------------------------------------- logit multiplier / softcap --
# The pages name an optional output multiplier m and a final logit softcap c
# applied to the unary logits; the reading pinned here is u -> c*tanh(m*u/c)
# (m*u when c = 0), the multiplier first and the cap last.

def pin_softcap_worked_values(o):
    """tanh(ln(3)/2) = 1/2 exactly, so with m = ln 3 and c = 2 a logit of 1 maps to
    1; halving the argument gives 2*(2 - sqrt 3); quartering it 2*(3^(1/4) - 1)/(3^(1/4) + 1);
    the map is odd.  h = e_0 puts the chosen logits in column 0 of W_lm."""
    col = [0.25, -1.0, 0.5, 0.0, -0.5, 1.0]
    V, D = len(col), 4
    W = np.zeros((V, D), np.float32)
    W[:, 0] = col
    h = np.zeros((1, D), np.float32)
    h[0, 0] = 1.0
    ids, vals, margin, _ = o.unary_topk(bf(h), bf(W), V, output_multiplier=math.log(3.0),
                                        final_logit_softcapping=2.0)
    q = 3.0 ** 0.25
    half, quarter = 4.0 - 2.0 * math.sqrt(3.0), 2.0 * (q - 1.0) / (q + 1.0)
    assert ids[0].tolist() == [5, 2, 0, 3, 4, 1], ids
    want = [1.0, half, quarter, 0.0, -half, -1.0]
    assert np.allclose(vals[0].astype(np.float64), want, rtol=0, atol=1e-6), (vals, want)
    assert margin[0] == math.inf


def pin_softcap_saturates_before_selection(o):
    """m*u/c >= 32 for every logit: tanh rounds to exactly 1 in double precision,
    every mapped logit equals c, and the top-K falls to the tie rule: the K lowest
    token ids, whatever their raw order; margin 0.  Shows the cap is applied to all
    V logits before the selection, not to the K kept ones."""
    rng = _rng("saturate")
    V, D, K = 40, 4, 6
    W = np.zeros((V, D), np.float32)
    W[:, 1] = rng.integers(1, 9, size=V) * 0.25      # logits in [0.25, 2], exact in bf16
    h = np.zeros((2, D), np.float32)
    h[:, 1] = 1.0
    ids, vals, margin, _ = o.unary_topk(bf(h), bf(W), K, output_multiplier=64.0, final_logit_softcapping=0.5)
    for p in range(2):
        assert ids[p].tolist() == list(range(K)), ids[p]
        assert np.all(vals[p] == np.float32(0.5))
        assert margin[p] == 0.0
    assert np.argsort(-W[:, 1], kind="stable")[:K].tolist() != list(range(K))


def _series_softcap(x, c):
    """c*tanh(x/c) by its Taylor series in x/c (|x/c| <= 1/16 here: terms past the
    fourth are below 1e-9 of x)."""
    t = x / c
    return c * (t - t ** 3 / 3.0 + 2.0 * t ** 5 / 15.0 - 17.0 * t ** 7 / 315.0)


def pin_softcap_small_argument_series(o):
    """Exact logits (multiples of 1/4, computed with integers) and m*|u| <= 3 under
    a cap of 64: the values follow the tanh series, the ids follow the brute-force
    order of the raw logits (the map is increasing and keeps ties), and with no
    cap the values are m*u exactly."""
    rng = _rng("series")
    P, V, D, K = 3, 30, 8, 9
    h = rng.integers(-2, 3, size=(P, D))
    W = rng.integers(-2, 3, size=(V, D))
    U = (h @ W.T) * 0.25 * 0.5                       # exact: h/2 and W/4 as bf16 operands
    m, c = 0.375, 64.0
    ids, vals, _, _ = o.unary_topk(bf(h * 0.5), bf(W * 0.25), K, output_multiplier=m,
                                   final_logit_softcapping=c)
    ids0, vals0, _, _ = o.unary_topk(bf(h * 0.5), bf(W * 0.25), K, output_multiplier=m)
    for p in range(P):
        order = sorted(range(V), key=lambda v: (-U[p, v], v))[:K]
        assert ids[p].tolist() == order and ids0[p].tolist() == order
        x = m * U[p, order]
        assert np.allclose(vals[p].astype(np.float64), _series_softcap(x, c), rtol=0, atol=1e-6)
        assert np.array_equal(vals0[p], (x).astype(np.float32))
        assert np.all(np.abs(vals[p]) <= c)


def pin_softcap_rejects_bad_parameters(o):
    """The multiplier must be finite and positive, the cap finite and >= 0."""
    h = bf(np.eye(4)[:1])
    W = bf(np.eye(4))
    for m, c in [(0.0, 0.0), (-1.0, 0.0), (math.nan, 0.0), (math.inf, 1.0), (1.0, -1.0), (1.0, math.inf),
                 (1.0, math.nan)]:
        try:
            o.unary_topk(h, W, 2, output_multiplier=m, final_logit_softcapping=c)
        except ValueError:
            continue
        raise AssertionError(f"multiplier={m} softcap={c} accepted")


# ------------------------------------------------------------ walk (o3/o4) --

def _walk_fixture(o, name):
    g = _golden(name)
    K, r, B = g["K"], g["r"], g["block"]
    ids = np.asarray(g["ids"], np.int32)
    vals = np.asarray(g["vals"], np.float32)
    G = np.asarray(g["G"], np.float32)
    A, Bc = bf(g["A"]), bf(g["Bc"])
    anchors = np.asarray([g["anchor"]], np.int32)
    path, score, margin, status = o.selector_walk(anchors, ids, vals, G, A, Bc, B)
    return g, (ids, vals, G, A, Bc), (path, score, margin, status)


def pin_walk_golden(o):
    g, _, (path, score, margin, status) = _walk_fixture(o, "walk_r1_k2.json")
    assert status == 0
    assert path[0].tolist() == g["path"]
    assert score[0].tolist() == g["path_score"]
    assert margin[0].tolist() == g["margin"]


def pin_walk_tie_lower_id(o):
    g, _, (path, score, margin, status) = _walk_fixture(o, "walk_tie.json")
    assert path[0].tolist() == g["path"] and score[0].tolist() == g["path_score"]
    assert margin[0].tolist() == g["margin"]


def pin_pair_scores_golden(o):
    g, (ids, vals, G, A, Bc), _ = _walk_fixture(o, "walk_r1_k2.json")
    pred = np.asarray(g["teacher_forced_pred"], np.int32)
    scores, status = o.pair_scores(pred, ids, vals, G, A, Bc)
    assert status == 0
    assert scores.tolist() == g["teacher_forced_scores"]


# ---------------------------------------------------------------- selector CE --
# The selector's K-way cross-entropy of teacher-forced scores against the ground
# truth, on rows whose ground truth is a candidate (verl-SpeCo PR #62, "Selector
# training objective"; vLLM Speculators "DFlash2" guide, "Training Objective").

def pin_ce_single_candidate_is_zero(o):
    """With one candidate that is the target, the cross-entropy is exactly 0."""
    scores = np.array([[3.5], [-7.25], [0.0]], np.float32)
    ids = np.array([[4], [9], [2]], np.int32)
    loss, label, st = o.selector_ce(scores, ids, np.array([4, 9, 2], np.int32), 10)
    assert st == 0 and label.tolist() == [0, 0, 0]
    assert loss.tolist() == [0.0, 0.0, 0.0]


def pin_ce_uniform_scores_is_log_k(o):
    """Equal scores over K candidates: the softmax is uniform, the loss is ln K."""
    for K in (2, 3, 16, 64, 1000):
        for c in (-5.0, 0.0, 12.5):
            scores = np.full((1, K), c, np.float32)
            ids = np.arange(K, dtype=np.int32)[None] * 3
            loss, label, _ = o.selector_ce(scores, ids, np.array([3 * (K // 2)], np.int32), 3 * K)
            assert label[0] == K // 2
            assert abs(float(loss[0]) - math.log(K)) <= 1e-6 * math.log(K), (K, c, loss[0])


def pin_ce_two_candidates_is_softplus(o):
    """K = 2: -log sigmoid(s_label - s_other) = softplus(s_other - s_label)."""
    rng = _rng("ce_two")
    for _ in range(50):
        a, b = (rng.standard_normal(2) * 6).astype(np.float32)
        loss, label, _ = o.selector_ce(np.array([[a, b]], np.float32), np.array([[7, 1]], np.int32),
                                       np.array([1], np.int32), 8)
        d = float(a) - float(b)
        want = d + math.log1p(math.exp(-d)) if d > 0 else math.log1p(math.exp(d))
        assert label[0] == 1 and abs(float(loss[0]) - want) <= 1e-6 * max(1.0, want), (a, b, loss[0], want)


def pin_ce_hand_worked(o):
    """Scores 1, 2, 3, 4 with the target in the second column:
    log(e + e^2 + e^3 + e^4) - 2 = 2 + log(1 + e^-1 + e^-2 + e^-3)."""
    loss, label, _ = o.selector_ce(np.array([[1, 2, 3, 4]], np.float32), np.array([[10, 20, 30, 40]], np.int32),
                                   np.array([20], np.int32), 50)
    want = 2.0 + math.log(1.0 + math.exp(-1.0) + math.exp(-2.0) + math.exp(-3.0))
    assert label[0] == 1 and abs(float(loss[0]) - want) <= 1e-6


def pin_ce_invariances(o):
    """A constant added to a row's scores leaves its loss unchanged; permuting the
    candidates (ids with their scores) leaves it unchanged and moves the label."""
    rng = _rng("ce_inv")
    P, K, V = 20, 16, 500
    scores = rng.integers(-40, 40, size=(P, K)).astype(np.float32) / 4
    ids = np.stack([rng.choice(V, size=K, replace=False) for _ in range(P)]).astype(np.int32)
    targets = ids[np.arange(P), rng.integers(0, K, size=P)]
    loss, label, _ = o.selector_ce(scores, ids, targets, V)
    loss2, label2, _ = o.selector_ce(scores + 64.0, ids, targets, V)  # exact in fp32
    assert np.array_equal(label, label2) and np.allclose(loss, loss2, rtol=1e-6, atol=1e-6)
    perm = rng.permutation(K)
    loss3, label3, _ = o.selector_ce(scores[:, perm], ids[:, perm], targets, V)
    assert np.allclose(loss, loss3, rtol=1e-6, atol=1e-6)
    assert np.array_equal(perm[label3], label)
    assert np.all(loss >= 0)  # -log of a probability


def pin_ce_rows_without_a_candidate_target(o):
    """A target outside the row's candidates (or no target, < 0) contributes nothing:
    label -1 and NaN loss, no status; a target id >= V is also flagged."""
    scores = np.zeros((4, 3), np.float32)
    ids = np.array([[1, 2, 3]] * 4, np.int32)
    loss, label, st = o.selector_ce(scores, ids, np.array([5, -1, 2, 3], np.int32), 10)
    assert label.tolist() == [-1, -1, 1, 2] and st == 0
    assert np.isnan(loss[0]) and np.isnan(loss[1]) and loss[2] == loss[3]
    loss, label, st = o.selector_ce(scores, ids, np.array([10, 1, 1, 1], np.int32), 10)
    assert st & 1 and label[0] == -1 and np.isnan(loss[0]) and label[1] == 0


def _random_lattice(tag, R, B, K, V, r, cb_std=1.0, G_std=1.0):
    rng = _rng(tag)
    ids = np.stack([np.stack([rng.choice(V, size=K, replace=False) for _ in range(B)]) for _ in range(R)])
    vals = -np.sort(-rng.standard_normal((R, B, K)).astype(np.float32), axis=-1)
    G = (rng.standard_normal((R, B, r)) * G_std).astype(np.float32)
    A = f32_to_bf16_bits((rng.standard_normal((V, r)) * cb_std).astype(np.float32))
    Bc = f32_to_bf16_bits((rng.standard_normal((V, r)) * cb_std).astype(np.float32))
    anchors = rng.integers(0, V, size=R).astype(np.int32)
    return (anchors, ids.reshape(R * B, K).astype(np.int32), vals.reshape(R * B, K), G.reshape(R * B, r),
            A, Bc)


def pin_walk_zero_successor_is_unary(o):
    """A zero successor codebook leaves the unary scores (SpecForge DFlash2 concept doc,
    'Architecture'): the path is each row's unary argmax (lower id on ties) and the
    path score its unary logit."""
    anchors, ids, vals, G, A, _ = _random_lattice("zeroB", 5, 6, 8, 97, 16)
    Bc = np.zeros_like(A)
    vals[3, 2] = vals[3, 0]  # an exact unary tie
    path, score, _, _ = o.selector_walk(anchors, ids, vals, G, A, Bc, 6)
    for q in range(5):
        for t in range(1, 6):
            row = q * 6 + t
            best = max(range(8), key=lambda j: (vals[row, j], -ids[row, j]))
            assert path[q, t - 1] == ids[row, best]
            assert score[q, t - 1] == vals[row, best]


def pin_walk_k1_is_top1(o):
    anchors, ids, vals, G, A, Bc = _random_lattice("k1", 4, 5, 1, 60, 8)
    path, score, margin, _ = o.selector_walk(anchors, ids, vals, G, A, Bc, 5)
    assert np.array_equal(path, ids.reshape(4, 5)[:, 1:])
    assert np.all(np.isinf(margin))


def pin_walk_unit_codebooks_closed_form(o):
    """A = B = 1: S_t(a, b) = U_t(b) + sum_i G_t[i] for every predecessor; integer
    G and unary values keep every score exact."""
    rng = _rng("ones")
    R, B, K, V, r = 3, 5, 4, 30, 6
    anchors, ids, _, _, _, _ = _random_lattice("ones", R, B, K, V, r)
    vals = rng.integers(-6, 7, size=(R * B, K)).astype(np.float32)
    G = rng.integers(-3, 4, size=(R * B, r)).astype(np.float32)
    one = bf(np.ones((V, r)))
    path, score, _, _ = o.selector_walk(anchors, ids, vals, G, one, one, B)
    scores, _ = o.pair_scores(np.zeros(R * B, np.int32), ids, vals, G, one, one)
    want = vals + G.sum(axis=1, keepdims=True)
    assert np.array_equal(scores, want)
    for q in range(R):
        for t in range(1, B):
            row = q * B + t
            best = max(range(K), key=lambda j: (want[row, j], -ids[row, j]))
            assert path[q, t - 1] == ids[row, best] and score[q, t - 1] == want[row, best]


def pin_walk_replay_matches_teacher_forced(o):
    """Replaying the walk's own predecessors through the teacher-forced scorer gives
    back the same path and scores (verl-SpeCo PR #62, 'Selector training objective')."""
    R, B, K, V, r = 6, 8, 5, 80, 12
    anchors, ids, vals, G, A, Bc = _random_lattice("replay", R, B, K, V, r)
    path, score, _, _ = o.selector_walk(anchors, ids, vals, G, A, Bc, B)
    pred = np.concatenate([anchors[:, None], anchors[:, None], path[:, :-1]], axis=1).reshape(-1)
    scores, _ = o.pair_scores(pred.astype(np.int32), ids, vals, G, A, Bc)
    scores = scores.reshape(R, B, K)
    idsr = ids.reshape(R, B, K)
    for q in range(R):
        for t in range(1, B):
            j = max(range(K), key=lambda jj: (scores[q, t, jj], -idsr[q, t, jj]))
            assert idsr[q, t, j] == path[q, t - 1]
            assert scores[q, t, j] == score[q, t - 1]


def pin_walk_feeds_back_choice(o):
    """The predecessor at row t is the token chosen at row t-1: changing only the
    row-1 unary values so that a different token is picked changes row 2's scores
    as the pair-score formula says (checked with the fixture's exact numbers)."""
    g = _golden("walk_r1_k2.json")
    ids = np.asarray(g["ids"], np.int32)
    vals = np.asarray(g["vals"], np.float32).copy()
    vals[1] = [10.0, 0.5]  # now token 0 wins row 1: S(1,0) = 12.0 > S(1,2) = 4.5
    path, score, _, _ = o.selector_walk(np.asarray([g["anchor"]], np.int32), ids, vals,
                                        np.asarray(g["G"], np.float32), bf(g["A"]), bf(g["Bc"]), 3)
    assert path[0].tolist() == [0, 3] and score[0].tolist() == [12.0, 0.5]


def pin_walk_rejects_bad_ids(o):
    anchors, ids, vals, G, A, Bc = _random_lattice("bad", 3, 4, 3, 20, 4)
    anchors = anchors.copy()
    anchors[1] = 20
    path, score, _, status = o.selector_walk(anchors, ids, vals, G, A, Bc, 4)
    assert status == 1 and np.all(path[1] == -1) and np.all(np.isnan(score[1]))
    assert np.all(path[0] >= 0) and np.all(path[2] >= 0)
    pred = np.zeros(12, np.int32)
    pred[5] = -1
    s, st = o.pair_scores(pred, ids, vals, G, A, Bc)
    assert st == 1 and np.all(np.isnan(s[5])) and not np.any(np.isnan(np.delete(s, 5, axis=0)))


# --------------------------------------------------------- lattice (next 1-2) --

def pin_lattice_golden(o):
    """Hand-worked table for the walk_r1_k2 inputs (tests/golden/lattice_r1_k2.json)."""
    want = _golden("lattice_r1_k2.json")
    g = _golden(want["inputs"])
    ids = np.asarray(g["ids"], np.int32)
    lat, status = o.lattice(np.asarray([g["anchor"]], np.int32), ids, np.asarray(g["vals"], np.float32),
                            np.asarray(g["G"], np.float32), bf(g["A"]), bf(g["Bc"]), g["block"])
    assert status == 0
    exp = np.asarray([[[np.nan if v is None else v for v in row] for row in slot] for slot in want["lattice"]],
                     np.float64)
    assert np.array_equal(np.isnan(lat[0]), np.isnan(exp))
    assert np.array_equal(np.nan_to_num(lat[0]), np.nan_to_num(exp))
    path, score, _, _ = o.lattice_walk(lat, ids, g["block"], g["V"])
    assert path[0].tolist() == want["greedy_path"] and score[0].tolist() == want["greedy_score"]


def pin_lattice_tie_lower_id(o):
    """The hand-worked tie case (walk_tie.json) walked over its table: equal scores go
    to the lower token id and report a zero margin."""
    g = _golden("walk_tie.json")
    ids = np.asarray(g["ids"], np.int32)
    lat, _ = o.lattice(np.asarray([g["anchor"]], np.int32), ids, np.asarray(g["vals"], np.float32),
                       np.asarray(g["G"], np.float32), bf(g["A"]), bf(g["Bc"]), g["block"])
    path, score, margin, _ = o.lattice_walk(lat, ids, g["block"], g["V"])
    assert path[0].tolist() == g["path"] and score[0].tolist() == g["path_score"]
    assert margin[0].tolist() == g["margin"]


def pin_lattice_greedy_is_the_walk(o):
    """'Greedy follows the best successor' over the precomputed table: the greedy
    lattice walk gives the sequential walk's path, scores and margins exactly."""
    R, B, K, V, r = 5, 7, 6, 90, 10
    anchors, ids, vals, G, A, Bc = _random_lattice("lat_greedy", R, B, K, V, r)
    vals[4, 1] = vals[4, 0]  # exact unary tie somewhere
    lat, st = o.lattice(anchors, ids, vals, G, A, Bc, B)
    p1, s1, m1, _ = o.selector_walk(anchors, ids, vals, G, A, Bc, B)
    p2, s2, m2, st2 = o.lattice_walk(lat, ids, B, V)
    assert st == 0 and st2 == 0
    assert np.array_equal(p1, p2) and np.array_equal(s1, s2) and np.array_equal(m1, m2)


def pin_lattice_rows_are_teacher_forced(o):
    """Row i of slot t-1 scores position t's candidates after predecessor
    ids[t-1, i]: the teacher-forced scorer with that predecessor gives the same row."""
    R, B, K, V, r = 3, 5, 4, 50, 8
    anchors, ids, vals, G, A, Bc = _random_lattice("lat_rows", R, B, K, V, r)
    lat, _ = o.lattice(anchors, ids, vals, G, A, Bc, B)
    for i in range(K):
        pred = np.empty(R * B, np.int32)
        for q in range(R):
            pred[q * B] = anchors[q]
            pred[q * B + 1] = anchors[q]
            for t in range(2, B):
                pred[q * B + t] = ids[q * B + t - 1, i]
        sc, _ = o.pair_scores(pred, ids, vals, G, A, Bc)
        sc = sc.reshape(R, B, K)
        for q in range(R):
            if i == 0:
                assert np.array_equal(lat[q, 0, 0], sc[q, 1])
            else:
                assert np.all(np.isnan(lat[q, 0, i]))
            for t in range(2, B):
                assert np.array_equal(lat[q, t - 1, i], sc[q, t])


def pin_lattice_unit_codebooks_closed_form(o):
    """A = B = 1 makes every row of slot t-1 equal U_t(b) + sum_i G_t[i] (exact with
    small integers), whatever the predecessor."""
    rng = _rng("lat_ones")
    R, B, K, V, r = 2, 4, 3, 25, 5
    anchors, ids, _, _, _, _ = _random_lattice("lat_ones", R, B, K, V, r)
    vals = rng.integers(-6, 7, size=(R * B, K)).astype(np.float32)
    G = rng.integers(-3, 4, size=(R * B, r)).astype(np.float32)
    one = bf(np.ones((V, r)))
    lat, _ = o.lattice(anchors, ids, vals, G, one, one, B)
    want = (vals + G.sum(axis=1, keepdims=True)).reshape(R, B, K)
    for q in range(R):
        assert np.array_equal(lat[q, 0, 0], want[q, 1])
        for t in range(2, B):
            for i in range(K):
                assert np.array_equal(lat[q, t - 1, i], want[q, t])
    # small integers tie often: the greedy table walk breaks them like the walk
    p1, s1, _, _ = o.selector_walk(anchors, ids, vals, G, one, one, B)
    p2, s2, _, _ = o.lattice_walk(lat, ids, B, V)
    assert np.array_equal(p1, p2) and np.array_equal(s1, s2)


def pin_lattice_rejects_bad_ids(o):
    anchors, ids, vals, G, A, Bc = _random_lattice("lat_bad", 3, 4, 3, 20, 4)
    ids = ids.copy()
    ids[2 * 4 + 3, 1] = 20  # request 2, last row
    lat, st = o.lattice(anchors, ids, vals, G, A, Bc, 4)
    assert st == 1 and np.all(np.isnan(lat[2])) and not np.any(np.isnan(lat[:2, 1:]))
    path, score, _, st2 = o.lattice_walk(lat, ids, 4, 20)
    assert st2 == 1 and np.all(path[2] == -1) and np.all(np.isnan(score[2])) and np.all(path[:2] >= 0)


def _sampling_fixture():
    g = _golden("lattice_sampling.json")
    lat = np.asarray(g["lattice"], np.float32)[None]
    ids = np.asarray(g["ids"], np.int32)
    return g, lat, ids


def pin_sampling_golden(o):
    """Hand-worked draws (tests/golden/lattice_sampling.json), including one where
    the sampled column, not the greedy one, selects the next row."""
    g, lat, ids = _sampling_fixture()
    for case in g["cases"]:
        u = np.asarray([case["u"]], np.float32)
        path, score, _, st = o.lattice_walk(lat, ids, g["block"], g["V"], uniforms=u,
                                            temperature=1.0 / math.log(2.0))
        assert st == 0
        assert path[0].tolist() == case["path"], case["work"]
        assert score[0].tolist() == case["score"]


def pin_sampling_two_candidates_closed_form(o):
    """K = 2: column 0 is drawn exactly when u < sigmoid((S_0 - S_1) / temperature),
    and the margin is the distance of u to that boundary."""
    rng = _rng("samp2")
    R, B, K = 400, 2, 2
    lat = np.full((R, 1, K, K), np.nan, np.float32)
    lat[:, 0, 0, :] = rng.standard_normal((R, K)).astype(np.float32) * 2
    ids = np.tile(np.asarray([[0, 0], [3, 5]], np.int32), (R, 1))
    u = rng.random((R, 1)).astype(np.float32)
    tau = 0.7
    path, score, margin, _ = o.lattice_walk(lat, ids, B, 8, uniforms=u, temperature=tau)
    for q in range(R):
        s0, s1 = float(lat[q, 0, 0, 0]), float(lat[q, 0, 0, 1])
        p0 = 1.0 / (1.0 + math.exp(-(s0 - s1) / tau))
        uq = float(u[q, 0])
        if abs(uq - p0) < 1e-12:
            continue
        assert path[q, 0] == (3 if uq < p0 else 5)
        assert abs(margin[q, 0] - abs(uq - p0)) < 1e-12


def pin_sampling_frequencies(o):
    """Draws with independent uniforms follow softmax(S / temperature): the count of
    every column stays within 5 binomial standard deviations of n * p_j."""
    rng = _rng("sampfreq")
    n, K = 20000, 5
    row = np.asarray([1.0, -0.5, 2.0, 0.25, 1.5], np.float32)
    tau = 1.3
    lat = np.broadcast_to(row, (n, 1, K, K)).astype(np.float32).copy()
    ids = np.tile(np.asarray([[0] * K, [10, 11, 12, 13, 14]], np.int32), (n, 1))
    u = rng.random((n, 1)).astype(np.float32)
    path, _, _, _ = o.lattice_walk(lat, ids, 2, 20, uniforms=u, temperature=tau)
    w = np.exp((row.astype(np.float64) - row.max()) / tau)
    p = w / w.sum()
    counts = np.bincount(path[:, 0] - 10, minlength=K)
    assert np.all(np.abs(counts - n * p) <= 5 * np.sqrt(n * p * (1 - p))), (counts, n * p)


def pin_sampling_cold_is_greedy(o):
    """As the temperature goes to zero the draw becomes the greedy pick: with every
    score gap >= 0.1 and temperature 1e-3, any u in [0.01, 0.99] gives the greedy path."""
    rng = _rng("cold")
    R, B, K, V, r = 6, 6, 5, 70, 8
    anchors, ids, vals, G, A, Bc = _random_lattice("cold", R, B, K, V, r)
    lat, _ = o.lattice(anchors, ids, vals, G, A, Bc, B)
    for q in range(R):  # keep each used row's order but space its scores 0.1 apart
        for t in range(B - 1):
            for i in range(K):
                row = lat[q, t, i]
                if np.isnan(row[0]):
                    continue
                order = np.argsort(-row, kind="stable")
                row[order] = row[order[0]] - np.float32(0.1) * np.arange(K, dtype=np.float32)
    gp, gs, _, _ = o.lattice_walk(lat, ids, B, V)
    u = rng.uniform(0.01, 0.99, size=(R, B - 1)).astype(np.float32)
    sp, ss, _, _ = o.lattice_walk(lat, ids, B, V, uniforms=u, temperature=1e-3)
    assert np.array_equal(gp, sp) and np.array_equal(gs, ss)


# ---------------------------------------------------------------- conv (o5) --

def pin_conv_golden(o):
    g = _golden("conv_2tap_1group.json")
    x = np.asarray(g["x"], np.float32)
    y, dyn = o.conv_prepare(x, g["block"], g["taps"], g["group"], bf(g["W_proj"]),
                            np.asarray(g["base"], np.float32))
    assert y.tolist() == g["y"] and dyn.tolist() == g["dyn_out"]
    z = np.asarray(g["z"], np.float32)
    yf = o.conv_finish(z, g["block"], g["taps"], g["group"], dyn, np.asarray(g["base"], np.float32))
    assert yf.tolist() == g["y_finish"]
    # the same case through bf16 activations (all values exact in bf16)
    yb, dynb = o.conv_prepare(bf(x), g["block"], g["taps"], g["group"], bf(g["W_proj"]),
                              np.asarray(g["base"], np.float32))
    assert bf16_bits_to_f32(yb).tolist() == g["y"] and dynb.tolist() == g["dyn_out"]


def _identity_base(taps, C):
    base = np.zeros((2, taps, C), np.float32)
    base[:, 0, :] = 1.0
    return base


def pin_conv_identity_at_init(o):
    """Base tap 0 = 1, later taps 0, projection 0: an exact no-op (verl-SpeCo PR #62,
    'Two deltas', item 2; SpecForge DFlash2 concept doc, 'Architecture')."""
    rng = _rng("ident")
    for taps, B in [(2, 8), (4, 4), (1, 3)]:
        P, C, g = 3 * B, 48, 16
        Wp = np.zeros((2 * taps * (C // g), C), np.uint16)
        base = _identity_base(taps, C)
        xf = rng.standard_normal((P, C)).astype(np.float32)
        xb = f32_to_bf16_bits(xf)
        for x in (xf, xb):
            y, dyn = o.conv_prepare(x, B, taps, g, Wp, base)
            assert np.array_equal(y, x) and not np.any(dyn)
            yf = o.conv_finish(x, B, taps, g, dyn, base)
            assert np.array_equal(yf, x)


def pin_conv_block_locality(o):
    """Changing the last row of block n leaves every row of block n+1 bit-identical
    (verl-SpeCo PR #62, 'Two deltas', item 1; vLLM guide, 'Local Convolution')."""
    rng = _rng("local")
    B, taps, C, g, nb = 4, 3, 32, 8, 3
    P = B * nb
    x = f32_to_bf16_bits(rng.standard_normal((P, C)).astype(np.float32))
    Wp = f32_to_bf16_bits((rng.standard_normal((2 * taps * (C // g), C)) * 0.1).astype(np.float32))
    base = rng.standard_normal((2, taps, C)).astype(np.float32)
    y0, d0 = o.conv_prepare(x, B, taps, g, Wp, base)
    f0 = o.conv_finish(x, B, taps, g, d0, base)
    x2 = x.copy()
    x2[B - 1] = f32_to_bf16_bits(rng.standard_normal(C).astype(np.float32) * 50)
    y1, d1 = o.conv_prepare(x2, B, taps, g, Wp, base)
    f1 = o.conv_finish(x2, B, taps, g, d0, base)
    assert np.array_equal(y0[B:], y1[B:]) and np.array_equal(d0[B:], d1[B:])
    assert np.array_equal(f0[B:], f1[B:])
    assert not np.array_equal(y0[B - 1], y1[B - 1])


def pin_conv_static_kernel_closed_form(o):
    """Zero projection: y_t = sum_{j<=t} base[j] * x_{t-j}, exact for small integers;
    taps = block makes the last position read the whole block."""
    rng = _rng("static")
    for taps, B in [(2, 4), (4, 4), (3, 5)]:
        P, C, g = 2 * B, 8, 4
        x = rng.integers(-5, 6, size=(P, C)).astype(np.float32)
        base = rng.integers(-3, 4, size=(2, taps, C)).astype(np.float32)
        Wp = np.zeros((2 * taps * (C // g), C), np.uint16)
        y, _ = o.conv_prepare(x, B, taps, g, Wp, base)
        yf = o.conv_finish(x, B, taps, g, np.zeros((P, taps, C // g), np.float32), base)
        for p in range(P):
            t = p % B
            want = sum(base[0, j] * x[p - j] for j in range(taps) if t - j >= 0)
            wantf = sum(base[1, j] * x[p - j] for j in range(taps) if t - j >= 0)
            assert np.array_equal(y[p], want) and np.array_equal(yf[p], wantf), (taps, B, p)


def pin_conv_group_sharing(o):
    """One non-zero projection row (input side, tap j, group gi) changes only the g
    channels of group gi, only through tap j, and leaves dyn_out at zero; a row on
    the output side changes only dyn_out[., j, gi] = W_proj row . x_p."""
    rng = _rng("group")
    B, taps, C, g = 4, 2, 24, 8
    G = C // g
    P = 2 * B
    x = rng.integers(-4, 5, size=(P, C)).astype(np.float32)
    base = rng.integers(-2, 3, size=(2, taps, C)).astype(np.float32)
    zero = np.zeros((2 * taps * G, C), np.float32)
    y0, _ = o.conv_prepare(x, B, taps, g, bf(zero), base)
    for j in range(taps):
        for gi in range(G):
            Wp = zero.copy()
            Wp[(0 * taps + j) * G + gi] = rng.integers(-2, 3, size=C)
            y, dyn = o.conv_prepare(x, B, taps, g, bf(Wp), base)
            assert not np.any(dyn)
            d = x @ Wp[(0 * taps + j) * G + gi]
            for p in range(P):
                t = p % B
                delta = np.zeros(C, np.float32)
                if t - j >= 0:
                    delta[gi * g:(gi + 1) * g] = d[p] * x[p - j, gi * g:(gi + 1) * g]
                assert np.array_equal(y[p], y0[p] + delta), (j, gi, p)
            Wo = zero.copy()
            Wo[(1 * taps + j) * G + gi] = rng.integers(-2, 3, size=C)
            y2, dyn2 = o.conv_prepare(x, B, taps, g, bf(Wo), base)
            assert np.array_equal(y2, y0)
            want = np.zeros((P, taps, G), np.float32)
            want[:, j, gi] = x @ Wo[(1 * taps + j) * G + gi]
            assert np.array_equal(dyn2, want)


def pin_conv_bf16_rounding(o):
    """bf16 output is the exact result rounded once to nearest-even: a value just
    above a bf16 midpoint by less than an fp32 ulp must round up (rounding through
    fp32 first would land on the midpoint and round to even, i.e. down)."""
    C, g, B, taps = 2, 2, 1, 1
    x = bf(np.ones((1, C)))
    base = np.zeros((2, taps, C), np.float32)
    base[0, 0, :] = np.float32(1 + 2.0**-8)
    Wp = np.zeros((2, C), np.float32)
    Wp[0, 0] = 2.0**-40   # d = 2^-40 for the single group
    y, _ = o.conv_prepare(x, B, taps, g, bf(Wp), base)
    assert bf16_bits_to_f32(y).tolist() == [[1 + 2.0**-7, 1 + 2.0**-7]]
    y2, _ = o.conv_prepare(x, B, taps, g, bf(np.zeros((2, C))), base)
    assert bf16_bits_to_f32(y2).tolist() == [[1.0, 1.0]]  # exact midpoint: ties to even
    base[0, 0, :] = np.float32(1 + 2.0**-8 + 2.0**-23)
    y3, _ = o.conv_prepare(x, B, taps, g, bf(np.zeros((2, C))), base)
    assert bf16_bits_to_f32(y3).tolist() == [[1 + 2.0**-7, 1 + 2.0**-7]]


def pin_conv_finish_prepare_identity(o):
    """Identity convs on both sides and zero projections: h = z + residual and
    y_next = h exactly, with dyn_next = 0 (quarter-integer values keep every sum
    exact in bf16).  A nonzero residual separates h from z, so a prepare that read
    z instead of h, or a dropped residual, shows."""
    rng = _rng("fin_prep_id")
    B, taps, C, g, nb = 4, 2, 32, 8, 2
    P, G = B * nb, C // g
    z = rng.integers(-4, 5, size=(P, C)) * 0.25
    r = rng.integers(-4, 5, size=(P, C)) * 0.25
    base = _identity_base(taps, C)
    dyn = np.zeros((P, taps, G), np.float32)
    Wp = np.zeros((2 * taps * G, C), np.uint16)
    h, y, d = o.conv_finish_prepare(bf(z), B, taps, g, dyn, base, Wp, base, residual=bf(r))
    assert np.array_equal(bf16_bits_to_f32(h), (z + r).astype(np.float32))
    assert np.array_equal(y, h) and not np.any(d)
    h0, y0, _ = o.conv_finish_prepare(bf(z), B, taps, g, dyn, base, Wp, base)
    assert np.array_equal(bf16_bits_to_f32(h0), z.astype(np.float32)) and np.array_equal(y0, h0)


def pin_conv_finish_prepare_static_closed_form(o):
    """Static kernels (no projection, no dynamic part) on fp32 small-integer data,
    so every value is exact: h_t = b1_0 z_t + b1_1 z_{t-1} + r_t with the finishing
    conv's output-side base b1, then y_t = c0_0 h_t + c0_1 h_{t-1} with the next
    conv's input-side base c0; no tap crosses a block (t-1 >= 0 inside the block)."""
    rng = _rng("fin_prep_static")
    B, taps, C, g, nb = 4, 2, 16, 4, 2
    P, G = B * nb, C // g
    z = rng.integers(-3, 4, size=(P, C)).astype(np.float32)
    r = rng.integers(-3, 4, size=(P, C)).astype(np.float32)
    base = rng.integers(-2, 3, size=(2, taps, C)).astype(np.float32)
    base_next = rng.integers(-2, 3, size=(2, taps, C)).astype(np.float32)
    dyn = np.zeros((P, taps, G), np.float32)
    Wp = np.zeros((2 * taps * G, C), np.uint16)
    h, y, d = o.conv_finish_prepare(z, B, taps, g, dyn, base, Wp, base_next, residual=r)
    t = np.arange(P) % B
    prev = lambda a: np.where((t >= 1)[:, None], np.roll(a, 1, axis=0), 0.0)
    want_h = base[1, 0] * z + base[1, 1] * prev(z) + r
    want_y = base_next[0, 0] * want_h + base_next[0, 1] * prev(want_h)
    assert np.array_equal(h, want_h.astype(np.float32))
    assert np.array_equal(y, want_y.astype(np.float32)) and not np.any(d)


def pin_conv_finish_prepare_block_locality(o):
    """Changing the last row of block n (z and the residual) leaves every output row
    of block n+1 bit-identical through both convs."""
    rng = _rng("fin_prep_local")
    B, taps, C, g, nb = 4, 3, 32, 8, 3
    P, G = B * nb, C // g
    bfr = lambda shape, s: f32_to_bf16_bits((rng.standard_normal(shape) * s).astype(np.float32))
    z, r = bfr((P, C), 1.0), bfr((P, C), 1.0)
    dyn = (rng.standard_normal((P, taps, G)) * 0.1).astype(np.float32)
    Wp = bfr((2 * taps * G, C), 0.1)
    base = rng.standard_normal((2, taps, C)).astype(np.float32)
    base_next = rng.standard_normal((2, taps, C)).astype(np.float32)
    out0 = o.conv_finish_prepare(z, B, taps, g, dyn, base, Wp, base_next, residual=r)
    z2, r2 = z.copy(), r.copy()
    z2[B - 1] = bfr(C, 50.0)
    r2[B - 1] = bfr(C, 50.0)
    out1 = o.conv_finish_prepare(z2, B, taps, g, dyn, base, Wp, base_next, residual=r2)
    for a, b in zip(out0, out1):
        assert np.array_equal(a[B:], b[B:])
        assert not np.array_equal(a[B - 1], b[B - 1])


def pin_conv_rejects_bad_shapes(o):
    x = np.zeros((6, 8), np.float32)
    base = np.zeros((2, 2, 8), np.float32)
    Wp = np.zeros((2 * 2 * 2, 8), np.uint16)
    for B, taps, g in [(4, 2, 4), (3, 4, 4), (3, 2, 3)]:  # P % B, taps > B, C % g
        try:
            o.conv_prepare(x, B, taps, g, Wp, base)
        except ValueError:
            continue
        raise AssertionError(f"accepted block={B} taps={taps} group={g}")


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_") and callable(v)]
