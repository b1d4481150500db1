"""The whole-batch comparator (parity.compare_chain) on the CPU: the oracle's own
outputs pass it, and each planted mistake in a copy of them is reported.

The comparator is what the at-scale GPU tests and the benchmark's parity block
rely on, so it must catch a wrong id at an unflagged position, a wrong path step,
a float outside tolerance and a conv output more than one bf16 step off, while
letting through a swap at a flagged near-tie."""
import numpy as np
import pytest

import workloads as W
from parity import MARGIN, compare_chain


@pytest.fixture(scope="module")
def case(orc):
    import bench
    w = W.TINY.scaled(R=4)
    inp = W.head_inputs(w, selector_std=0.3)
    conv = W.conv_inputs(w)
    out = bench.oracle_step(orc, w, inp, conv)
    return w, inp, conv, out


def _run(orc, case, mutate=None):
    w, inp, conv, out = case
    g = {k: np.array(v, copy=True) for k, v in out.items()}
    if mutate is not None:
        mutate(g, inp)
    return compare_chain(orc, w, inp, g, range(w.R), conv=conv, check=False)


def test_oracle_against_itself_passes(orc, case):
    s = _run(orc, case)
    assert s["ok"], s["failures"]
    assert s["topk"]["mismatched"] == 0 and s["walk"]["mismatched"] == 0
    assert s["topk"]["compared"] == case[0].P and s["conv_rows"] == case[0].P


def _unflagged_row(orc, case):
    w, inp, _, out = case
    _, _, margin, _ = orc.unary_topk(inp["h"], inp["W_lm"], w.K, W_H=inp["W_H"])
    for p in range(w.P):
        if margin[p] >= MARGIN and np.all(np.abs(np.diff(out["vals"][p])) >= MARGIN):
            return p
    pytest.skip("no unflagged row")


def test_swapped_ids_at_an_unflagged_row_fail(orc, case):
    p = _unflagged_row(orc, case)

    def m(g, inp):
        g["ids"][p, [0, 1]] = g["ids"][p, [1, 0]]
    s = _run(orc, case, m)
    assert not s["ok"] and s["topk"]["unexplained"] == 1


def test_foreign_id_at_an_unflagged_row_fails(orc, case):
    p = _unflagged_row(orc, case)

    def m(g, inp):
        g["ids"][p, -1] = (int(g["ids"][p].max()) + 1) % case[0].V
    assert not _run(orc, case, m)["ok"]


def test_wrong_G_fails(orc, case):
    def m(g, inp):
        g["G"][3, 5] *= 1.01
    s = _run(orc, case, m)
    assert not s["ok"] and any(" G" in f for f in s["failures"])


def test_wrong_path_step_fails(orc, case):
    w, inp, _, out = case
    _, _, wmargin, _ = orc.selector_walk(inp["anchors"], out["ids"], out["vals"], out["G"], inp["A"], inp["Bc"],
                                         w.B)
    q, t = map(int, np.argwhere(wmargin >= MARGIN)[0])
    ids = out["ids"].reshape(w.R, w.B, w.K)

    def m(g, inp):
        other = [i for i in ids[q, t + 1] if i != g["path"][q, t]]
        g["path"][q, t] = other[0]
    s = _run(orc, case, m)
    assert not s["ok"] and s["walk"]["mismatched"] == 1


def test_path_score_outside_tolerance_fails(orc, case):
    def m(g, inp):
        g["pscore"][1, 2] += 0.05 * max(1.0, abs(float(g["pscore"][1, 2])))
    assert not _run(orc, case, m)["ok"]


def test_teacher_forced_score_outside_tolerance_fails(orc, case):
    def m(g, inp):
        g["scores"][9, 1] += 0.1
    s = _run(orc, case, m)
    assert not s["ok"] and any("teacher-forced" in f for f in s["failures"])


def test_conv_two_steps_off_fails_one_step_passes(orc, case):
    w = case[0]
    is_bf16 = case[3]["y"].dtype == np.uint16

    def one(g, inp):
        if is_bf16:
            g["y"][2, 7] += 1
        else:
            g["y"][2, 7] *= 1 + 1e-4

    def far(g, inp):
        if is_bf16:
            g["y2"][2, 7] += 3
        else:
            g["y2"][2, 7] += 1.0
    assert _run(orc, case, one)["ok"]
    s = _run(orc, case, far)
    assert not s["ok"] and any("finish" in f for f in s["failures"])


# ------------------------------------------------ ids at a flagged K/K+1 boundary --

def _lists():
    """A row whose oracle K-th and (K+1)-th logits are 4e-4 apart (flagged)."""
    ref_ids = np.array([[10, 11, 12, 13]], np.int32)
    ref_vals = np.array([[4.0, 3.0, 2.0, 1.0]], np.float32)
    return ref_ids, ref_vals, np.array([4e-4])


def test_foreign_id_checked_against_the_oracle_logit():
    """At a flagged boundary the GPU may keep the oracle's (K+1)-th token instead of
    its K-th, but only if the oracle's own logit of that token is within MARGIN of the
    K-th value and the GPU's value for it is right: a value the GPU reports is not
    evidence."""
    from parity import compare_topk
    ref_ids, ref_vals, margin = _lists()
    gpu_ids = np.array([[10, 11, 12, 99]], np.int32)
    gpu_vals = np.array([[4.0, 3.0, 2.0, 0.9996]], np.float32)
    near = {99: 0.9996}
    far = {99: 0.5}
    ok = compare_topk(gpu_ids, gpu_vals, ref_ids, ref_vals, margin, logit_of=lambda p, ids: [near[i] for i in ids])
    assert ok.mismatched == 1 and not ok.unexplained
    bad = compare_topk(gpu_ids, gpu_vals, ref_ids, ref_vals, margin, logit_of=lambda p, ids: [far[i] for i in ids])
    assert len(bad.unexplained) == 1
    # the right token with a wrong value
    off = gpu_vals.copy()
    off[0, 3] = 0.95
    wrong = compare_topk(gpu_ids, off, ref_ids, ref_vals, margin, logit_of=lambda p, ids: [near[i] for i in ids])
    assert len(wrong.unexplained) == 1


def test_planted_tie_swap_passes_and_a_false_claim_fails(orc):
    """The whole-batch comparator on a planted exact tie: token X gets the W_lm row
    of row p's K-th token, so the two tie at rank K / K+1 and the oracle keeps the
    lower id.  A GPU list holding X instead passes (a flagged near-tie); one holding
    an unrelated token with the K-th value written beside it fails, because the
    comparator asks the oracle for that token's logit."""
    import bench
    w = W.TINY.scaled(R=2)
    inp = W.head_inputs(w, selector_std=0.3)
    oi, _, _, _ = orc.unary_topk(inp["h"], inp["W_lm"], w.K + 1)
    p = w.B + 1
    a = int(oi[p, w.K - 1])
    taken = set(int(i) for i in oi[p])
    X = next(v for v in range(a + 1, w.V) if v not in taken)
    Wl = inp["W_lm"].copy()
    Wl[X] = Wl[a]
    inp = dict(inp, W_lm=Wl)
    conv = W.conv_inputs(w)
    out = bench.oracle_step(orc, w, inp, conv)
    assert int(out["ids"][p, w.K - 1]) == a
    _, _, margin, _ = orc.unary_topk(inp["h"][p:p + 1], Wl, w.K)
    assert margin[0] == 0.0

    def run(mutate):
        g = {k: np.array(v, copy=True) for k, v in out.items()}
        mutate(g)
        return compare_chain(orc, w, inp, g, range(w.R), conv=conv, check=False)

    def swap(g):
        # a GPU that kept X: the same logit, and its walk and teacher-forced scores
        # computed on the list it kept
        g["ids"][p, w.K - 1] = X
        g["path"], g["pscore"], _, _ = orc.selector_walk(inp["anchors"], g["ids"], g["vals"], g["G"], inp["A"],
                                                         inp["Bc"], w.B)
        g["scores"], _ = orc.pair_scores(inp["pred"], g["ids"], g["vals"], g["G"], inp["A"], inp["Bc"])
    s = run(swap)
    assert s["topk"]["mismatched"] == 1 and s["topk"]["unexplained"] == 0, s["failures"]
    assert s["walk"]["requests_on_gpu_lists"] == 1 and s["walk"]["unexplained"] == 0
    # the walk and scores over the GPU's list agree; what fails is only the fraction
    # rule (one mismatch in 16 compared rows is above 0.1%)
    assert len(s["failures"]) == 1 and "mismatched positions" in s["failures"][0], s["failures"]

    U = orc.logits(inp["h"][p:p + 1], Wl)[0]
    far = int(np.argmin(U))   # the token with the lowest logit of the row

    def claim(g):
        g["ids"][p, w.K - 1] = far
    assert U[a] - U[far] >= MARGIN
    s = run(claim)
    assert s["topk"]["unexplained"] == 1 and not s["ok"]
