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
