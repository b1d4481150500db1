"""Parity of the selector's K-way cross-entropy (verl-SpeCo PR #62, "Selector training
objective") with the CPU oracle, through the C-ABI: the label column exactly, the
loss within 2e-3 of max(|oracle|, 1) (fp32 log-sum-exp against fp64), NaN on the
same rows."""
import numpy as np
import pytest

import workloads as W

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

TOL = 2e-3


@pytest.fixture(scope="module")
def df2():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import dflash2_draft_block_gb300 as m
    m.lib()
    return m


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to("cuda")


def case(rng, P, K, V, scale=3.0, covered=0.7, none=0.1):
    """Candidate rows of distinct ids, scores ~ N(0, scale) (the teacher-forced scores'
    spread at the workloads' unary scale), and targets: a candidate of the row with
    probability `covered`, -1 with probability `none`, otherwise a random token."""
    ids = np.stack([rng.choice(V, size=K, replace=False) for _ in range(P)]).astype(np.int32)
    scores = (rng.standard_normal((P, K)) * scale).astype(np.float32)
    u = rng.random(P)
    targets = rng.integers(0, V, size=P).astype(np.int32)
    pick = ids[np.arange(P), rng.integers(0, K, size=P)]
    targets = np.where(u < covered, pick, targets).astype(np.int32)
    targets = np.where(u > 1.0 - none, -1, targets).astype(np.int32)
    return scores, ids, targets


def check(df2, orc, scores, ids, targets, V, what):
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    loss, label = df2.selector_ce(dev(scores), dev(ids), dev(targets), V, dev_status=status)
    torch.cuda.synchronize()
    loss, label = loss.cpu().numpy(), label.cpu().numpy()
    ol, olab, ost = orc.selector_ce(scores, ids, targets, V)
    assert np.array_equal(label, olab), what + ": label columns"
    assert np.array_equal(np.isnan(loss), np.isnan(ol)), what + ": excluded rows"
    ok = ~np.isnan(ol)
    err = np.abs(loss[ok] - ol[ok]) / np.maximum(np.abs(ol[ok]), 1.0)
    assert err.size == 0 or err.max() <= TOL, f"{what}: loss error {err.max():.3g}"
    assert (int(status.item()) != 0) == (ost != 0), what + ": status"
    return int(ok.sum())


@pytest.mark.parametrize("P,K,V", [
    (1, 1, 10),          # one candidate: loss 0 where covered
    (37, 16, 5000),      # batch shapes, a ragged last CTA of warps
    (64, 64, 20000),     # K = 64
    (5, 1000, 3000),     # K near the maximum: many strides per lane
    (300, 33, 4096),     # K just past one warp's width
])
def test_selector_ce_shapes(orc, df2, P, K, V):
    rng = np.random.default_rng(P * 7 + K)
    scores, ids, targets = case(rng, P, K, V)
    n = check(df2, orc, scores, ids, targets, V, f"P{P} K{K}")
    assert n > 0 or P == 1


def test_selector_ce_edge_rows(orc, df2):
    """Equal scores (ln K), a dominant label (loss ~ 0), -inf scores beside the
    label, NaN scores (NaN loss), targets < 0, absent and >= V."""
    K, V = 8, 100
    ids = np.tile(np.arange(K, dtype=np.int32) * 3, (7, 1))
    scores = np.zeros((7, K), np.float32)
    scores[1, 2] = 40.0
    scores[2, :] = -np.inf
    scores[2, 5] = 1.0
    scores[3, 4] = np.nan
    targets = np.array([9, 6, 15, 0, -1, 1, 100], np.int32)  # 1 is not a candidate; 100 >= V
    check(df2, orc, scores, ids, targets, V, "edge rows")
    loss, label = df2.selector_ce(dev(scores), dev(ids), dev(targets), V)
    loss = loss.cpu().numpy()
    assert abs(loss[0] - np.log(K)) <= 1e-6 * np.log(K)
    assert 0.0 <= loss[1] <= 1e-12 and loss[2] == 0.0
    assert np.isnan(loss[3]) and np.isnan(loss[4]) and np.isnan(loss[5]) and np.isnan(loss[6])


def test_selector_ce_empty(df2):
    z = torch.zeros((0, 4), dtype=torch.float32, device="cuda")
    loss, label = df2.selector_ce(z, z.to(torch.int32), torch.zeros(0, dtype=torch.int32, device="cuda"), 10)
    assert loss.numel() == 0 and label.numel() == 0


@pytest.mark.parametrize("name", ["batch1", "batched", "stress"])
def test_full_size_selector_ce(orc, df2, name):
    """The workloads' row counts and K: every row compared."""
    w = W.BY_NAME[name]
    rng = np.random.default_rng(w.seed + 300)
    scores, ids, targets = case(rng, w.P, w.K, w.V)
    n = check(df2, orc, scores, ids, targets, w.V, name)
    assert n >= (w.P // 2 if w.P >= 64 else 1)  # rows with a covered target were compared
