"""Parity of the lattice schedule (all adjacent pair scores at once, then a greedy
or sampling walk over the table) with the CPU oracle, through the C-ABI."""
import math

import numpy as np
import pytest

import workloads as W
from parity import close, compare_walk

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def df2():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import dflash2_draft_block_gb300 as m
    m.lib()
    return m


def bf_dev(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to("cuda").view(torch.bfloat16)


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to("cuda")


def host(t):
    return t.cpu().numpy()


def candidates(rng, R, B, K, V, r, cb_std=0.3):
    ids = np.stack([rng.choice(V, size=K, replace=False) for _ in range(R * B)]).astype(np.int32)
    vals = -np.sort(-rng.standard_normal((R * B, K)).astype(np.float32), axis=-1)
    G = rng.standard_normal((R * B, r)).astype(np.float32)
    A = W.f32_to_bf16_bits((rng.standard_normal((V, r)) * cb_std).astype(np.float32))
    Bc = W.f32_to_bf16_bits((rng.standard_normal((V, r)) * cb_std).astype(np.float32))
    anchors = rng.integers(0, V, size=R).astype(np.int32)
    return anchors, ids, vals, G, A, Bc


def gpu_lattice(df2, anchors, ids, vals, G, A, Bc, B, dev_status=None):
    lat = df2.selector_lattice(dev(anchors), dev(ids), dev(vals), dev(G), bf_dev(A), bf_dev(Bc), B,
                               dev_status=dev_status)
    torch.cuda.synchronize()
    return host(lat)


def gpu_walk(df2, lat, ids, B, V, uniforms=None, temperature=1.0):
    path, score = df2.lattice_walk(dev(lat), dev(ids), B, V,
                                   uniforms=None if uniforms is None else dev(uniforms),
                                   temperature=temperature)
    torch.cuda.synchronize()
    return host(path), host(score)


def check_table(gpu, ref, what):
    """NaN exactly where the oracle has NaN (slot 0 rows 1..K-1), values within the
    float tolerance of the row scale elsewhere."""
    assert gpu.shape == ref.shape, what
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(gpu), nan), what
    R, T, K, _ = ref.shape
    if R == 0:
        return
    # compare each defined row (slot, predecessor) as a row of K scores
    g = gpu.reshape(-1, K)
    o = ref.reshape(-1, K)
    keep = ~np.isnan(o[:, 0])
    close(g[keep], o[keep], what=what)


def compare_sampled(gpu_path, gpu_score, ref_path, ref_score, ref_margin, what):
    """Sampling draws: like compare_walk, a divergence must sit where u lies within
    MARGIN (probability units) of an end of the oracle's chosen interval."""
    return compare_walk(gpu_path, gpu_score, ref_path, ref_score, ref_margin, what)


@pytest.mark.parametrize("R,B,K,V,r", [
    (2, 8, 4, 4096, 32),
    (3, 2, 1, 500, 8),
    (5, 16, 17, 3000, 264),
    (4, 8, 64, 10000, 512),
    (3, 6, 40, 7000, 200),    # 32 < K < 64 (N = 48), a ragged last rank slice
    (2, 5, 33, 3000, 72),
    (2, 4, 100, 3000, 64),
    (1, 3, 1024, 5000, 16),
    (37, 8, 16, 5000, 256),
])
def test_lattice_shapes(orc, df2, R, B, K, V, r):
    rng = np.random.default_rng(R * 1000 + B * 100 + K + r)
    anchors, ids, vals, G, A, Bc = candidates(rng, R, B, K, V, r)
    gl = gpu_lattice(df2, anchors, ids, vals, G, A, Bc, B)
    ol, st = orc.lattice(anchors, ids, vals, G, A, Bc, B)
    assert st == 0
    check_table(gl, ol, f"lattice {R}x{B} K{K} r{r}")
    # greedy over the GPU table against the oracle's sequential walk
    gp, gs = gpu_walk(df2, gl, ids, B, V)
    op, os_, om, _ = orc.selector_walk(anchors, ids, vals, G, A, Bc, B)
    compare_walk(gp, gs, op, os_, om, "lattice greedy").check("lattice greedy")
    # sampling over the GPU table against the oracle's draw over the oracle's table
    u = rng.random((R, B - 1)).astype(np.float32)
    sp, ss = gpu_walk(df2, gl, ids, B, V, uniforms=u, temperature=0.8)
    op2, os2, om2, _ = orc.lattice_walk(ol, ids, B, V, uniforms=u, temperature=0.8)
    compare_sampled(sp, ss, op2, os2, om2, "lattice sampling").check("lattice sampling")


def test_walk_on_the_oracle_table_is_exact(orc, df2):
    """Fed the oracle's own table, the greedy walk takes exactly the oracle's
    decisions (same fp32 scores, same tie rule); the sampled walk differs only where
    u is within fp32 rounding of an interval end."""
    rng = np.random.default_rng(5)
    R, B, K, V, r = 64, 8, 16, 4000, 64
    anchors, ids, vals, G, A, Bc = candidates(rng, R, B, K, V, r)
    vals[:, 1] = vals[:, 0]  # exact unary ties at the top of every list
    Bc[:] = 0                # ... which stay ties in the table: the id rule decides
    ol, _ = orc.lattice(anchors, ids, vals, G, A, Bc, B)
    gp, gs = gpu_walk(df2, ol, ids, B, V)
    op, os_, _, _ = orc.lattice_walk(ol, ids, B, V)
    assert np.array_equal(gp, op) and np.array_equal(gs, os_)
    anchors, ids, vals, G, A, Bc = candidates(rng, R, B, K, V, r)
    ol, _ = orc.lattice(anchors, ids, vals, G, A, Bc, B)
    u = rng.random((R, B - 1)).astype(np.float32)
    sp, ss = gpu_walk(df2, ol, ids, B, V, uniforms=u, temperature=1.0)
    op, os_, om, _ = orc.lattice_walk(ol, ids, B, V, uniforms=u, temperature=1.0)
    rep = compare_sampled(sp, ss, op, os_, om, "sampling on oracle table")
    rep.check("sampling on oracle table")


def test_greedy_lattice_matches_the_direct_walk_gpu(orc, df2):
    """Both GPU schedules of the greedy walk agree wherever the oracle's decision
    margin is not a near-tie."""
    rng = np.random.default_rng(6)
    R, B, K, V, r = 48, 16, 64, 8000, 512
    anchors, ids, vals, G, A, Bc = candidates(rng, R, B, K, V, r)
    gl = gpu_lattice(df2, anchors, ids, vals, G, A, Bc, B)
    lp, ls = gpu_walk(df2, gl, ids, B, V)
    wp, ws = df2.selector_walk(dev(anchors), dev(ids), dev(vals), dev(G), bf_dev(A), bf_dev(Bc), B)
    wp, ws = host(wp), host(ws)
    op, os_, om, _ = orc.selector_walk(anchors, ids, vals, G, A, Bc, B)
    compare_walk(lp, ls, op, os_, om, "lattice").check("lattice vs oracle")
    compare_walk(wp, ws, op, os_, om, "direct").check("direct vs oracle")
    rep = compare_walk(lp, ls, wp, ws, om, "lattice vs direct")
    rep.check("lattice vs direct")


def test_sampling_golden_gpu(df2):
    """The hand-worked draws of tests/golden/lattice_sampling.json on the GPU."""
    import json
    import os
    g = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "lattice_sampling.json")))
    lat = np.asarray(g["lattice"], np.float32)[None]
    ids = np.asarray(g["ids"], np.int32)
    for case in g["cases"]:
        u = np.asarray([case["u"]], np.float32)
        path, score = gpu_walk(df2, lat, ids, g["block"], g["V"], uniforms=u,
                               temperature=1.0 / math.log(2.0))
        assert path[0].tolist() == case["path"], case["work"]
        assert score[0].tolist() == case["score"]


def test_sampling_frequencies_gpu(df2):
    """20,000 independent draws from one row follow softmax(S / temperature)."""
    rng = np.random.default_rng(7)
    n, K = 20000, 5
    row = np.asarray([1.0, -0.5, 2.0, 0.25, 1.5], np.float32)
    tau = 1.3
    lat = np.broadcast_to(row, (n, 1, K, K)).astype(np.float32).copy()
    ids = np.tile(np.asarray([[0] * K, [10, 11, 12, 13, 14]], np.int32), (n, 1))
    u = rng.random((n, 1)).astype(np.float32)
    path, _ = gpu_walk(df2, lat, ids, 2, 20, uniforms=u, temperature=tau)
    w = np.exp((row.astype(np.float64) - row.max()) / tau)
    p = w / w.sum()
    counts = np.bincount(path[:, 0] - 10, minlength=K)
    assert np.all(np.abs(counts - n * p) <= 5 * np.sqrt(n * p * (1 - p))), (counts, n * p)


def test_cold_sampling_is_greedy_gpu(df2):
    """Temperature 1e-3 over rows whose scores are 0.1 apart gives the greedy path."""
    rng = np.random.default_rng(8)
    R, B, K, V = 32, 8, 16, 3000
    ids = np.stack([rng.choice(V, size=K, replace=False) for _ in range(R * B)]).astype(np.int32)
    lat = np.empty((R, B - 1, K, K), np.float32)
    for q in range(R):
        for s in range(B - 1):
            for i in range(K):
                lat[q, s, i] = rng.permutation(K).astype(np.float32) * np.float32(0.1) + np.float32(3.0)
    gp, gs = gpu_walk(df2, lat, ids, B, V)
    u = rng.uniform(0.01, 0.99, size=(R, B - 1)).astype(np.float32)
    sp, ss = gpu_walk(df2, lat, ids, B, V, uniforms=u, temperature=1e-3)
    assert np.array_equal(gp, sp) and np.array_equal(gs, ss)


def test_lattice_bad_ids_gpu(df2):
    rng = np.random.default_rng(9)
    R, B, K, V, r = 3, 4, 8, 100, 32
    anchors, ids, vals, G, A, Bc = candidates(rng, R, B, K, V, r)
    ids[2 * B + 3, 1] = V  # request 2, last row
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    gl = gpu_lattice(df2, anchors, ids, vals, G, A, Bc, B, dev_status=status)
    assert int(status.item()) & df2.DF2_STATUS_ID_OUT_OF_RANGE
    assert np.all(np.isnan(gl[2])) and not np.isnan(gl[:2, 1:]).any()
    status.zero_()
    path, score = df2.lattice_walk(dev(gl), dev(ids), B, V, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & df2.DF2_STATUS_ID_OUT_OF_RANGE
    path, score = host(path), host(score)
    assert np.all(path[2] == -1) and np.all(np.isnan(score[2])) and np.all(path[:2] >= 0)


def test_lattice_empty(df2):
    z = torch.zeros(0, dtype=torch.int32, device="cuda")
    ids = torch.zeros((0, 4), dtype=torch.int32, device="cuda")
    vals = torch.zeros((0, 4), dtype=torch.float32, device="cuda")
    G = torch.zeros((0, 8), dtype=torch.float32, device="cuda")
    A = torch.zeros((16, 8), dtype=torch.bfloat16, device="cuda")
    lat = df2.selector_lattice(z, ids, vals, G, A, A, 4)
    assert tuple(lat.shape) == (0, 3, 4, 4)
    path, score = df2.lattice_walk(lat, ids, 4, 16)
    assert tuple(path.shape) == (0, 3)


@pytest.mark.parametrize("name", ["batch1", "batched", "stress"])
def test_full_size_lattice(orc, df2, name):
    """The workload's shapes in the launch configuration the benchmark uses, every
    request compared: the GPU table against the oracle's; the GPU walks over the
    oracle's table against the oracle's walks over it (greedy exactly, sampled under
    the probability margin); and the GPU walks over the GPU table against the
    oracle's walks over its own table (the flagged-margin rule).  The oracle only
    ever reads its own table."""
    w = W.BY_NAME[name]
    rng = np.random.default_rng(w.seed + 200)
    anchors, ids, vals, G, A, Bc = candidates(rng, w.R, w.B, w.K, w.V, w.r)
    gl = gpu_lattice(df2, anchors, ids, vals, G, A, Bc, w.B)
    ol, st = orc.lattice(anchors, ids, vals, G, A, Bc, w.B)
    assert st == 0
    check_table(gl, ol, name + " lattice")
    op, os_, om, _ = orc.lattice_walk(ol, ids, w.B, w.V)
    gp, gs = gpu_walk(df2, ol, ids, w.B, w.V)
    assert np.array_equal(gp, op) and np.array_equal(gs, os_), name + " greedy walk over the oracle table"
    gp, gs = gpu_walk(df2, gl, ids, w.B, w.V)
    compare_walk(gp, gs, op, os_, om, name + " greedy").check(name + " greedy")
    u = rng.random((w.R, w.B - 1)).astype(np.float32)
    op2, os2, om2, _ = orc.lattice_walk(ol, ids, w.B, w.V, uniforms=u, temperature=1.0)
    for table, what in ((ol, " sampling over the oracle table"), (gl, " sampling")):
        sp, ss = gpu_walk(df2, table, ids, w.B, w.V, uniforms=u, temperature=1.0)
        compare_sampled(sp, ss, op2, os2, om2, name + what).check(name + what)
