"""Parity of the CUDA path (through the C-ABI) with the CPU oracle, on the GPU.

Small cases compare every output; the full-size workloads compare sampled rows
(the head) or whole anchor blocks (the conv) that the oracle computes one by one,
in the same launch configuration the benchmark uses.  Token ids must match
exactly outside flagged near-ties; floats within 2e-3 of the row scale."""
import numpy as np
import pytest

import workloads as W
from parity import (check_path_valid, close, close_bf16, compare_topk, compare_topk_values,
                    compare_walk)

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


def host_bf(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def host(t):
    return t.cpu().numpy()


def _rng(seed):
    return np.random.default_rng(seed)


def rand_bf16(rng, shape, std=1.0):
    return W.f32_to_bf16_bits((rng.standard_normal(shape) * std).astype(np.float32))


# ------------------------------------------------------------------ head ----

def run_head(df2, h, Wlm, K, WH=None):
    ids, vals, G = df2.unary_topk(bf_dev(h), bf_dev(Wlm), K, None if WH is None else bf_dev(WH))
    torch.cuda.synchronize()
    return host(ids), host(vals), (None if G is None else host(G))


def check_head(orc, df2, h, Wlm, K, WH=None, what="head"):
    gi, gv, gG = run_head(df2, h, Wlm, K, WH)
    oi, ov, om, oG = orc.unary_topk(h, Wlm, K, W_H=WH)
    rep = compare_topk(gi, gv, oi, ov, om, what,
                       logit_of=lambda p, ids: orc.logits(h[p:p + 1], Wlm[np.asarray(ids, np.int64)])[0])
    rep.check(what)
    compare_topk_values(gi, gv, oi, ov, what + " vals")
    if WH is not None:
        close(gG, oG, what=what + " G")
    return rep


def test_tiny_head(orc, df2):
    w = W.TINY
    inp = W.head_inputs(w)
    check_head(orc, df2, inp["h"], inp["W_lm"], w.K, inp["W_H"], "tiny")


@pytest.mark.parametrize("P,D,V,K", [
    (1, 64, 100, 1),          # single row, K = 1
    (5, 264, 1000, 37),       # ragged everything, D not a multiple of 64
    (13, 128, 64, 64),        # K = V
    (16, 256, 4096, 16),      # several tiles
    (2, 64, 1024, 1024),      # K = V = the build's K limit
    (9, 512, 20011, 64),      # prime V, K = 64
    (33, 1024, 3000, 16),     # more rows than one position group
])
def test_head_shapes(orc, df2, P, D, V, K):
    rng = _rng(P * 7919 + D * 31 + V + K)
    h = rand_bf16(rng, (P, D))
    Wlm = rand_bf16(rng, (V, D), 0.02)
    WH = rand_bf16(rng, (8 * (1 + P % 3), D), 0.02)
    check_head(orc, df2, h, Wlm, K, WH, f"head{P}x{D}x{V}k{K}")


@pytest.mark.parametrize("P,D,V,K", [
    (129, 256, 1000, 16),     # many-position tensor-core path: ragged M tile, V % 256 != 0
    (200, 320, 777, 64),      # D not a multiple of 64, K = 64
    (130, 128, 513, 1),       # K = 1
    (257, 64, 300, 33),       # three M tiles, K just above one register row
    (48, 512, 5000, 16),      # just above the few-position path
    # an even number of 256-position pairs: clusters of two pairs share the W_lm tiles
    (512, 256, 7001, 16),     # two pairs, ragged V
    (1000, 128, 4000, 64),    # four pairs, the last one ragged, K = 64
])
def test_head_many_positions(orc, df2, P, D, V, K):
    rng = _rng(P * 131 + D + V * 7 + K)
    h = rand_bf16(rng, (P, D))
    Wlm = rand_bf16(rng, (V, D), 0.02)
    WH = rand_bf16(rng, (16 * (1 + P % 3), D), 0.02)
    check_head(orc, df2, h, Wlm, K, WH, f"wide{P}x{D}x{V}k{K}")


@pytest.mark.parametrize("P,D,V,K,r", [
    # on a 152-SM part the last vocabulary range holds one tile where the others
    # hold two, so G = H(h) is computed there, inside the top-K launch
    (200, 256, 19600, 16, 40),    # CTA pairs, ragged M tile, r not a multiple of 16
    (256, 192, 19600, 8, 256),    # CTA pairs, G exactly one tile wide
    (48, 128, 39000, 16, 24),     # one CTA per M tile
    (200, 256, 19600, 16, 264),   # G wider than one tile: a store launch of its own
    (512, 256, 19600, 16, 40),    # two pairs sharing W_lm tiles, G in the top-K launch
])
def test_head_many_positions_with_H(orc, df2, P, D, V, K, r):
    rng = _rng(P * 17 + V + r)
    h = rand_bf16(rng, (P, D))
    Wlm = rand_bf16(rng, (V, D), 0.02)
    WH = rand_bf16(rng, (r, D), 0.02)
    check_head(orc, df2, h, Wlm, K, WH, f"wideH{P}x{D}x{V}k{K}r{r}")


def test_head_many_positions_exact_ties(orc, df2):
    rng = _rng(77)
    P, D, V, K = 140, 128, 3000, 16
    Wlm = rand_bf16(rng, (V, D), 0.02)
    Wlm[1500:2400] = Wlm[0:900]          # duplicates in other CTA ranges and tiles
    Wlm[2999] = Wlm[5]
    h = rand_bf16(rng, (P, D))
    gi, gv, _ = run_head(df2, h, Wlm, K)
    oi, ov, om, _ = orc.unary_topk(h, Wlm, K)
    assert np.array_equal(gi, oi)


def test_head_exact_ties_break_to_lower_id(orc, df2):
    rng = _rng(5)
    P, D, V, K = 6, 128, 2000, 16
    Wlm = rand_bf16(rng, (V, D), 0.02)
    h = rand_bf16(rng, (P, D))
    # duplicate rows everywhere: equal logits must rank the lower id first
    Wlm[1000:1600] = Wlm[0:600]
    Wlm[1999] = Wlm[3]
    gi, gv, _ = run_head(df2, h, Wlm, K)
    oi, ov, om, _ = orc.unary_topk(h, Wlm, K)
    assert np.array_equal(gi, oi)
    assert np.array_equal(gv, ov) or np.allclose(gv, ov, rtol=2e-3, atol=2e-3)


# ------------------------------------------- logit multiplier / softcap ----

@pytest.mark.parametrize("P,D,V,K,m,c", [
    (8, 1024, 20011, 16, 1.0, 30.0),     # few positions (the streaming head), a cap only
    (3, 264, 3000, 37, 0.5, 0.0),        # ragged shapes, a multiplier only
    (140, 256, 5000, 16, 2.0, 0.75),     # many positions (the tensor-core GEMM), a tight cap
    (20, 256, 3000, 100, 1.5, 4.0),      # K > 64: the CUDA-core path
])
def test_head_logit_map(orc, df2, P, D, V, K, m, c):
    """Top-K of c*tanh(m*U/c) against the oracle, which maps all V logits before
    selecting; the kernels select on U and map the K kept values, so their ids
    equal the unmapped call's and their values are the map of its values."""
    rng = _rng(P * 17 + D + V * 3 + K)
    h = rand_bf16(rng, (P, D))
    Wlm = rand_bf16(rng, (V, D), 0.02)
    ids, vals, _ = df2.unary_topk(bf_dev(h), bf_dev(Wlm), K, output_multiplier=m, final_logit_softcapping=c)
    ids0, vals0, _ = df2.unary_topk(bf_dev(h), bf_dev(Wlm), K)
    torch.cuda.synchronize()
    gi, gv, gi0, gv0 = host(ids), host(vals), host(ids0), host(vals0)
    oi, ov, om, _ = orc.unary_topk(h, Wlm, K, output_multiplier=m, final_logit_softcapping=c)
    what = f"map{P}x{D}x{V}k{K}"
    compare_topk(gi, gv, oi, ov, om, what).check(what)
    compare_topk_values(gi, gv, oi, ov, what + " vals")
    assert np.array_equal(gi, gi0)
    x = np.float32(m) * gv0.astype(np.float64)
    want = np.float32(c) * np.tanh(x / np.float32(c)) if c > 0 else x
    assert np.allclose(gv, want, rtol=1e-6, atol=1e-6 * max(c, 1.0)), np.abs(gv - want).max()
    if c > 0:
        assert np.all(np.abs(gv) <= np.float32(c))


def saturating_case(seed, P, D, V, K, n_sat=6):
    """Exact logits with a saturating cap: h[p] is one-hot on column p % D, so
    U[p, v] = W_lm[v, p % D] exactly.  Per column, n_sat tokens get logits 20, 20.5,
    ... (tanh rounds every one of them to exactly 1 in fp32) with larger ids
    holding larger raw logits, then K - n_sat tokens sit well apart in (0.3, 0.5),
    and every other token below 0.2: the kept set is clear, but the saturated
    entries tie and must come out in id order, not in raw-logit order."""
    rng = _rng(seed)
    Wf = rng.uniform(-0.2, 0.2, size=(V, D)).astype(np.float32)
    for c in range(min(P, D)):
        ids = np.sort(rng.choice(V, size=K, replace=False))
        sat, mid = ids[:n_sat], rng.permutation(ids[n_sat:])
        Wf[sat, c] = 20.0 + 0.5 * np.arange(n_sat)
        Wf[mid, c] = 0.3 + 0.0125 * np.arange(K - n_sat)
    h = np.zeros((P, D), np.float32)
    h[np.arange(P), np.arange(P) % D] = 1.0
    return W.f32_to_bf16_bits(h), W.f32_to_bf16_bits(Wf)


@pytest.mark.parametrize("P,D,V,K", [
    (8, 256, 5000, 16),      # the streaming head: merge of the per-CTA lists
    (140, 256, 5000, 16),    # the tensor-core GEMM for many positions
    (20, 256, 3000, 100),    # K > 64: the CUDA-core path
])
def test_head_saturating_cap_ties_break_to_lower_id(orc, df2, P, D, V, K):
    h, Wlm = saturating_case(P + V + K, P, D, V, K)
    ids, vals, _ = df2.unary_topk(bf_dev(h), bf_dev(Wlm), K, output_multiplier=1.0, final_logit_softcapping=1.0)
    torch.cuda.synchronize()
    oi, ov, om, _ = orc.unary_topk(h, Wlm, K, output_multiplier=1.0, final_logit_softcapping=1.0)
    assert (ov[:, :6] == 1.0).all() and (om > 1e-3).all()
    assert np.array_equal(host(ids), oi)
    assert np.array_equal(host(vals)[:, :6], ov[:, :6])
    close(host(vals), ov, what="saturating cap vals")


def test_draft_head_saturating_cap_ties_break_to_lower_id(orc, df2):
    R, B, D, V, K, r = 2, 8, 256, 5000, 16, 64
    h, Wlm = saturating_case(7, R * B, D, V, K)
    rng = _rng(8)
    WH, A, Bc = rand_bf16(rng, (r, D), 0.02), rand_bf16(rng, (V, r), 0.3), rand_bf16(rng, (V, r), 0.3)
    anchors = rng.integers(0, V, R).astype(np.int32)
    out = df2.draft_head(bf_dev(h), bf_dev(Wlm), K, bf_dev(WH), bf_dev(A), bf_dev(Bc), dev(anchors), B,
                         output_multiplier=1.0, final_logit_softcapping=1.0)
    torch.cuda.synchronize()
    oi, ov, om, oG = orc.unary_topk(h, Wlm, K, W_H=WH, output_multiplier=1.0, final_logit_softcapping=1.0)
    assert np.array_equal(host(out[0]), oi)
    op, os_, omg, _ = orc.selector_walk(anchors, oi, ov, oG, A, Bc, B)
    compare_walk(host(out[3]), host(out[4]), op, os_, omg, "capped walk").check("capped walk")


def test_head_logit_map_defaults_are_the_identity(df2):
    """m = 1, c = 0 leaves every value bit for bit as the call without the map."""
    rng = _rng(3)
    h = bf_dev(rand_bf16(rng, (8, 512)))
    Wlm = bf_dev(rand_bf16(rng, (9000, 512), 0.02))
    a = df2.unary_topk(h, Wlm, 16, output_multiplier=1.0, final_logit_softcapping=0.0)
    b = df2.unary_topk(h, Wlm, 16)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_head_empty(df2):
    h = torch.empty((0, 64), dtype=torch.bfloat16, device="cuda")
    Wlm = torch.zeros((100, 64), dtype=torch.bfloat16, device="cuda")
    ids, vals, _ = df2.unary_topk(h, Wlm, 4)
    assert ids.shape == (0, 4)


# -------------------------------------------------------------- selector ----

def lattice(rng, R, B, K, V, r, cb_std=0.3):
    ids = np.stack([rng.choice(V, size=K, replace=False) for _ in range(R * B)]).astype(np.int32)
    vals = -np.sort(-rng.standard_normal((R * B, K)).astype(np.float32), axis=-1)
    G = rng.standard_normal((R * B, r)).astype(np.float32)
    A = rand_bf16(rng, (V, r), cb_std)
    Bc = rand_bf16(rng, (V, r), cb_std)
    anchors = rng.integers(0, V, size=R).astype(np.int32)
    return anchors, ids, vals, G, A, Bc


def run_walk(df2, anchors, ids, vals, G, A, Bc, B):
    path, score = df2.selector_walk(dev(anchors), dev(ids), dev(vals), dev(G), bf_dev(A), bf_dev(Bc), B)
    torch.cuda.synchronize()
    return host(path), host(score)


def check_walk(orc, df2, anchors, ids, vals, G, A, Bc, B, what="walk"):
    gp, gs = run_walk(df2, anchors, ids, vals, G, A, Bc, B)
    op, os_, om, st = orc.selector_walk(anchors, ids, vals, G, A, Bc, B)
    assert st == 0
    rep = compare_walk(gp, gs, op, os_, om, what)
    rep.check(what)
    check_path_valid(orc, gp, anchors, ids, vals, G, A, Bc, B)
    return rep


@pytest.mark.parametrize("R,B,K,V,r", [
    (2, 8, 4, 4096, 32),
    (3, 2, 1, 500, 8),
    (5, 16, 17, 3000, 264),
    (4, 8, 64, 10000, 512),
    (1, 5, 16, 2000, 1024),
    (37, 8, 16, 5000, 256),
    (3, 6, 12, 1500, 2000),     # gathers past shared memory, 8 rank chunks, ragged
    (2, 4, 8, 1000, 4096),      # the largest rank: 16 chunks
])
def test_walk_shapes(orc, df2, R, B, K, V, r):
    rng = _rng(R * 1000 + B * 100 + K + r)
    check_walk(orc, df2, *lattice(rng, R, B, K, V, r), B, f"walk{R}x{B}k{K}r{r}")


@pytest.mark.parametrize("P,K,V,r", [(16, 4, 4096, 32), (77, 16, 3000, 256), (9, 64, 900, 520),
                                     (5, 8, 700, 4096)])
def test_pair_scores_shapes(orc, df2, P, K, V, r):
    rng = _rng(P + K + r)
    _, ids, vals, G, A, Bc = lattice(rng, P, 1, K, V, r)
    pred = rng.integers(0, V, size=P).astype(np.int32)
    gs = host(df2.selector_pair_scores(dev(pred), dev(ids), dev(vals), dev(G), bf_dev(A), bf_dev(Bc)))
    os_, st = orc.pair_scores(pred, ids, vals, G, A, Bc)
    assert st == 0
    close(gs, os_, what="pair scores")


def test_walk_replay_through_teacher_forced_gpu(df2):
    """Replaying the GPU walk's predecessors through the GPU teacher-forced scorer
    gives back the GPU path (verl-SpeCo PR #62, 'Selector training objective')."""
    rng = _rng(11)
    R, B, K, V, r = 8, 8, 16, 3000, 256
    anchors, ids, vals, G, A, Bc = lattice(rng, R, B, K, V, r)
    gp, gs = run_walk(df2, anchors, ids, vals, G, A, Bc, B)
    pred = np.concatenate([anchors[:, None], anchors[:, None], gp[:, :-1]], axis=1).reshape(-1)
    sc = host(df2.selector_pair_scores(dev(pred.astype(np.int32)), dev(ids), dev(vals), dev(G),
                                       bf_dev(A), bf_dev(Bc))).reshape(R, B, K)
    idsr = ids.reshape(R, B, K)
    for q in range(R):
        for t in range(1, B):
            j = max(range(K), key=lambda jj: (sc[q, t, jj], -idsr[q, t, jj]))
            assert idsr[q, t, j] == gp[q, t - 1]
            assert sc[q, t, j] == gs[q, t - 1]


def test_zero_successor_codebook_gives_unary_argmax_gpu(df2):
    rng = _rng(12)
    R, B, K, V, r = 6, 8, 16, 2000, 256
    anchors, ids, vals, G, A, Bc = lattice(rng, R, B, K, V, r)
    gp, gs = run_walk(df2, anchors, ids, vals, G, A, np.zeros_like(Bc), B)
    assert np.array_equal(gp, ids.reshape(R, B, K)[:, 1:, 0])
    assert np.array_equal(gs, vals.reshape(R, B, K)[:, 1:, 0])


def test_bad_ids_flagged(df2):
    rng = _rng(13)
    R, B, K, V, r = 3, 4, 4, 100, 32
    anchors, ids, vals, G, A, Bc = lattice(rng, R, B, K, V, r)
    anchors[1] = V + 5
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    path, score = df2.selector_walk(dev(anchors), dev(ids), dev(vals), dev(G), bf_dev(A), bf_dev(Bc), B,
                                    dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & df2.DF2_STATUS_ID_OUT_OF_RANGE
    path, score = host(path), host(score)
    assert np.all(path[1] == -1) and np.all(np.isnan(score[1])) and np.all(path[0] >= 0)
    status.zero_()
    pred = np.zeros(R * B, np.int32)
    pred[2] = -3
    s = host(df2.selector_pair_scores(dev(pred), dev(ids), dev(vals), dev(G), bf_dev(A), bf_dev(Bc),
                                      dev_status=status))
    torch.cuda.synchronize()
    assert int(status.item()) & df2.DF2_STATUS_ID_OUT_OF_RANGE
    assert np.all(np.isnan(s[2])) and not np.isnan(np.delete(s, 2, axis=0)).any()


def test_tiny_walk_strong_and_weak_selector(orc, df2):
    w = W.TINY
    for std in (None, 0.3):
        inp = W.head_inputs(w, selector_std=std)
        oi, ov, _, oG = orc.unary_topk(inp["h"], inp["W_lm"], w.K, W_H=inp["W_H"])
        check_walk(orc, df2, inp["anchors"], oi, ov, oG, inp["A"], inp["Bc"], w.B, f"tiny walk {std}")
        gs = host(df2.selector_pair_scores(dev(inp["pred"]), dev(oi), dev(ov), dev(oG), bf_dev(inp["A"]),
                                           bf_dev(inp["Bc"])))
        os_, _ = orc.pair_scores(inp["pred"], oi, ov, oG, inp["A"], inp["Bc"])
        close(gs, os_, what="tiny pair")


def test_tiny_chain(orc, df2):
    """GPU head -> GPU walk against oracle head -> oracle walk."""
    w = W.TINY
    inp = W.head_inputs(w, selector_std=0.3)
    gi, gv, gG = run_head(df2, inp["h"], inp["W_lm"], w.K, inp["W_H"])
    gp, gs = run_walk(df2, inp["anchors"], gi, gv, gG, inp["A"], inp["Bc"], w.B)
    oi, ov, om, oG = orc.unary_topk(inp["h"], inp["W_lm"], w.K, W_H=inp["W_H"])
    op, os_, omg, _ = orc.selector_walk(inp["anchors"], oi, ov, oG, inp["A"], inp["Bc"], w.B)
    compare_topk(gi, gv, oi, ov, om).check("chain topk")
    compare_walk(gp, gs, op, os_, omg).check("chain walk")


# ------------------------------------------------------------------ conv ----

def run_conv(df2, x, z, B, taps, g, Wp, base):
    xd = bf_dev(x) if x.dtype == np.uint16 else dev(x)
    zd = bf_dev(z) if z.dtype == np.uint16 else dev(z)
    y, dyn = df2.conv_prepare(xd, B, taps, g, bf_dev(Wp), dev(base))
    y2 = df2.conv_finish(zd, B, taps, g, dyn, dev(base))
    torch.cuda.synchronize()
    conv = host_bf if x.dtype == np.uint16 else host
    return conv(y), host(dyn), conv(y2)


def check_conv(orc, df2, x, z, B, taps, g, Wp, base, what="conv"):
    gy, gd, gy2 = run_conv(df2, x, z, B, taps, g, Wp, base)
    oy, od = orc.conv_prepare(x, B, taps, g, Wp, base)
    close(gd, od, what=what + " dyn_out")
    # finish on the oracle's own correction and on the GPU's, so finish is judged alone
    oy2 = orc.conv_finish(z, B, taps, g, od, base)
    if x.dtype == np.uint16:
        close_bf16(gy, oy, what=what + " y")
        close_bf16(gy2, oy2, what=what + " finish")
    else:
        close(gy, oy, what=what + " y")
        close(gy2, oy2, what=what + " finish")


def test_tiny_conv(orc, df2):
    w = W.TINY
    c = W.conv_inputs(w)
    check_conv(orc, df2, c["x"], c["z"], w.B, w.taps, w.g, c["W_proj"], c["base"], "tiny conv")


@pytest.mark.parametrize("P,C,B,taps,g,dt", [
    (16, 64, 8, 2, 16, "bf16"),
    (24, 264, 8, 1, 8, "bf16"),
    (30, 48, 5, 5, 4, "f32"),       # taps = block
    (32, 128, 16, 4, 16, "bf16"),
    (27, 40, 9, 3, 2, "f32"),       # groups narrower than a 16-byte chunk
    (64, 512, 8, 6, 64, "bf16"),    # generic-taps path
    (8, 8, 8, 8, 8, "f32"),
    (136, 264, 8, 3, 8, "bf16"),    # many rows: tensor-core projection, column split not /16
    (80, 512, 16, 4, 16, "bf16"),   # many rows, taps 4
    (72, 40, 9, 2, 4, "f32"),       # many fp32 rows: CUDA-core projection
    # many bf16 rows: the fused tensor-core prepare (projection, dyn_out and apply in one kernel)
    (200, 512, 8, 2, 16, "bf16"),   # CTA pairs, ragged last row tile
    (72, 256, 8, 1, 8, "bf16"),     # one row tile, taps 1
    (384, 1024, 8, 3, 32, "bf16"),  # taps 3, three row tiles (the last pair's second CTA idle)
    (640, 512, 8, 2, 4, "bf16"),    # groups narrower than an 8-channel chunk
    (1032, 256, 8, 2, 16, "bf16"),  # nine row tiles, the last one 8 rows
    (256, 512, 32, 4, 16, "bf16"),  # blocks of 32, taps 4
    (96, 256, 16, 3, 16, "bf16"),   # one partial row tile, blocks of 16
    (5120, 512, 8, 3, 4, "bf16"),   # a last round of half tiles (clusters of two pairs)
    (5376, 512, 8, 3, 4, "bf16"),   # a last round of half tiles (CTA pairs)
])
def test_conv_shapes(orc, df2, P, C, B, taps, g, dt):
    rng = _rng(P * 13 + C + taps * 7 + g)
    G = C // g
    if dt == "bf16":
        x, z = rand_bf16(rng, (P, C)), rand_bf16(rng, (P, C))
    else:
        x = rng.standard_normal((P, C)).astype(np.float32)
        z = rng.standard_normal((P, C)).astype(np.float32)
    Wp = rand_bf16(rng, (2 * taps * G, C), 0.05)
    base = (rng.standard_normal((2, taps, C)) * 0.3).astype(np.float32)
    base[:, 0] += 1
    check_conv(orc, df2, x, z, B, taps, g, Wp, base, f"conv{P}x{C}b{B}t{taps}g{g}{dt}")


@pytest.mark.parametrize("P,C,B,taps,g", [(200, 512, 8, 2, 16), (1032, 256, 8, 2, 16), (256, 512, 32, 4, 16)])
def test_conv_prepare_many_rows_is_one_kernel(df2, P, C, B, taps, g):
    """Many bf16 rows: conv prepare is a single launch (the corrections for the
    conv it applies never leave the chip)."""
    rng = _rng(P + C)
    x = bf_dev(rand_bf16(rng, (P, C)))
    Wp = bf_dev(rand_bf16(rng, (2 * taps * (C // g), C), 0.05))
    base = dev((rng.standard_normal((2, taps, C)) * 0.3).astype(np.float32))
    df2.conv_prepare(x, B, taps, g, Wp, base)
    torch.cuda.synchronize()
    before = df2.kernels_launched()
    df2.conv_prepare(x, B, taps, g, Wp, base)
    torch.cuda.synchronize()
    assert df2.kernels_launched() - before == 1


@pytest.mark.parametrize("P", [32, 256])   # few rows; many rows (the fused tensor-core prepare)
def test_conv_identity_and_locality_gpu(df2, P):
    rng = _rng(21)
    C, B, taps, g = 256, 8, 2, 16
    x = rand_bf16(rng, (P, C))
    base = np.zeros((2, taps, C), np.float32)
    base[:, 0] = 1
    Wp = np.zeros((2 * taps * (C // g), C), np.uint16)
    y, dyn, y2 = run_conv(df2, x, x, B, taps, g, Wp, base)
    assert np.array_equal(y, x) and np.array_equal(y2, x) and not dyn.any()
    # block locality: perturb the last row of block 1
    Wp = rand_bf16(rng, (2 * taps * (C // g), C), 0.05)
    base = (rng.standard_normal((2, taps, C)) * 0.3).astype(np.float32)
    a = run_conv(df2, x, x, B, taps, g, Wp, base)
    x2 = x.copy()
    x2[2 * B - 1] = rand_bf16(rng, (C,), 30.0)
    b = run_conv(df2, x2, x2, B, taps, g, Wp, base)
    for u, v in zip(a, b):
        assert np.array_equal(u[2 * B:], v[2 * B:]) and np.array_equal(u[:B], v[:B])


# ------------------------------------------------------ full-size workloads ----

def _sample_rows(P, n, extra=()):
    rows = sorted(set(np.linspace(0, P - 1, n).astype(int).tolist()) | set(int(e) for e in extra))
    return np.asarray(rows)


@pytest.mark.parametrize("name", ["batch1", "batched", "stress"])
def test_full_size_selector(orc, df2, name):
    w = W.BY_NAME[name]
    rng = _rng(w.seed + 100)
    anchors, ids, vals, G, A, Bc = lattice(rng, w.R, w.B, w.K, w.V, w.r, cb_std=0.3)
    check_walk(orc, df2, anchors, ids, vals, G, A, Bc, w.B, name + " walk")
    pred = rng.integers(0, w.V, size=w.P).astype(np.int32)
    gs = host(df2.selector_pair_scores(dev(pred), dev(ids), dev(vals), dev(G), bf_dev(A), bf_dev(Bc)))
    os_, _ = orc.pair_scores(pred, ids, vals, G, A, Bc)
    close(gs, os_, what=name + " pair")


@pytest.mark.parametrize("name", ["batch1", "conv", "stress"])
def test_full_size_conv(orc, df2, name):
    w = W.BY_NAME[name]
    c = W.conv_inputs(w)
    gy, gd, gy2 = run_conv(df2, c["x"], c["z"], w.B, w.taps, w.g, c["W_proj"], c["base"])
    nb = w.P // w.B
    blocks = _sample_rows(nb, 16)
    rows = (blocks[:, None] * w.B + np.arange(w.B)[None, :]).reshape(-1)
    x, z = c["x"][rows], c["z"][rows]
    oy, od = orc.conv_prepare(x, w.B, w.taps, w.g, c["W_proj"], c["base"])
    close(gd[rows], od, what=name + " dyn_out")
    close_bf16(gy[rows], oy, what=name + " y")
    oy2 = orc.conv_finish(z, w.B, w.taps, w.g, od, c["base"])
    close_bf16(gy2[rows], oy2, what=name + " finish")


# ------------------------------------------------------- failure detection ----

def test_bounded_wait_reports_timeout_and_device_stays_usable(df2):
    """A pipeline stage whose copies are never issued: the tensor-core head's
    bounded waits must give up, report DF2_STATUS_WAIT_TIMEOUT and leave the
    device usable for the next call (no trap, no fault)."""
    import ctypes as ct
    lib = df2.lib()
    P, D, V, K = 8, 256, 4096, 16
    h = torch.randn(P, D, device="cuda").to(torch.bfloat16)
    Wlm = (torch.randn(V, D, device="cuda") * 0.02).to(torch.bfloat16)
    ids = torch.empty(P, K, dtype=torch.int32, device="cuda")
    vals = torch.empty(P, K, dtype=torch.float32, device="cuda")
    nb = df2.unary_topk_workspace_size(P, D, V, K)
    ws = torch.empty(nb, dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    stream = ct.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = lib.dflash2_selftest_wait_timeout(ct.c_void_p(h.data_ptr()), P, D, ct.c_void_p(Wlm.data_ptr()), V, K,
                                           ct.c_void_p(ids.data_ptr()), ct.c_void_p(vals.data_ptr()),
                                           ct.c_void_p(ws.data_ptr()), nb, ct.c_void_p(status.data_ptr()),
                                           stream)
    assert rc == 0
    torch.cuda.synchronize()
    assert int(status.item()) & df2.DF2_STATUS_WAIT_TIMEOUT
    # the same call without the stall works right after, with no timeout
    status.zero_()
    ids2, vals2, _ = df2.unary_topk(h, Wlm, K, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref = torch.topk((h.float() @ Wlm.float().T), K, dim=1)
    assert (ids2.long() == ref.indices).float().mean() > 0.9
