"""The fused draft-head call against the separate calls it stands for (bit-identical
outputs) and against the oracle, through the C-ABI."""
import numpy as np
import pytest

import workloads as W
from parity import compare_topk, compare_walk

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
    return None if t is None else t.cpu().numpy()


def inputs(seed, R, B, D, V, K, r, cb_std=0.3):
    rng = np.random.default_rng(seed)
    bf = lambda shape, std: W.f32_to_bf16_bits((rng.standard_normal(shape) * std).astype(np.float32))
    return dict(h=bf((R * B, D), 1.0), W_lm=bf((V, D), 0.02), W_H=bf((r, D), 0.02), A=bf((V, r), cb_std),
                Bc=bf((V, r), cb_std), anchors=rng.integers(0, V, R).astype(np.int32),
                pred=rng.integers(0, V, R * B).astype(np.int32), K=K, B=B, R=R, V=V)


def fused(df2, x, with_pred=True, status=None):
    out = df2.draft_head(bf_dev(x["h"]), bf_dev(x["W_lm"]), x["K"], bf_dev(x["W_H"]), bf_dev(x["A"]),
                         bf_dev(x["Bc"]), dev(x["anchors"]), x["B"],
                         dev(x["pred"]) if with_pred else None, dev_status=status,
                         output_multiplier=x.get("m", 1.0), final_logit_softcapping=x.get("c", 0.0))
    torch.cuda.synchronize()
    return [host(t) for t in out]


def separate(df2, x, status=None):
    h, Wlm, WH, A, Bc = (bf_dev(x[k]) for k in ("h", "W_lm", "W_H", "A", "Bc"))
    ids, vals, G = df2.unary_topk(h, Wlm, x["K"], WH, dev_status=status, output_multiplier=x.get("m", 1.0),
                                  final_logit_softcapping=x.get("c", 0.0))
    path, ps = df2.selector_walk(dev(x["anchors"]), ids, vals, G, A, Bc, x["B"], dev_status=status)
    pair = df2.selector_pair_scores(dev(x["pred"]), ids, vals, G, A, Bc, dev_status=status)
    torch.cuda.synchronize()
    return [host(t) for t in (ids, vals, G, path, ps, pair)]


@pytest.mark.parametrize("R,B,D,V,K,r", [
    (1, 8, 4096, 151936, 16, 256),   # the batch-1 shape: skinny head + fused tail
    (2, 8, 256, 4096, 4, 32),        # the tiny shape
    (1, 16, 512, 20000, 64, 512),    # K = 64: the separate calls
    (2, 16, 512, 20000, 32, 512),    # K = 32, a 16-CTA cluster
    (2, 8, 520, 9001, 17, 264),      # ragged K, D and r
    (2, 8, 256, 9000, 13, 128),      # K < 16 and not a multiple of 4
    (2, 8, 256, 20000, 32, 1280),    # a slot's predecessor rows too large to send: the L2 prefetch path
    (16, 8, 256, 30000, 16, 256),    # 128 positions: the tensor-core GEMM head + fused tail
    (64, 8, 256, 20000, 16, 256),    # 512 positions: 64 clusters
])
def test_fused_equals_separate_calls(df2, R, B, D, V, K, r):
    x = inputs(R * 7 + K + r, R, B, D, V, K, r)
    got = fused(df2, x)
    want = separate(df2, x)
    for name, g, w in zip(["ids", "vals", "G", "path", "path_scores", "pair_scores"], got, want):
        assert np.array_equal(g, w, equal_nan=True), name


@pytest.mark.parametrize("R,B,D,V,K,r,m,c", [
    (1, 8, 4096, 151936, 16, 256, 1.25, 20.0),   # the batch-1 shape, capped logits
    (16, 8, 256, 30000, 16, 256, 0.5, 2.0),      # the tensor-core GEMM head
    (1, 16, 512, 20000, 64, 512, 2.0, 0.0),      # K = 64 (the separate calls), multiplier only
])
def test_fused_with_logit_map_equals_separate_calls(df2, R, B, D, V, K, r, m, c):
    x = inputs(R * 5 + K + r, R, B, D, V, K, r)
    x["m"], x["c"] = m, c
    got = fused(df2, x)
    want = separate(df2, x)
    for name, g, w in zip(["ids", "vals", "G", "path", "path_scores", "pair_scores"], got, want):
        assert np.array_equal(g, w, equal_nan=True), name


@pytest.mark.parametrize("m,c", [(1.0, 0.0), (1.5, 3.0)])
def test_fused_against_the_oracle(orc, df2, m, c):
    R, B, D, V, K, r = 3, 8, 256, 3000, 16, 64
    x = inputs(99, R, B, D, V, K, r)
    x["m"], x["c"] = m, c
    ids, vals, G, path, ps, pair = fused(df2, x)
    oi, ov, om, oG = orc.unary_topk(x["h"], x["W_lm"], K, W_H=x["W_H"], output_multiplier=m,
                                    final_logit_softcapping=c)
    compare_topk(ids, vals, oi, ov, om, "fused topk").check("fused topk")
    op, os_, omg, _ = orc.selector_walk(x["anchors"], oi, ov, oG, x["A"], x["Bc"], B)
    compare_walk(path, ps, op, os_, omg, "fused walk").check("fused walk")


def test_fused_without_pred(df2):
    x = inputs(5, 1, 8, 512, 8000, 16, 128)
    got = fused(df2, x, with_pred=False)
    want = separate(df2, x)
    assert got[5] is None
    for g, w in zip(got[:5], want[:5]):
        assert np.array_equal(g, w)


def test_fused_bad_ids_flagged(df2):
    x = inputs(6, 2, 8, 256, 4000, 16, 64)
    x["anchors"][1] = x["V"] + 3
    x["pred"][5] = -2
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ids, vals, G, path, ps, pair = fused(df2, x, status=status)
    assert int(status.item()) & df2.DF2_STATUS_ID_OUT_OF_RANGE
    assert np.all(path[1] == -1) and np.all(np.isnan(ps[1])) and np.all(path[0] >= 0)
    assert np.all(np.isnan(pair[5])) and not np.isnan(np.delete(pair, 5, axis=0)).any()


def test_fused_repeated_calls_reuse_the_workspace(df2):
    """Calls on a workspace that starts as garbage, repeated, give the same results."""
    x = inputs(7, 2, 8, 512, 8000, 16, 128)
    ws = torch.empty(df2.draft_head_workspace_size(2, 8, 512, 8000, 16, 128), dtype=torch.uint8, device="cuda")
    ws.fill_(0xAB)
    args = (bf_dev(x["h"]), bf_dev(x["W_lm"]), 16, bf_dev(x["W_H"]), bf_dev(x["A"]), bf_dev(x["Bc"]),
            dev(x["anchors"]), 8, dev(x["pred"]))
    first = [host(t) for t in df2.draft_head(*args, workspace=ws)]
    for _ in range(3):
        again = [host(t) for t in df2.draft_head(*args, workspace=ws)]
        for g, w in zip(again, first):
            assert np.array_equal(g, w)
