"""The fused conv finish -> next conv prepare, through the C-ABI: bit-identical to
dflash2_conv_finish, a separate elementwise add of the residual in the activation
dtype, and dflash2_conv_prepare; and within the parity tolerance of the oracle."""
import numpy as np
import pytest

from parity import close, close_bf16

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


def act_dev(a):
    return bf_dev(a) if a.dtype == np.uint16 else dev(a)


def act_host(t):
    if t.dtype == torch.bfloat16:
        return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy()


def inputs(seed, P, C, B, taps, g, dt, with_res):
    import workloads as W
    rng = np.random.default_rng(seed)
    G = C // g
    if dt == "bf16":
        act = lambda s: W.f32_to_bf16_bits((rng.standard_normal((P, C)) * s).astype(np.float32))
    else:
        act = lambda s: (rng.standard_normal((P, C)) * s).astype(np.float32)
    base = (rng.standard_normal((2, taps, C)) * 0.3).astype(np.float32)
    base[:, 0] += 1
    base_next = (rng.standard_normal((2, taps, C)) * 0.3).astype(np.float32)
    base_next[:, 0] += 1
    return dict(z=act(1.0), res=act(1.0) if with_res else None,
                dyn=(rng.standard_normal((P, taps, G)) * 0.1).astype(np.float32),
                base=base, base_next=base_next,
                Wp=W.f32_to_bf16_bits((rng.standard_normal((2 * taps * G, C)) * 0.05).astype(np.float32)))


def fused(df2, x, B, taps, g):
    res = None if x["res"] is None else act_dev(x["res"])
    h, y, d = df2.conv_finish_prepare(act_dev(x["z"]), B, taps, g, dev(x["dyn"]), dev(x["base"]),
                                      bf_dev(x["Wp"]), dev(x["base_next"]), res)
    torch.cuda.synchronize()
    return act_host(h), act_host(y), d.cpu().numpy()


def separate(df2, x, B, taps, g):
    h = df2.conv_finish(act_dev(x["z"]), B, taps, g, dev(x["dyn"]), dev(x["base"]))
    if x["res"] is not None:
        h = h + act_dev(x["res"])      # the elementwise add in the activation dtype
    y, d = df2.conv_prepare(h, B, taps, g, bf_dev(x["Wp"]), dev(x["base_next"]))
    torch.cuda.synchronize()
    return act_host(h), act_host(y), d.cpu().numpy()


SHAPES = [
    (8, 4096, 8, 2, 16, "bf16"),     # the batch-1 layer: one fused kernel
    (16, 64, 8, 2, 16, "bf16"),
    (30, 48, 5, 5, 4, "f32"),        # taps = block
    (27, 40, 9, 3, 2, "f32"),        # groups narrower than a 16-byte chunk
    (64, 512, 8, 6, 64, "bf16"),     # generic taps
    (32, 128, 16, 4, 16, "bf16"),    # block 16
    (136, 264, 8, 3, 8, "bf16"),     # many rows: finish kernel, then the prepare path
    (72, 40, 9, 2, 4, "f32"),        # many fp32 rows
]


@pytest.mark.parametrize("with_res", [True, False])
@pytest.mark.parametrize("P,C,B,taps,g,dt", SHAPES)
def test_fused_equals_separate_calls(df2, P, C, B, taps, g, dt, with_res):
    x = inputs(P * 31 + C + taps + int(with_res), P, C, B, taps, g, dt, with_res)
    got = fused(df2, x, B, taps, g)
    want = separate(df2, x, B, taps, g)
    for name, a, b in zip(["h", "y_next", "dyn_out_next"], got, want):
        assert np.array_equal(a, b), name


@pytest.mark.parametrize("P,C,B,taps,g,dt", [(16, 64, 8, 2, 16, "bf16"), (27, 40, 9, 3, 2, "f32"),
                                             (136, 264, 8, 3, 8, "bf16")])
def test_fused_against_the_oracle(orc, df2, P, C, B, taps, g, dt):
    x = inputs(P + C * 3, P, C, B, taps, g, dt, True)
    gh, gy, gd = fused(df2, x, B, taps, g)
    oh, oy, od = orc.conv_finish_prepare(x["z"], B, taps, g, x["dyn"], x["base"], x["Wp"], x["base_next"],
                                         residual=x["res"])
    cmp = close_bf16 if dt == "bf16" else close
    cmp(gh, oh, what="h")
    close(gd, od, what="dyn_out_next")
    cmp(gy, oy, what="y_next")


def test_fused_identity_convs(df2):
    """Identity convs and zero projections: h = z + residual (exact for these
    quarter-integer values) and y_next = h, dyn_out_next = 0."""
    import workloads as W
    rng = np.random.default_rng(4)
    P, C, B, taps, g = 16, 256, 8, 2, 16
    z = rng.integers(-4, 5, size=(P, C)) * 0.25
    r = rng.integers(-4, 5, size=(P, C)) * 0.25
    base = np.zeros((2, taps, C), np.float32)
    base[:, 0] = 1
    x = dict(z=W.f32_to_bf16_bits(z.astype(np.float32)), res=W.f32_to_bf16_bits(r.astype(np.float32)),
             dyn=np.zeros((P, taps, C // g), np.float32), base=base, base_next=base,
             Wp=np.zeros((2 * taps * (C // g), C), np.uint16))
    h, y, d = fused(df2, x, B, taps, g)
    assert np.array_equal(W.bf16_bits_to_f32(h), (z + r).astype(np.float32))
    assert np.array_equal(y, h) and not d.any()
