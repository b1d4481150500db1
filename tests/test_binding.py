"""The Python binding's argument checks, on the CPU.

A tensor the kernels would write or read out of bounds (a caller's `out` of the
wrong size or type, a short workspace, a status word of the wrong type, weights of
the wrong shape, tensors of two devices) has to raise in Python before the library
is called: on a GPU it would be a memory fault, not an error.  Here every wrapper
runs against a stand-in for the library that records its arguments, with CPU
tensors standing in for device tensors, so the checks and the marshalling are
exercised without a GPU."""
import ctypes as ct

import pytest

torch = pytest.importorskip("torch")

import dflash2_draft_block_gb300 as df2  # noqa: E402


class FakeLib:
    """Records each call; status 0; workspace queries answer 256 bytes."""

    def __init__(self):
        self.calls = []

    def __getattr__(self, name):
        if name.endswith("_workspace_size"):
            return lambda *a: 256
        if name == "dflash2_status_string":
            return lambda code: b"DF2_TEST"

        def call(*args):
            self.calls.append((name, args))
            return 0
        return call


@pytest.fixture
def fake(monkeypatch):
    lib = FakeLib()
    monkeypatch.setattr(df2, "lib", lambda: lib)
    monkeypatch.setattr(df2, "_on_device", lambda t: True)
    monkeypatch.setattr(df2, "_stream", lambda stream, device: ct.c_void_p(0))
    return lib


def bf(*shape):
    return torch.zeros(shape, dtype=torch.bfloat16)


def f32(*shape):
    return torch.zeros(shape, dtype=torch.float32)


def i32(*shape):
    return torch.zeros(shape, dtype=torch.int32)


P, D, V, K, r, R, B = 16, 64, 500, 4, 32, 2, 8


def head_args():
    return bf(P, D), bf(V, D), K, bf(r, D)


def sel_args():
    return i32(R), i32(R * B, K), f32(R * B, K), f32(R * B, r), bf(V, r), bf(V, r)


# ------------------------------------------------------------- valid calls --

def test_valid_calls_reach_the_library_with_their_outputs(fake):
    ids, vals, G = df2.unary_topk(*head_args())
    assert ids.shape == (P, K) and vals.shape == (P, K) and G.shape == (P, r)
    path, ps = df2.selector_walk(*sel_args(), B)
    assert path.shape == (R, B - 1) and ps.shape == (R, B - 1)
    s = df2.selector_pair_scores(i32(R * B), *sel_args()[1:])
    assert s.shape == (R * B, K)
    loss, label = df2.selector_ce(f32(P, K), i32(P, K), i32(P), V)
    assert loss.shape == (P,) and label.dtype == torch.int32
    out = df2.draft_head(bf(R * B, D), bf(V, D), K, bf(r, D), bf(V, r), bf(V, r), i32(R), B, i32(R * B))
    assert [tuple(t.shape) for t in out] == [(R * B, K), (R * B, K), (R * B, r), (R, B - 1), (R, B - 1), (R * B, K)]
    lat = df2.selector_lattice(*sel_args(), B)
    assert lat.shape == (R, B - 1, K, K)
    path, ps = df2.lattice_walk(lat, i32(R * B, K), B, V, uniforms=f32(R, B - 1))
    assert path.shape == (R, B - 1)
    C, taps, g = 64, 2, 16
    y, dyn = df2.conv_prepare(bf(P, C), 8, taps, g, bf(2 * taps * C // g, C), f32(2, taps, C))
    assert y.shape == (P, C) and dyn.shape == (P, taps, C // g)
    y2 = df2.conv_finish(bf(P, C), 8, taps, g, dyn, f32(2, taps, C))
    assert y2.shape == (P, C)
    h, yn, dn = df2.conv_finish_prepare(bf(P, C), 8, taps, g, dyn, f32(2, taps, C), bf(2 * taps * C // g, C),
                                        f32(2, taps, C), residual=bf(P, C))
    assert h.shape == yn.shape == (P, C) and dn.shape == (P, taps, C // g)
    names = [n for n, _ in fake.calls]
    assert names == ["dflash2_unary_topk", "dflash2_selector_walk", "dflash2_selector_pair_scores",
                     "dflash2_selector_ce", "dflash2_draft_head", "dflash2_selector_lattice",
                     "dflash2_lattice_walk", "dflash2_conv_prepare", "dflash2_conv_finish",
                     "dflash2_conv_finish_prepare"]


def test_no_alloc_call_checks_its_inputs_and_outputs(fake):
    ids, vals, G = df2.unary_topk_noalloc(*head_args())
    assert ids.shape == (P, K) and G.shape == (P, r)
    assert fake.calls[-1][0] == "dflash2_unary_topk_noalloc"
    n = len(fake.calls)
    with pytest.raises(ValueError):
        df2.unary_topk_noalloc(bf(P, D), bf(V, D + 8), K)                  # W_lm not [V, D]
    with pytest.raises(ValueError):
        df2.unary_topk_noalloc(bf(P, D), bf(V, D), K, bf(r, D - 8))         # W_H not [r, D]
    with pytest.raises(ValueError):
        df2.unary_topk_noalloc(*head_args(), out=(i32(P, K), f32(P, K), f32(P, r - 1)))
    assert len(fake.calls) == n


def test_workspace_sizes_are_passed_in_bytes(fake):
    ws = torch.zeros(64, dtype=torch.float32)   # 256 bytes in 64 elements
    df2.unary_topk(*head_args(), workspace=ws)
    assert fake.calls[-1][1][14] == 256      # (…, workspace, workspace_bytes, dev_status, stream)
    df2.draft_head(bf(R * B, D), bf(V, D), K, bf(r, D), bf(V, r), bf(V, r), i32(R), B, workspace=ws)
    assert fake.calls[-1][1][22] == 256


def test_caller_outputs_of_the_right_size_are_used(fake):
    ids, vals, G = i32(P, K), f32(P, K), f32(P, r)
    got = df2.unary_topk(*head_args(), out=(ids, vals, G))
    assert got[0] is ids and got[1] is vals and got[2] is G
    # the element count is what the kernels write; the shape may be flat
    df2.unary_topk(*head_args(), out=(i32(P * K), f32(P * K), f32(P * r)))


# ------------------------------------------------------------ failed checks --

@pytest.mark.parametrize("bad, err", [
    ((i32(P, K + 1), f32(P, K), f32(P, r)), ValueError),   # ids too long
    ((i32(P, K), f32(P, K - 1), f32(P, r)), ValueError),   # vals too short
    ((i32(P, K), f32(P, K), None), TypeError),             # G missing though W_H is given
    ((f32(P, K), f32(P, K), f32(P, r)), TypeError),        # ids of the wrong type
    ((i32(P, K), f32(K, P).t(), f32(P, r)), ValueError),   # vals not contiguous
])
def test_bad_head_outputs_raise_before_the_call(fake, bad, err):
    with pytest.raises(err):
        df2.unary_topk(*head_args(), out=bad)
    assert not fake.calls


def test_bad_status_and_workspace_raise(fake):
    with pytest.raises(TypeError):
        df2.unary_topk(*head_args(), dev_status=f32(1))
    with pytest.raises(ValueError):
        df2.unary_topk(*head_args(), dev_status=i32(0))
    with pytest.raises(ValueError):
        df2.unary_topk(*head_args(), workspace=torch.zeros(255, dtype=torch.uint8))
    with pytest.raises(ValueError):
        df2.draft_head(bf(R * B, D), bf(V, D), K, bf(r, D), bf(V, r), bf(V, r), i32(R), B,
                       workspace=torch.zeros(8, dtype=torch.uint8))
    assert not fake.calls


def test_bad_selector_and_lattice_outputs_raise(fake):
    with pytest.raises(ValueError):
        df2.selector_walk(*sel_args(), B, out=(i32(R, B), f32(R, B - 1)))
    with pytest.raises(ValueError):
        df2.selector_pair_scores(i32(R * B), *sel_args()[1:], out=f32(R * B, K - 1))
    with pytest.raises(ValueError):
        df2.selector_pair_scores(i32(R * B), *sel_args()[1:5], bf(V, r + 8))   # Bc unlike A
    with pytest.raises(ValueError):
        df2.selector_ce(f32(P, K), i32(P, K), i32(P), V, out=(f32(P - 1), i32(P)))
    with pytest.raises(ValueError):
        df2.selector_lattice(*sel_args(), B, out=f32(R, B - 1, K, K - 1))
    lat = f32(R, B - 1, K, K)
    with pytest.raises(ValueError):
        df2.lattice_walk(lat, i32(R * B, K), B, V, out=(i32(R, B - 1), f32(R, B)))
    with pytest.raises(TypeError):   # pred given, no tensor for its scores
        df2.draft_head(bf(R * B, D), bf(V, D), K, bf(r, D), bf(V, r), bf(V, r), i32(R), B, i32(R * B),
                       out=(i32(R * B, K), f32(R * B, K), f32(R * B, r), i32(R, B - 1), f32(R, B - 1), None))
    assert not fake.calls


def test_bad_conv_shapes_and_outputs_raise(fake):
    C, taps, g = 64, 2, 16
    Wp, base, dyn = bf(2 * taps * C // g, C), f32(2, taps, C), f32(P, taps, C // g)
    with pytest.raises(ValueError):
        df2.conv_prepare(bf(P, C), 8, taps, g, bf(2 * taps * C // g - 1, C), base)   # W_proj short
    with pytest.raises(ValueError):
        df2.conv_prepare(bf(P, C), 8, taps, g, Wp, f32(2, taps + 1, C))             # base of other taps
    with pytest.raises(ValueError):
        df2.conv_prepare(bf(P, C), 8, taps, g, Wp, base, out=(bf(P, C), f32(P, taps, C // g - 1)))
    with pytest.raises(TypeError):
        df2.conv_prepare(bf(P, C), 8, taps, g, Wp, base, out=(f32(P, C), dyn))       # y not like x
    with pytest.raises(ValueError):
        df2.conv_finish(bf(P, C), 8, taps, g, f32(P - 1, taps, C // g), base)         # dyn_out short
    with pytest.raises(ValueError):
        df2.conv_finish(bf(P, C), 8, taps, g, dyn, base, out=bf(P, C - 8))
    with pytest.raises(ValueError):
        df2.conv_finish_prepare(bf(P, C), 8, taps, g, dyn, base, Wp, f32(2, taps, C - 8))
    with pytest.raises(ValueError):
        df2.conv_finish_prepare(bf(P, C), 8, taps, g, dyn, base, Wp, base, residual=bf(P, C - 8))
    assert not fake.calls
    # an invalid group is left to the library, which answers with a status
    df2.conv_prepare(bf(P, C), 8, taps, 3, Wp, base)
    assert fake.calls[-1][0] == "dflash2_conv_prepare"


def test_tensors_on_two_devices_raise(fake):
    """A tensor of another device (the meta device stands in for a second GPU)."""
    h, W, K_, WH = head_args()
    with pytest.raises(ValueError):
        df2.unary_topk(h, torch.empty((V, D), dtype=torch.bfloat16, device="meta"), K_, WH)
    with pytest.raises(ValueError):
        df2.unary_topk(h, W, K_, WH, out=(i32(P, K), f32(P, K), torch.empty((P, r), device="meta")))
    with pytest.raises(ValueError):
        df2.unary_topk(h, W, K_, WH, dev_status=torch.zeros(1, dtype=torch.int32, device="meta"))
    assert not fake.calls


def test_cpu_tensors_are_refused_without_the_stand_in():
    """The real check: a host tensor is never handed to a kernel."""
    with pytest.raises(TypeError):
        df2.unary_topk(*head_args())
    with pytest.raises(TypeError):
        df2.conv_finish(bf(P, 64), 8, 2, 16, f32(P, 2, 4), f32(2, 2, 64))
