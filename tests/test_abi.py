"""Host-side checks of the C-ABI library: it builds, loads, exports every symbol
include/dflash2.h declares, and rejects invalid arguments before any launch
(no GPU needed: these calls return before touching the device)."""
import ctypes as ct
import os
import subprocess

import pytest

from dflash2_draft_block_gb300 import _abi, build

VP = ct.c_void_p


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _abi.load()


def test_exports_every_declared_symbol(lib):
    declared = _abi.header_functions()
    assert len(declared) >= 9
    out = subprocess.run(["nm", "-D", "--defined-only", build.LIB], capture_output=True, text=True,
                         check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    missing = [f for f in declared if f not in exported]
    assert not missing, missing
    assert set(_abi.SIGNATURES) == set(declared)
    # nothing but the C-ABI is exported
    ours = {e for e in exported if e.startswith("dflash2_")}
    assert ours == set(declared)


def test_status_strings(lib):
    names = [lib.dflash2_status_string(i).decode() for i in range(6)]
    assert names == ["DF2_OK", "DF2_ERR_INVALID_ARGUMENT", "DF2_ERR_UNSUPPORTED", "DF2_ERR_CUDA",
                     "DF2_ERR_WORKSPACE_TOO_SMALL", "DF2_ERR_TIMEOUT"]
    assert lib.dflash2_status_string(99).decode() == "DF2_ERR_UNKNOWN"
    assert lib.dflash2_abi_version() == 2


def test_header_compiles_as_c(tmp_path):
    src = tmp_path / "t.c"
    src.write_text('#include "dflash2.h"\nint main(void){return DF2_OK;}\n')
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-I", build.INCLUDE, str(src), "-o",
                    str(tmp_path / "t")], check=True)


def test_head_validation(lib):
    f = lib.dflash2_unary_topk
    fake = VP(0x1000)
    # K > V, K < 1, P < 0, D not multiple of 8, K above the build limit
    assert f(fake, 4, 64, fake, 10, 11, 1.0, 0.0, None, 0, None, fake, fake, fake, 1 << 20, None, None) == 1
    assert f(fake, 4, 64, fake, 10, 0, 1.0, 0.0, None, 0, None, fake, fake, fake, 1 << 20, None, None) == 1
    assert f(fake, -1, 64, fake, 10, 2, 1.0, 0.0, None, 0, None, fake, fake, fake, 1 << 20, None, None) == 1
    assert f(fake, 4, 60, fake, 10, 2, 1.0, 0.0, None, 0, None, fake, fake, fake, 1 << 20, None, None) == 2
    assert f(fake, 4, 64, fake, 5000, 2000, 1.0, 0.0, None, 0, None, fake, fake, fake, 1 << 20, None, None) == 2
    # W_H given with r < 1
    assert f(fake, 4, 64, fake, 10, 2, 1.0, 0.0, fake, 0, fake, fake, fake, fake, 1 << 20, None, None) == 1
    # V above the build limit (DF2_MAX_VOCAB = 2^30), and at the int32 edge
    for V in ((1 << 30) + 1, (1 << 31) - 1):
        assert f(fake, 4, 64, fake, V, 16, 1.0, 0.0, None, 0, None, fake, fake, fake, 1 << 20, None, None) == 2
        assert lib.dflash2_unary_topk_path(8, 4096, V, 16) == -1
    assert lib.dflash2_unary_topk_path(8, 4096, 1 << 30, 16) == 0
    # P == 0 is a no-op
    assert f(fake, 0, 64, fake, 10, 2, 1.0, 0.0, None, 0, None, fake, fake, fake, 0, None, None) == 0
    # output multiplier finite and > 0, final softcap finite and >= 0
    inf, nan = float("inf"), float("nan")
    for m, c in [(0.0, 0.0), (-1.0, 0.0), (nan, 0.0), (inf, 0.0), (1.0, -1.0), (1.0, inf), (1.0, nan)]:
        assert f(fake, 4, 64, fake, 10, 2, m, c, None, 0, None, fake, fake, fake, 1 << 20, None, None) == 1


def test_head_path_query(lib):
    """The head's kernel path is a host decision: few positions stream the LM head,
    many positions run the GEMM with a top-K epilogue, K > 64 the CUDA cores."""
    f = lib.dflash2_unary_topk_path
    assert f(8, 4096, 151936, 16) == 0          # batch-1 shape
    assert f(512, 5120, 248320, 16) == 1        # batched shape
    assert f(4096, 4096, 151936, 64) == 1       # stress shape
    assert f(20, 256, 3000, 100) == 2           # K > 64
    assert f(8, 100, 1000, 16) == -1            # D % 8 != 0
    assert f(8, 256, 10, 16) == -1              # K > V


def test_selector_validation(lib):
    fake = VP(0x1000)
    w = lib.dflash2_selector_walk
    assert w(fake, 2, 1, fake, fake, fake, fake, fake, 100, 4, 32, fake, fake, None, None) == 1  # B < 2
    assert w(fake, 2, 8, fake, fake, fake, fake, fake, 100, 101, 32, fake, fake, None, None) == 1  # K > V
    assert w(fake, 2, 8, fake, fake, fake, fake, fake, 100, 4, 12, fake, fake, None, None) == 2  # r % 8
    assert w(fake, 0, 8, fake, fake, fake, fake, fake, 100, 4, 32, fake, fake, None, None) == 0
    assert w(fake, 2, 8, fake, fake, fake, fake, fake, (1 << 30) + 1, 4, 32, fake, fake, None, None) == 2
    assert lib.dflash2_lattice_walk(fake, fake, 2, 8, 4, (1 << 30) + 1, None, 1.0, fake, fake, None, None) == 2
    assert lib.dflash2_selector_ce(fake, fake, fake, 4, 4, (1 << 30) + 1, fake, fake, None, None) == 2
    dh = lib.dflash2_draft_head
    f8 = [fake] * 8
    # B < 2, K > V, r % 8, W_H missing, workspace too small
    assert dh(fake, 1, 1, 64, fake, 100, 4, 1.0, 0.0, fake, 32, fake, fake, fake, None, *f8[:5], None, fake, 1 << 20, None, None) == 1
    assert dh(fake, 1, 8, 64, fake, 100, 101, 1.0, 0.0, fake, 32, fake, fake, fake, None, *f8[:5], None, fake, 1 << 20, None, None) == 1
    assert dh(fake, 1, 8, 64, fake, 100, 4, 1.0, 0.0, fake, 12, fake, fake, fake, None, *f8[:5], None, fake, 1 << 20, None, None) == 2
    assert dh(fake, 1, 8, 64, fake, 100, 4, 1.0, 0.0, None, 32, fake, fake, fake, None, *f8[:5], None, fake, 1 << 20, None, None) == 1
    assert dh(fake, 0, 8, 64, fake, 100, 4, 1.0, 0.0, fake, 32, fake, fake, fake, None, *f8[:5], None, fake, 0, None, None) == 0
    # a bad output multiplier or softcap
    assert dh(fake, 1, 8, 64, fake, 100, 4, -2.0, 0.0, fake, 32, fake, fake, fake, None, *f8[:5], None, fake, 1 << 20, None, None) == 1
    assert dh(fake, 1, 8, 64, fake, 100, 4, 1.0, -0.5, fake, 32, fake, fake, fake, None, *f8[:5], None, fake, 1 << 20, None, None) == 1
    assert lib.dflash2_draft_head_workspace_size(1, 1, 64, 100, 4, 32) == 0
    lt = lib.dflash2_selector_lattice
    assert lt(fake, 2, 1, fake, fake, fake, fake, fake, 100, 4, 32, fake, None, None) == 1  # B < 2
    assert lt(fake, 2, 8, fake, fake, fake, fake, fake, 100, 101, 32, fake, None, None) == 1  # K > V
    assert lt(fake, 2, 8, fake, fake, fake, fake, fake, 100, 4, 12, fake, None, None) == 2  # r % 8
    assert lt(fake, 2, 8, fake, fake, fake, fake, fake, 5000, 2000, 32, fake, None, None) == 2  # K cap
    assert lt(fake, 0, 8, fake, fake, fake, fake, fake, 100, 4, 32, fake, None, None) == 0
    # more CTAs than one launch can address
    assert lt(fake, 1 << 24, 8, fake, fake, fake, fake, fake, 5000, 1024, 32, fake, None, None) == 2
    lw = lib.dflash2_lattice_walk
    assert lw(fake, fake, 2, 1, 4, 100, None, 1.0, fake, fake, None, None) == 1  # B < 2
    assert lw(fake, fake, 2, 8, 0, 100, None, 1.0, fake, fake, None, None) == 1  # K < 1
    assert lw(fake, fake, 2, 8, 4, 100, fake, 0.0, fake, fake, None, None) == 1  # temperature 0
    assert lw(fake, fake, 2, 8, 4, 100, fake, -1.0, fake, fake, None, None) == 1
    assert lw(fake, fake, 2, 8, 4, 100, fake, float("inf"), fake, fake, None, None) == 1
    assert lw(fake, fake, 2, 8, 4, 100, fake, float("nan"), fake, fake, None, None) == 1
    assert lw(fake, fake, 0, 8, 4, 100, fake, 0.5, fake, fake, None, None) == 0
    ps = lib.dflash2_selector_pair_scores
    assert ps(fake, -1, fake, fake, fake, fake, fake, 100, 4, 32, fake, None, None) == 1
    assert ps(fake, 4, fake, fake, fake, fake, fake, 100, 0, 32, fake, None, None) == 1
    assert ps(fake, 0, fake, fake, fake, fake, fake, 100, 4, 32, fake, None, None) == 0


def test_conv_validation(lib):
    fake, fake2 = VP(0x1000), VP(0x2000)
    p = lib.dflash2_conv_prepare
    # P % B != 0 (raises in the training path of the pages), taps > B, C % g, dtype
    assert p(fake, 0, 12, 64, 8, 2, 16, fake, fake, fake2, fake, fake, 1 << 20, None) == 1
    assert p(fake, 0, 16, 64, 8, 9, 16, fake, fake, fake2, fake, fake, 1 << 20, None) == 1
    assert p(fake, 0, 16, 64, 8, 2, 24, fake, fake, fake2, fake, fake, 1 << 20, None) == 1
    assert p(fake, 7, 16, 64, 8, 2, 16, fake, fake, fake2, fake, fake, 1 << 20, None) == 1
    assert p(fake, 0, 16, 64, 8, 0, 16, fake, fake, fake2, fake, fake, 1 << 20, None) == 1
    # y aliasing x
    assert p(fake, 0, 16, 64, 8, 2, 16, fake, fake, fake, fake, fake, 1 << 20, None) == 1
    # workspace too small
    assert p(fake, 0, 16, 64, 8, 2, 16, fake, fake, fake2, fake, fake, 16, None) == 4
    fin = lib.dflash2_conv_finish
    assert fin(fake, 0, 12, 64, 8, 2, 16, fake, fake, fake2, None) == 1
    assert fin(fake, 0, 0, 64, 8, 2, 16, fake, fake, fake2, None) == 0
    assert lib.dflash2_conv_prepare_workspace_size(16, 64, 2, 16, 0) == 512
    fp = lib.dflash2_conv_finish_prepare
    f3, f4, f5, f6 = VP(0x3000), VP(0x4000), VP(0x5000), VP(0x6000)
    ok = dict(z=fake, dyn=fake2, base=f3, res=None, h=f4, W=f5, bn=f3, y=f6, dn=VP(0x7000))
    call = lambda d, P=16, B=8, ws=1 << 20: fp(d["z"], 0, P, 64, B, 2, 16, d["dyn"], d["base"], d["res"], d["h"],
                                             d["W"], d["bn"], d["y"], d["dn"], fake, ws, None)
    assert call(ok, P=12) == 1                                   # P % B != 0
    assert call({**ok, "h": fake}) == 1                          # h aliases z
    assert call({**ok, "res": f4}) == 1                          # h aliases the residual
    assert call({**ok, "y": f4}) == 1                            # y_next aliases h
    assert call({**ok, "y": fake}) == 1                          # y_next aliases z
    assert call({**ok, "dn": fake2}) == 1                        # dyn_out_next aliases dyn_out
    assert call(ok, ws=16) == 4                                  # workspace too small
    assert call(ok, P=0) == 0
    assert lib.dflash2_conv_finish_prepare_workspace_size(16, 64, 2, 16, 0) == 512


def test_product_path_does_not_reach_the_oracle():
    """The package never imports or loads the oracle (test infrastructure only)."""
    pkg = os.path.dirname(build.__file__)
    for root, _, files in os.walk(pkg):
        for fn in files:
            if fn.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(root, fn)).read()
                for bad in ("import oracle", "from oracle", "df2o_", "dflash2_oracle"):
                    assert bad not in text, (fn, bad)
