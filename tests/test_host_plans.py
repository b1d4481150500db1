"""The kernels' tile schedules, compiled on the CPU from their own source text and
swept over many shapes.

The schedules are host arithmetic plus a few device lambdas that turn a tile index
into rows and groups; a GPU test only sees the shapes it runs.  Here the very text
of those functions (taken out of the .cu files by brace matching, so an edit to the
kernels is what gets tested) is compiled with g++ and checked for every shape of a
wide sweep:

- the batch-1 head's vocabulary tiling (`v_tiling` and the kernel's `tile_row0` /
  `tile_rows`): the tiles cover rows 0 .. V-1 once each, in order, none of them
  empty, none taller than the MMA's 128 rows, the W_H tiles after them, and every
  CTA streams the same number of tiles whenever the tiling is not the plain one;
- the many-row conv prepare's schedule (`ctc_split_last_round` and the kernel's
  `tile(k)`), for single CTAs, CTA pairs and clusters of two pairs, with and without
  the last round in half tiles: every (128-row tile, channel group) pair of the
  problem is computed by exactly one CTA, and nothing past the padded last pair
  tile or the last group is touched.
"""
import ctypes
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "dflash2_draft_block_gb300", "csrc")


def _read(name):
    with open(os.path.join(CSRC, name)) as f:
        return f.read()


def _block(text, start):
    """`start` (which must occur once) through its balanced closing brace, and a
    ';' right after it if there is one."""
    assert text.count(start) == 1, start
    i = text.index(start)
    depth = 0
    for k in range(text.index("{", i), len(text)):
        if text[k] == "{":
            depth += 1
        elif text[k] == "}":
            depth -= 1
            if depth == 0:
                end = k + 1
                if text[end:end + 1] == ";":
                    end += 1
                return text[i:end]
    raise AssertionError("unbalanced braces after " + start)


def _line(text, start):
    assert text.count(start) == 1, start
    i = text.index(start)
    return text[i:text.index("\n", i)]


def _harness():
    head = _read("head_tc.cu")
    conv = _read("conv_tc.cu")
    kernel = conv[conv.index("conv_prepare_tc_kernel("):]
    frag_start = kernel.index("    const int n_rows_units")
    frag = kernel[frag_start:kernel.index(_block(kernel, "auto tile = [&](int k) {"))] + \
        _block(kernel, "auto tile = [&](int k) {")
    return f"""
#include <cstdint>
#include <vector>

namespace head {{
{_line(head, "constexpr int BM = ")}
{_block(head, "struct VTiling {")}
{_block(head, "VTiling v_tiling(int64_t V, int n_wh, int grid) {")}
}}  // namespace head

// 0, or the first V of [V0, V1) (step) whose tiling breaks a rule
extern "C" int64_t head_sweep(int64_t V0, int64_t V1, int64_t step, int sms, int n_wh) {{
    using namespace head;
    for (int64_t V = V0; V < V1; V += step) {{
        const int n_v128 = int((V + BM - 1) / BM);
        const int grid = n_v128 < sms ? n_v128 : sms;
        const VTiling vt = v_tiling(V, n_wh, grid);
        const int n_vtiles = vt.n_vtiles, n_hi = vt.n_hi, bm_hi = vt.bm_hi, bm_lo = vt.bm_lo;
        {_block(head, "auto tile_row0 = [&](int t) {")}
        {_block(head, "auto tile_rows = [&](int t) {")}
        int64_t next = 0;
        for (int t = 0; t < n_vtiles; ++t) {{
            const int64_t r0 = tile_row0(t), nr = tile_rows(t);
            if (r0 != next || r0 >= V || nr < 8 || nr > BM || nr % 8 != 0) return V;
            next = r0 + nr;
        }}
        if (next < V || next - V >= BM) return V;
        for (int t = n_vtiles; t < n_vtiles + n_wh; ++t)
            if (tile_row0(t) != int64_t(t - n_vtiles) * BM || tile_rows(t) != BM) return V;
        const bool plain = n_vtiles == n_v128 && n_hi == n_vtiles && bm_hi == BM && bm_lo == BM;
        if (!plain && (n_vtiles + n_wh) % grid != 0) return V;
    }}
    return 0;
}}

namespace conv {{
{_block(conv, "struct CtcPlan {")}
{_block(conv, "void ctc_split_last_round(CtcPlan& p, int64_t total) {")}

struct Args {{
    int n_units, n_full_rounds, n_half, n_gt, n_mu;
}};

// Every CTA of the launch walks its tiles; cnt counts each (128-row tile, half of a
// group tile).  Returns 0 when every cell of the problem is covered once and nothing
// lies outside the padded tiles and groups, else a code naming the broken rule.
template <bool PAIR, bool MC>
int cover(int n_mt, int n_gt, int ng, int slots, int* n_half_out) {{
    const int n_mu = PAIR ? (n_mt + 1) / 2 : n_mt;
    if (MC && n_mu % 2 != 0) return 0;
    const int64_t total = int64_t(MC ? n_mu / 2 : n_mu) * n_gt;
    CtcPlan p;
    p.ok = true;
    p.pair = PAIR;
    p.mc = MC;
    p.ng = ng;
    p.n_gt = n_gt;
    p.n_mu = n_mu;
    p.units = int(total < slots ? total : slots);
    ctc_split_last_round(p, total);
    *n_half_out = p.n_half;
    const Args a{{p.units, p.n_full_rounds, p.n_half, n_gt, n_mu}};
    const int n_mt_pad = PAIR ? 2 * n_mu : n_mu;
    std::vector<int> cnt(size_t(n_mt_pad) * 2 * n_gt, 0);
    for (int unit = 0; unit < a.n_units; ++unit)
        for (int pp = 0; pp < (MC ? 2 : 1); ++pp)
            for (int rank = 0; rank < (PAIR ? 2 : 1); ++rank) {{
{frag}
                for (int k = 0; k < ntiles; ++k) {{
                    const Tile tl = tile(k);
                    if (tl.mt < 0 || tl.mt >= n_mt_pad) return 1;
                    if (tl.ngt != ng && tl.ngt != ng / 2) return 2;
                    if (tl.g0 % (ng / 2) != 0 || tl.g0 < 0 || tl.g0 + tl.ngt > n_gt * ng) return 3;
                    for (int c = tl.g0 / (ng / 2); c < (tl.g0 + tl.ngt) / (ng / 2); ++c)
                        ++cnt[size_t(tl.mt) * 2 * n_gt + c];
                }}
            }}
    for (int mt = 0; mt < n_mt_pad; ++mt)
        for (int c = 0; c < 2 * n_gt; ++c) {{
            const int v = cnt[size_t(mt) * 2 * n_gt + c];
            if (v > 1) return 4;                 // computed twice
            if (v == 0 && mt < n_mt) return 5;   // never computed
        }}
    return 0;
}}
}}  // namespace conv

// kind: 0 single CTAs, 1 CTA pairs, 2 clusters of two pairs
extern "C" int conv_cover(int kind, int n_mt, int n_gt, int ng, int slots, int* n_half) {{
    if (kind == 0) return conv::cover<false, false>(n_mt, n_gt, ng, slots, n_half);
    if (kind == 1) return conv::cover<true, false>(n_mt, n_gt, ng, slots, n_half);
    return conv::cover<true, true>(n_mt, n_gt, ng, slots, n_half);
}}
"""


@pytest.fixture(scope="module")
def plans(tmp_path_factory):
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        pytest.skip("no C++ compiler")
    d = tmp_path_factory.mktemp("plans")
    src = d / "plans.cpp"
    src.write_text(_harness())
    lib = d / "libplans.so"
    subprocess.run([cxx, "-std=c++17", "-O2", "-shared", "-fPIC", "-o", str(lib), str(src)], check=True)
    so = ctypes.CDLL(str(lib))
    so.head_sweep.restype = ctypes.c_int64
    so.head_sweep.argtypes = [ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int, ctypes.c_int]
    so.conv_cover.restype = ctypes.c_int
    so.conv_cover.argtypes = [ctypes.c_int] * 5 + [ctypes.POINTER(ctypes.c_int)]
    return so


@pytest.mark.parametrize("n_wh", [0, 1, 2, 32])   # no W_H; r = 128, 256, 4096
@pytest.mark.parametrize("sms", [152, 148, 132])
def test_head_vocabulary_tiling(plans, sms, n_wh):
    assert plans.head_sweep(1, 40000, 1, sms, n_wh) == 0
    assert plans.head_sweep(40000, 2_000_000, 97, sms, n_wh) == 0
    for V in (151936, 248320, 152064, 256000, 1 << 20, (1 << 30) - 1, 1 << 30):
        assert plans.head_sweep(V, V + 1, 1, sms, n_wh) == 0, V


def test_conv_prepare_schedule(plans):
    n_half = ctypes.c_int(0)
    split = 0
    for kind, slots_list in ((0, (148, 152, 37)), (1, (74, 76, 19)), (2, (36, 38, 9))):
        for slots in slots_list:
            for ng in (8, 16, 32, 40, 64):
                for n_gt in list(range(1, 13)) + [20, 40]:
                    for n_mt in list(range(1, 41)) + [63, 64, 65, 127, 128, 129, 255, 256]:
                        rc = plans.conv_cover(kind, n_mt, n_gt, ng, slots, ctypes.byref(n_half))
                        assert rc == 0, (kind, n_mt, n_gt, ng, slots, rc)
                        split += n_half.value > 0
    assert split > 100   # the half-tile last round was among the schedules checked


def test_conv_prepare_schedule_at_the_workloads(plans):
    """The training-packed conv (P 16384: 128 tiles of 128 rows, G 320) and its
    neighbours in the half-tile tests, under the plans the launch picks there."""
    n_half = ctypes.c_int(0)
    for n_mt in (40, 42, 112, 128, 144):
        for ng, kind, slots in ((40, 1, 76), (32, 2, 36), (40, 2, 36), (64, 0, 152)):
            if 320 % ng == 0:
                assert plans.conv_cover(kind, n_mt, 320 // ng, ng, slots, ctypes.byref(n_half)) == 0
