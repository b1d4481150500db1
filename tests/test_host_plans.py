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
- the batch-1 head's plan and shared-memory layout (`pick_plan`, `smem_layout`) for
  every supported (positions, K): it fits the 227 KB a CTA may have, the stages
  start on 1024-byte swizzle boundaries, and the end-of-kernel list exchange, which
  reuses the start of the W stage ring, stays inside that ring (clear of the h
  stages and the barriers other warps may still be waiting on);
- the many-row conv prepare's schedule (`ctc_split_last_round` and the kernel's
  `tile(k)`), for single CTAs, CTA pairs and clusters of two pairs, with and without
  the last round in half tiles: every (128-row tile, channel group) pair of the
  problem is computed by exactly one CTA, and nothing past the padded last pair
  tile or the last group is touched;
- the many-position GEMM's plan (`wide_plan`) and the kernel's tile walk, for the
  top-K epilogue (CTAs, pairs, clusters of two pairs, with G riding on the short
  last vocabulary range) and the store epilogue (the linear round-robin walk):
  every (M tile, N tile) is computed once, every row gets exactly the partial lists
  the workspace holds, the G tile once per M tile, and the two pairs of a cluster
  share their vocabulary range.  The occupancy queries the plan makes on a GPU
  (pipeline stages, clusters that fit) are parameters of the sweep;
- the conv apply ring (`bulk_plan` and the producer warp's copy loop): every 1-D
  bulk copy starts and ends on a 16-byte boundary on both sides (the instruction
  faults otherwise), stays inside its tensor and inside its ring buffer, the copies
  of one item tile the buffer's bytes without overlap, and they add up to the byte
  count the buffer's barrier is told to expect (a mismatch would stall it).
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
    gemm = _read("gemm_tc.cu")
    wk = gemm[gemm.index("gemm_wide_kernel(const __grid_constant__"):]
    w_start = wk.index("    const int n_groups = (args.n_nt + args.tiles_per_cta - 1) / args.tiles_per_cta;")
    w_last = _block(wk, "auto tile_mt = [&](int k) {")
    frag_w = wk[w_start:wk.index(w_last)] + w_last
    capp = _read("conv.cu")
    ck = capp[capp.index("conv_apply_bulk_kernel(const T* __restrict__ x"):]
    ck = ck[:ck.index("// Few rows: one thread per (row")]
    c_start = ck.index("            const int64_t item = blockIdx.x + k * stride;")
    c_loop = _block(ck[c_start:], "for (int e = lane; e < B * per_row; e += 32) {")
    frag_c = ck[c_start:ck.index(c_loop, c_start)] + c_loop
    ln_ngrp = _line(ck, "    const int ngrp = nt * N / g;")
    ln_row = _line(ck, "    const uint32_t row = uint32_t(nt) * 16;")
    ln_xbytes = _line(ck, "    const uint32_t xbytes = uint32_t(B) * row;")
    ln_rbytes = _line(ck, "    const uint32_t rbytes = RES ? xbytes : 0u;")
    ln_per_row = _line(ck, "        const int per_row = (RES ? 2 : 1) + TAPS;")
    ln_n_mine = _line(ck, "    const int64_t n_mine = blockIdx.x < n_items ?")
    return f"""
#include <algorithm>
#include <utility>
#include <cstdint>
#include <vector>

namespace head {{
{_line(head, "constexpr int BM = ")}
{_block(head, "struct VTiling {")}
{_block(head, "VTiling v_tiling(int64_t V, int n_wh, int grid) {")}
}}  // namespace head

namespace headplan {{
{_line(head, "constexpr int BM = ")}
{_line(head, "constexpr int BK = ")}
{_line(head, "constexpr int kEpiWarps = ")}
{_line(head, "constexpr uint32_t kWBytes = ")}
{_line(head, "constexpr int kMaxStages = ")}
{_line(head, "constexpr int kMaxK = ")}
{_line(head, "#define DF2_HEAD_KBOX ")}
#define __host__
#define __device__
{_block(head, "struct SmemLayout {")}
{_block(head, "__host__ __device__ inline SmemLayout smem_layout(int N, int R, int nstages, int kbox) {")}
#undef __host__
#undef __device__
{_line(head, "int pick_n(int64_t P) {")}
{_block(head, "struct Plan {")}
{_block(head, "Plan pick_plan(int64_t P, int K) {")}
}}  // namespace headplan

// 0 when every supported (P, K) gets a plan that fits and keeps its regions apart;
// else 1000 * P + K of the first that does not
extern "C" int head_plans() {{
    using namespace headplan;
    for (int P = 1; P <= 32; ++P)
        for (int K = 1; K <= kMaxK; ++K) {{
            if (!(P <= 16 || K <= 32)) continue;   // not taken by this kernel
            const Plan pl = pick_plan(P, K);
            if (pl.nstages < 2) return 1000 * P + K;
            const SmemLayout L = smem_layout(pl.N, pl.R, pl.nstages, pl.kbox);
            const uint32_t xch = uint32_t(kEpiWarps * pl.N * pl.R * 32) * 8;
            if (L.total + 1024 > 227u * 1024u) return 1000 * P + K;
            if (L.stage_w % 1024 || L.h_off % 1024 || L.stage_h % 1024 || L.bar_off % 8) return 1000 * P + K;
            if (xch > L.h_off) return 1000 * P + K;   // the exchange would reach the h stages or barriers
            if (pl.N < P || (K > 32 && pl.R < 2)) return 1000 * P + K;
        }}
    return 0;
}}

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

namespace wide {{
using std::min;
{_line(gemm, "constexpr int WM = ")}
{_line(gemm, "enum { EPI_STORE = 0, EPI_TOPK = 1 };")}
{_block(gemm, "struct WideArgs {")}
// the plan's two occupancy queries, as sweep parameters
int g_stages = 3, g_mc_slots = 0;
int wide_stages(int, int, bool) {{ return g_stages; }}
int mc_cluster_slots(int, int) {{ return g_mc_slots; }}
{_block(gemm, "int wide_bn(int epi, int K) {")}
{_block(gemm, "int wide_groups(int n_mt, int n_nt, int num_sms) {")}
{_block(gemm, "struct WidePlan {")}
{_block(gemm, "WidePlan wide_plan(int epi, int64_t M, int64_t N, int K, int num_sms, bool persistent) {")}
namespace tc {{
uint32_t g_crank = 0;
inline uint32_t cluster_ctarank() {{ return g_crank; }}
}}

template <int EPI, bool PAIR, bool GT, bool MC>
int cover(const WidePlan& p, const WideArgs& args) {{
    const int grid = (p.pair ? 2 : 1) * p.units;
    const int pad_mt = PAIR ? 2 * ((args.n_mt + 1) / 2) : args.n_mt;
    std::vector<int> cnt(size_t(pad_mt) * args.n_nt, 0), gcnt(pad_mt, 0), lists(size_t(pad_mt) * p.n_groups, 0);
    std::vector<int> grp_of(grid, -1), mu_of(grid, -1);
    for (int bid = 0; bid < grid; ++bid) {{
        tc::g_crank = MC ? bid % 4 : (PAIR ? bid % 2 : 0);
{frag_w}
        grp_of[bid] = grp;
        mu_of[bid] = mu;
        for (int k = 0; k < ntiles; ++k) {{
            const int nt = tile_nt(k), mtk = tile_mt(k);
            if (mtk < 0 || mtk >= pad_mt) return 1;
            if (tile_is_g(k)) {{
                if (nt != 0) return 2;
                ++gcnt[mtk];
            }} else {{
                if (nt < 0 || nt >= args.n_nt) return 3;
                ++cnt[size_t(mtk) * args.n_nt + nt];
            }}
        }}
        if (EPI == EPI_TOPK) {{
            if (grp < 0 || grp >= p.n_groups) return 4;   // a list slot the workspace lacks
            ++lists[size_t(mt) * p.n_groups + grp];
        }}
    }}
    for (int m = 0; m < pad_mt; ++m) {{
        for (int n = 0; n < args.n_nt; ++n) {{
            const int v = cnt[size_t(m) * args.n_nt + n];
            if (v > 1 || (v == 0 && m < args.n_mt)) return 5;
        }}
        if (m < args.n_mt && gcnt[m] != (GT ? 1 : 0)) return 6;
        if (EPI == EPI_TOPK && m < args.n_mt)
            for (int g = 0; g < p.n_groups; ++g)
                if (lists[size_t(m) * p.n_groups + g] != 1) return 7;
    }}
    if (MC)
        for (int bid = 0; bid < grid; bid += 4)
            if (grp_of[bid] != grp_of[bid + 2] || mu_of[bid + 2] != mu_of[bid] + 1) return 8;
    return 0;
}}
}}  // namespace wide

// 0 when the plan of this shape covers it (see cover), else the broken rule's code;
// plan_out: pair, mc, units, n_groups, G folded
extern "C" int wide_cover(int epi, int64_t M, int64_t N, int K, int sms, int stages, int mc_slots, int64_t r,
                          int* plan_out) {{
    using namespace wide;
    g_stages = stages;
    g_mc_slots = mc_slots;
    const WidePlan p = wide_plan(epi, M, N, K, sms, epi == EPI_TOPK);
    WideArgs a{{}};
    a.M = int(M);
    a.N = int(N);
    a.n_mt = p.n_mt;
    a.n_nt = p.n_nt;
    a.tiles_per_cta = p.tiles_per_cta;
    a.K = K;
    bool fold = false;
    if (epi == EPI_STORE) {{
        a.m_major = 1;
        a.linear = p.linear ? 1 : 0;
        a.n_units = p.units;
    }} else {{
        const bool want_g = r > 0;
        float* G = nullptr;
        const int n_groups = p.n_groups;
        {_line(gemm, "    const int last_rng = p.n_nt - (p.n_groups - 1) * p.tiles_per_cta;").strip()}
        {_line(gemm, "    const bool fold_g = want_g && r <= 256 && last_rng < p.tiles_per_cta;").strip()}
        {_block(gemm, "if (fold_g) {")}
        fold = fold_g;
        (void)n_groups;
    }}
    plan_out[0] = p.pair;
    plan_out[1] = p.mc;
    plan_out[2] = p.units;
    plan_out[3] = p.n_groups;
    plan_out[4] = fold;
    if (epi == EPI_STORE)
        return p.pair ? cover<EPI_STORE, true, false, false>(p, a) : cover<EPI_STORE, false, false, false>(p, a);
    if (a.n_gt > 0) {{
        if (p.mc) return cover<EPI_TOPK, true, true, true>(p, a);
        return p.pair ? cover<EPI_TOPK, true, true, false>(p, a) : cover<EPI_TOPK, false, true, false>(p, a);
    }}
    if (p.mc) return cover<EPI_TOPK, true, false, true>(p, a);
    return p.pair ? cover<EPI_TOPK, true, false, false>(p, a) : cover<EPI_TOPK, false, false, false>(p, a);
}}

namespace capply {{
template <typename T>
struct Vec {{
    static constexpr int N = 16 / int(sizeof(T));
}};
{_line(capp, "constexpr int kBulkMaxStages = ")}
{_block(capp, "struct BulkPlan {")}
{_block(capp, "template <typename T>" + chr(10) + "BulkPlan bulk_plan(")}

struct Copy {{
    uint64_t dst, src, bytes;
}};
std::vector<Copy> g_copies;
uint64_t g_expect = 0;
namespace tc {{
inline void mbar_arrive_expect_tx(uint64_t*, uint32_t bytes) {{ g_expect += bytes; }}
inline void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t*, uint64_t) {{
    g_copies.push_back(Copy{{uint64_t(reinterpret_cast<uintptr_t>(dst)), uint64_t(reinterpret_cast<uintptr_t>(src)), bytes}});
}}
}}  // namespace tc
inline void __syncwarp() {{}}

// The launch's copies, CTA by CTA and item by item, for one shape; the tensors sit
// at 16-byte-aligned addresses that are never dereferenced.  0, -1 (no ring plan:
// the launch takes another kernel), or the code of the broken rule.
template <typename T, int TAPS, bool RES>
int check(int64_t nblocks, int C, int B, int g, int dyn_mult, int grid) {{
    const int G = C / g;
    const int64_t dyn_ld = int64_t(dyn_mult) * TAPS * G;
    const int64_t P = nblocks * B;
    const BulkPlan bp = bulk_plan<T>(C, B, TAPS, g, G, dyn_ld, RES);
    if (bp.nt == 0) return -1;
    if (bp.smem > 227u * 1024u || bp.stages < 2 || bp.stages > kBulkMaxStages) return 10;
    if (bp.buf % 128 != 0 || bp.smem < uint32_t(bp.stages) * bp.buf + 2 * kBulkMaxStages * 8 + 4) return 11;
    constexpr int N = Vec<T>::N;
    const int nt = bp.nt, strips = bp.strips, stages = bp.stages;
    const uint32_t buf_bytes = bp.buf;
{ln_ngrp}
{ln_row}
{ln_xbytes}
{ln_rbytes}
{ln_per_row}
    if (int64_t(strips) * nt * N != C) return 12;
    const T* x = reinterpret_cast<const T*>(uintptr_t(1) << 40);
    const T* res = reinterpret_cast<const T*>(uintptr_t(2) << 40);
    const float* dyn = reinterpret_cast<const float*>(uintptr_t(3) << 40);
    uint8_t* smem = reinterpret_cast<uint8_t*>(uintptr_t(4) << 40);
    uint64_t full[kBulkMaxStages] = {{}};
    const uint64_t pol = 0;
    const int64_t n_items = nblocks * strips;
    const int64_t stride = grid;
    for (int64_t bx = 0; bx < grid; ++bx) {{
        const struct {{
            int64_t x;
        }} blockIdx = {{bx}};
{ln_n_mine}
        for (int64_t k = 0; k < n_mine; ++k) {{
            const int s = int(k % stages);
            g_copies.clear();
            g_expect = 0;
            for (int lane = 0; lane < 32; ++lane) {{
{frag_c}
            }}
            // every copy: 16-byte aligned at both ends, inside its tensor or buffer
            uint64_t sum = 0;
            const uint64_t b0 = (uintptr_t(4) << 40) + uint64_t(s) * buf_bytes;
            std::vector<std::pair<uint64_t, uint64_t>> spans;
            for (const Copy& c : g_copies) {{
                if (c.bytes == 0 || c.bytes % 16 || c.src % 16 || c.dst % 16) return 1;
                const uint64_t base = c.src >> 40 << 40;
                const uint64_t size = base == (uintptr_t(3) << 40) ? uint64_t(P) * dyn_ld * 4 : uint64_t(P) * C * sizeof(T);
                if (c.src + c.bytes > base + size) return 2;
                if (base == (uintptr_t(2) << 40) && !RES) return 3;
                if (c.dst < b0 || c.dst + c.bytes > b0 + buf_bytes) return 4;
                spans.push_back({{c.dst - b0, c.dst - b0 + c.bytes}});
                sum += c.bytes;
            }}
            if (sum != g_expect) return 5;
            std::sort(spans.begin(), spans.end());
            uint64_t at = 0;
            for (const auto& sp : spans) {{
                if (sp.first != at) return 6;   // a gap or an overlap
                at = sp.second;
            }}
            if (at != xbytes + rbytes + uint64_t(B) * TAPS * ngrp * 4) return 7;
        }}
    }}
    return 0;
}}
}}  // namespace capply

extern "C" int conv_apply_copies(int f32, int taps, int res, int64_t nblocks, int C, int B, int g, int dyn_mult,
                                 int grid) {{
    using namespace capply;
#define DF2T_CASE(TP)                                                                           \
    if (taps == TP) {{                                                                            \
        if (f32) return res ? check<float, TP, true>(nblocks, C, B, g, dyn_mult, grid)            \
                            : check<float, TP, false>(nblocks, C, B, g, dyn_mult, grid);          \
        return res ? check<uint16_t, TP, true>(nblocks, C, B, g, dyn_mult, grid)                  \
                   : check<uint16_t, TP, false>(nblocks, C, B, g, dyn_mult, grid);                \
    }}
    DF2T_CASE(1) DF2T_CASE(2) DF2T_CASE(3) DF2T_CASE(4)
#undef DF2T_CASE
    return 99;
}}

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
    so.head_plans.restype = ctypes.c_int
    so.head_sweep.restype = ctypes.c_int64
    so.head_sweep.argtypes = [ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int, ctypes.c_int]
    so.wide_cover.restype = ctypes.c_int
    so.wide_cover.argtypes = [ctypes.c_int, ctypes.c_int64, ctypes.c_int64] + [ctypes.c_int] * 4 + [
        ctypes.c_int64, ctypes.POINTER(ctypes.c_int)]
    so.conv_apply_copies.restype = ctypes.c_int
    so.conv_apply_copies.argtypes = [ctypes.c_int] * 3 + [ctypes.c_int64] + [ctypes.c_int] * 5
    so.conv_cover.restype = ctypes.c_int
    so.conv_cover.argtypes = [ctypes.c_int] * 5 + [ctypes.POINTER(ctypes.c_int)]
    return so


def test_head_plan_and_shared_memory(plans):
    assert plans.head_plans() == 0


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


_M = list(range(1, 65)) + [100, 127, 128, 129, 255, 256, 257, 384, 511, 512, 513, 1000, 1024, 2048, 4096, 4097]


@pytest.mark.parametrize("N", [151936, 248320, 40000, 9000, 3000, 257, 256, 100])
def test_wide_gemm_topk_schedule(plans, N):
    out = (ctypes.c_int * 5)()
    seen = set()
    for M in _M:
        for K in (16, 64):
            for sms in (152, 148):
                for stages, mc in ((3, 0), (2, 0), (3, 18), (3, 36), (4, 19)):
                    for r in (0, 64, 256, 512):
                        rc = plans.wide_cover(1, M, N, K, sms, stages, mc, r, out)
                        assert rc == 0, (M, N, K, sms, stages, mc, r, rc, list(out))
                        seen.add((out[0], out[1], out[4]))
    if N >= 40000:
        # CTAs and pairs, clusters of two pairs, with and without G on the last range
        assert {(0, 0), (1, 0), (1, 1)} <= {(p, m) for p, m, _ in seen}, seen
        assert {0, 1} <= {f for _, _, f in seen}, seen


@pytest.mark.parametrize("N", [256, 512, 1280, 2560, 10240, 100, 300])
def test_wide_gemm_store_schedule(plans, N):
    out = (ctypes.c_int * 5)()
    for M in _M + [16384]:
        for sms in (152, 148):
            assert plans.wide_cover(0, M, N, 0, sms, 3, 0, 0, out) == 0, (M, N, sms)


@pytest.mark.parametrize("f32", [0, 1])
@pytest.mark.parametrize("taps", [1, 2, 3, 4])
def test_conv_apply_bulk_copies(plans, f32, taps):
    planned = 0
    for res in (0, 1):
        for C in (512, 640, 2048, 4096, 5120, 8192):
            for B in (1, 2, 4, 8, 16, 32):
                if taps > B:
                    continue
                for g in (8, 16, 64):
                    for dyn_mult in (1, 2):
                        for nblocks, grid in ((5, 3), (2, 152)):
                            rc = plans.conv_apply_copies(f32, taps, res, nblocks, C, B, g, dyn_mult, grid)
                            assert rc in (0, -1), (f32, taps, res, C, B, g, dyn_mult, nblocks, grid, rc)
                            planned += rc == 0
    assert planned > 50   # shapes the ring takes, not only the fallbacks
