// Conv prepare for many rows, fused on the tensor cores: the projection of x, the
// output-side correction written out and the conv applied in the same kernel.
//
//   d[p, (io*taps + j)*G + gi] = sum_c x[p, c] * W_proj[(io*taps + j)*G + gi, c]
//   y[p, c] = sum_{j < taps, t-j >= 0} (base[0, j, c] + d[p, (0*taps + j)*G + c/g]) * x[p-j, c]
//   dyn_out[p, j, gi] = d[p, (1*taps + j)*G + gi]
//
// (verl-SpeCo PR #62, "What DFlash2 adds": one projection of the hidden state gives
// the corrections of the conv before the sublayer and of the one after it; prepare
// applies the first and emits the second.  "Two deltas", item 1: the taps stay
// inside an anchor block.)
//
// A tile is 128 rows of x (a whole number of anchor blocks) times the projection
// rows of `ng` consecutive groups: the input-side rows of every tap, then the
// output-side ones (2*taps*ng columns, at most 256), gathered from 2*taps TMA boxes
// of ng W_proj rows.  In a CTA pair (cta_group::2, 256 rows of x) CTA 0 stages the
// input-side rows and CTA 1 the output-side ones; each CTA's TMEM receives all the
// tile's columns for its own 128 rows.
//
// Epilogue (warps 2-9; thread = TMEM lane = row, the two warps of a lane quarter
// taking alternate column chunks): the output-side columns go to dyn_out, the
// input-side ones to shared memory; then the eight warps apply the conv to the
// tile's rows and its groups' ng*g channels, reading x again (from L2: the units
// work on consecutive tiles, which share their x rows) and writing y.  The
// input-side corrections never reach HBM and x is read from HBM once.
//
// Roles (320 threads): warp 0 lane 0 issues the TMA loads, warp 1 lane 0 (CTA 0 of
// a pair) the MMAs into one of two TMEM accumulators, warps 2-9 the epilogue, which
// releases an accumulator as soon as it has read it, so the apply of one tile runs
// beside the MMAs of the next two.  All waits are bounded; the epilogue warps
// decide together, at a barrier that ORs their wait results, whether to go on.
#include <cudaTypedefs.h>

#include <map>
#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "tc_pair.cuh"
#include "tc_ptx.cuh"

namespace df2 {

namespace {

constexpr int CM = 128;   // rows of x per CTA tile (MMA M per CTA, TMEM lanes)
constexpr int CK = 64;    // reduction elements per box (one 128-byte swizzle row)
constexpr int kCtcThreads = 320;
constexpr int kCtcEpi = 256;                 // epilogue threads (warps 2-9)
constexpr uint32_t kXBox = CM * CK * 2;      // 16 KB
constexpr int kCtcMaxStages = 8;
constexpr uint32_t kBufCols = 256;           // TMEM columns per accumulator buffer

struct ConvTcArgs {
    const uint16_t* x;      // [P][C] bf16
    const float* base;      // [taps][C]: the input-side base kernel
    uint16_t* y;            // [P][C] bf16
    float* dyn_out;         // [P][taps][G]
    int32_t* dev_status;
    int P, C, B, g, G;
    int ng;                 // groups per tile
    int n_gt;               // group tiles (G / ng)
    int n_mu;               // units along the rows: 128-row tiles, or pairs of them
    int n_units;            // units launched (CTAs, CTA pairs or clusters of two pairs)
    int n_full_rounds;      // with n_half > 0: every unit's whole tiles, then its half tile
    int n_half;             // the last round's tiles split in two along the groups (0: none)
    int nstages;
    int ds_ld;              // floats per row of the staged input-side corrections
};

// W_proj rows one CTA stages per tile: all 2*taps*ng, or (pair) its side's taps*ng.
__host__ __device__ inline uint32_t ctc_b_rows(int taps, int ng, bool pair) {
    return uint32_t((pair ? 1 : 2) * taps * ng);
}
__host__ __device__ inline uint32_t ctc_stage_bytes(int taps, int ng, bool pair) {
    return kXBox + ctc_b_rows(taps, ng, pair) * CK * 2;
}
__host__ __device__ inline uint32_t ctc_ds_off(int nstages, int taps, int ng, bool pair) {
    uint32_t off = uint32_t(nstages) * ctc_stage_bytes(taps, ng, pair);
    off += uint32_t(2 * nstages + 5) * 8 + 16;  // barriers, TMEM address, abort flag
    return (off + 15) / 16 * 16;
}
__host__ __device__ inline uint32_t ctc_smem(int nstages, int taps, int ng, bool pair, int ds_ld) {
    return ctc_ds_off(nstages, taps, ng, pair) + uint32_t(CM) * uint32_t(ds_ld) * 4;
}

// 16-byte load / store with an L2 eviction-priority hint (the apply's last use of
// x, and outputs no kernel reads soon: they should not push x out of L2 before the
// other group tiles of its rows and their applies have read it).
__device__ __forceinline__ uint4 ld16_hint(const void* p, uint64_t pol) {
    uint4 v;
    asm volatile("ld.global.nc.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p), "l"(pol));
    return v;
}
__device__ __forceinline__ void st16_hint(void* p, uint4 v, uint64_t pol) {
    asm volatile("st.global.L2::cache_hint.v4.u32 [%0], {%1, %2, %3, %4}, %5;" ::"l"(p), "r"(v.x), "r"(v.y),
                 "r"(v.z), "r"(v.w), "l"(pol)
                 : "memory");
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// The conv of rows [m0, m0 + rows) (whole anchor blocks) on channels
// [c_lo, c_lo + nch*8), with the input-side corrections ds[r][j*ng + gi - g0] of
// the tile's groups.  Item = one 8-channel chunk of one block, walked row by row
// with the last TAPS rows of x in registers (the arithmetic of the standalone
// apply: acc = fma(base + d, x, acc) over the taps in order).  Consecutive threads
// take consecutive chunks of the same block, so every load and store of a row is
// coalesced.  Rows are loaded eight at a time; with PREF the next eight rows (of
// this item or the thread's next one) are in flight while the current ones are
// computed, so the epilogue keeps two groups of loads outstanding.
template <int TAPS, bool PREF>
__device__ __forceinline__ void ctc_apply(const ConvTcArgs& a, const float* ds, int64_t m0, int rows, int g0,
                                          int ngt, int etid) {
    const int nch = ngt * a.g / 8;
    const int c_lo = g0 * a.g;
    const int B = a.B, C = a.C;
    const int total = (rows / B) * nch;
    const bool one_group = (a.g % 8) == 0;  // a chunk's 8 channels share one group
    const uint64_t pol = tc::l2_policy_evict_first();
    auto load_rows = [&](int item, int t0, uint4 (&buf)[8]) {
        const int blk = item / nch, ch = item - blk * nch;
        const uint16_t* src = a.x + (m0 + int64_t(blk) * B + t0) * C + c_lo + ch * 8;
#pragma unroll
        for (int u = 0; u < 8; ++u)
            if (t0 + u < B) buf[u] = ld16_hint(src + int64_t(u) * C, pol);
    };
    uint4 cur[8], nxt[8];
    if (etid < total) load_rows(etid, 0, cur);
    for (int item = etid; item < total; item += kCtcEpi) {
        const int blk = item / nch, ch = item - blk * nch;
        const int c = c_lo + ch * 8;
        const int r0 = blk * B;
        float kb[TAPS][8], hist[TAPS][8];
#pragma unroll
        for (int j = 0; j < TAPS; ++j) {
            const float4 lo = __ldg(reinterpret_cast<const float4*>(a.base + int64_t(j) * C + c));
            const float4 hi = __ldg(reinterpret_cast<const float4*>(a.base + int64_t(j) * C + c + 4));
            kb[j][0] = lo.x; kb[j][1] = lo.y; kb[j][2] = lo.z; kb[j][3] = lo.w;
            kb[j][4] = hi.x; kb[j][5] = hi.y; kb[j][6] = hi.z; kb[j][7] = hi.w;
#pragma unroll
            for (int e = 0; e < 8; ++e) hist[j][e] = 0.f;
        }
        const int gl0 = c / a.g - g0;
        for (int t0 = 0; t0 < B; t0 += 8) {
            if (!PREF && t0 > 0) load_rows(item, t0, cur);
            if (PREF) {
                if (t0 + 8 < B) load_rows(item, t0 + 8, nxt);
                else if (item + kCtcEpi < total) load_rows(item + kCtcEpi, 0, nxt);
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int t = t0 + u;
                if (t >= B) break;
                const int r = r0 + t;
#pragma unroll
                for (int j = TAPS - 1; j > 0; --j)
#pragma unroll
                    for (int e = 0; e < 8; ++e) hist[j][e] = hist[j - 1][e];
                unpack8(cur[u], hist[0]);
                float acc[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) acc[e] = 0.f;
                const float* drow = ds + size_t(r) * a.ds_ld;
#pragma unroll
                for (int j = 0; j < TAPS; ++j) {
                    if (j > t) break;
                    if (one_group) {
                        const float d = drow[j * ngt + gl0];
#pragma unroll
                        for (int e = 0; e < 8; ++e) acc[e] = fmaf(kb[j][e] + d, hist[j][e], acc[e]);
                    } else {
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            const float d = drow[j * ngt + (c + e) / a.g - g0];
                            acc[e] = fmaf(kb[j][e] + d, hist[j][e], acc[e]);
                        }
                    }
                }
                uint4 w;
                w.x = pack_bf16x2(acc[0], acc[1]);
                w.y = pack_bf16x2(acc[2], acc[3]);
                w.z = pack_bf16x2(acc[4], acc[5]);
                w.w = pack_bf16x2(acc[6], acc[7]);
                st16_hint(a.y + (m0 + r) * C + c, w, pol);
            }
            if (PREF) {
#pragma unroll
                for (int u = 0; u < 8; ++u) cur[u] = nxt[u];
            }
        }
        if (!PREF && item + kCtcEpi < total) load_rows(item + kCtcEpi, 0, cur);
    }
}

// MC (with PAIR): clusters of two pairs on consecutive 256-row tiles and one group
// tile; the first pair loads the W_proj boxes once, multicast to the CTA of the same
// pair rank in the other pair, and a stage is free again when both pairs' MMAs have
// read it.  The units are then clusters: cluster step c + k * n_units covers row
// tiles (pair units) 2 mg and 2 mg + 1 of group tile gt, numbered gt-fastest.
//
// Half tiles: when the last round would leave units idle (a.n_half > 0), its tiles
// are split in two along the groups, ng/2 each (tm_wh: W_proj boxes of ng/2 rows,
// an MMA of half the N), so that 2L units share the last round's L tiles.
template <int TAPS, bool PAIR, bool MC = false>
__global__ void __launch_bounds__(kCtcThreads, 1)
conv_prepare_tc_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w,
                       const __grid_constant__ CUtensorMap tm_wh, const ConvTcArgs a) {
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte aligned by pointer arithmetic on the shared array (keeps every
    // access derived from it in the shared address space)
    uint8_t* smem = smem_raw + ((1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u);
    const int ng = a.ng, nstages = a.nstages;
    const uint32_t brows = ctc_b_rows(TAPS, ng, PAIR);
    const uint32_t stage_bytes = kXBox + brows * CK * 2;
    uint8_t* stages = smem;              // stage s: one x box, then the W_proj boxes
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + size_t(nstages) * stage_bytes);
    uint64_t* empty = full + nstages;
    uint64_t* tfull = empty + nstages;
    uint64_t* tempty = tfull + 2;
    uint64_t* mma_done = tempty + 2;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(mma_done + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
    float* ds = reinterpret_cast<float*>(smem + ctc_ds_off(nstages, TAPS, ng, PAIR));  // [CM][ds_ld]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int bid = int(blockIdx.x);
    const uint32_t crank = PAIR ? tc::cluster_ctarank() : 0u;
    const uint32_t rank = crank & 1u;        // rank inside the CTA pair
    const uint32_t lead_rank = crank & ~1u;  // cluster rank of this CTA's pair leader
    const int pp = int(crank >> 1);          // MC: which pair of the cluster
    const bool leader = rank == 0;
    const int unit = MC ? bid >> 2 : (PAIR ? bid >> 1 : bid);
    // tiles numbered group-tile fastest, dealt round-robin to the units: at every
    // step the units work on consecutive tiles, which share their x rows in L2
    const int n_rows_units = MC ? (a.n_mu + 1) / 2 : a.n_mu;
    const int total = n_rows_units * a.n_gt;
    // the unit's tiles: unit, unit + n_units, ...; with half tiles, its whole rounds
    // and then (unit < n_half) half `unit % 2` of whole tile F + unit / 2
    const int ntiles = a.n_half > 0 ? a.n_full_rounds + (unit < a.n_half ? 1 : 0)
                                    : (unit < total ? (total - unit + a.n_units - 1) / a.n_units : 0);
    struct Tile {
        int mt, g0, ngt;  // this CTA's 128-row tile, first group, groups
    };
    auto tile = [&](int k) {
        int T = unit + k * a.n_units, sub = -1;
        if (a.n_half > 0 && k == a.n_full_rounds) {
            T = a.n_full_rounds * a.n_units + unit / 2;
            sub = unit % 2;
        }
        const int mu0 = T / a.n_gt, gt = T - mu0 * a.n_gt;
        const int mu = MC ? 2 * mu0 + pp : mu0;
        Tile tl;
        tl.mt = PAIR ? 2 * mu + int(rank) : mu;
        tl.ngt = sub < 0 ? ng : ng / 2;
        tl.g0 = gt * ng + (sub > 0 ? ng / 2 : 0);
        return tl;
    };
    const int nbox = (a.C + CK - 1) / CK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < nstages; ++s) {
            tc::mbar_init(&full[s], 1);
            tc::mbar_init(&empty[s], MC ? 2 : 1);  // MC: both pairs' MMAs release a stage
        }
        for (int b = 0; b < 2; ++b) {
            tc::mbar_init(&tfull[b], 1);
            tc::mbar_init(&tempty[b], PAIR ? 16 : 8);  // the epilogue warps of one CTA, or of both
        }
        tc::mbar_init(mma_done, 1);
        *abort_flag = 0;
        tc::fence_mbar_init();
    }
    if (warp == 1) {
        if (PAIR) {
            tc::tmem_alloc_pair(tmem_holder, 512);
            tc::tmem_relinquish_pair();
        } else {
            tc::tmem_alloc(tmem_holder, 512);
            tc::tmem_relinquish();
        }
    }
    if (warp == 0 && lane == 0) {
        tc::prefetch_tmap(&tm_x);
        tc::prefetch_tmap(&tm_w);
    }
    tc::fence_before_sync();
    __syncthreads();
    if (PAIR) tc::cluster_sync_all();  // the peer's barriers are initialised before any remote use
    tc::fence_after_sync();
    const uint32_t tmem_base = *tmem_holder;

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------------ TMA producer
            // x: its rows are read by the group tiles of one row tile, then by the
            // epilogue; W_proj (a few MB) is read by every row tile
            const uint64_t pol_x = tc::l2_policy_evict_normal();
            const uint64_t pol_w = tc::l2_policy_evict_last();
            int stage = 0;
            uint32_t phase = 0;
            int8_t armed[kCtcMaxStages];
            for (int s = 0; s < kCtcMaxStages; ++s) armed[s] = -1;
            bool ok = true;
            for (int k = 0; k < ntiles && ok; ++k) {
                const Tile tl = tile(k);
                const int mt = tl.mt, g0 = tl.g0, ngt = tl.ngt;
                const uint32_t tile_bytes = kXBox + ctc_b_rows(TAPS, ngt, PAIR) * CK * 2;
                const CUtensorMap* wm = ngt == ng ? &tm_w : &tm_wh;
                for (int kb = 0; kb < nbox; ++kb) {
                    if (!tc::mbar_wait(&empty[stage], phase ^ 1, abort_flag)) { ok = false; break; }
                    // PAIR: CTA 0's full barrier counts the bytes both CTAs stage
                    if (leader) tc::mbar_arrive_expect_tx(&full[stage], tile_bytes * (PAIR ? 2u : 1u));
                    uint8_t* st = stages + size_t(stage) * stage_bytes;
                    const int xk = kb * CK;
                    if (PAIR) {
                        const uint32_t fb = tc::mapa_shared(tc::smem_u32(&full[stage]), lead_rank);
                        tc::tma_load_2d_pair(st, &tm_x, fb, xk, mt * CM, pol_x);
                        if (MC) {
                            // the first pair loads the W_proj boxes for both pairs
                            const uint16_t mask = uint16_t((1u << crank) | (1u << (crank + 2)));
                            if (pp == 0)
#pragma unroll
                                for (int j = 0; j < TAPS; ++j)
                                    tc::tma_load_2d_pair_mc(st + kXBox + size_t(j) * ngt * CK * 2, wm, fb, mask, xk,
                                                            (int(rank) * TAPS + j) * a.G + g0, pol_w);
                        } else {
#pragma unroll
                            for (int j = 0; j < TAPS; ++j)
                                tc::tma_load_2d_pair(st + kXBox + size_t(j) * ngt * CK * 2, wm, fb, xk,
                                                     (int(rank) * TAPS + j) * a.G + g0, pol_w);
                        }
                    } else {
                        tc::tma_load_2d(st, &tm_x, &full[stage], xk, mt * CM, pol_x);
#pragma unroll
                        for (int q = 0; q < 2 * TAPS; ++q)
                            tc::tma_load_2d(st + kXBox + size_t(q) * ngt * CK * 2, wm, &full[stage], xk,
                                            q * a.G + g0, pol_w);
                    }
                    armed[stage] = int8_t(phase);
                    if (++stage == nstages) { stage = 0; phase ^= 1; }
                }
            }
            if (!ok && leader) {
                // wait (bounded) for the copies in flight; PAIR: CTA 1's copies complete on
                // CTA 0's barriers, and CTA 1 leaves only after the closing cluster barrier
                volatile int never = 0;
                for (int s = 0; s < nstages; ++s)
                    if (armed[s] >= 0) tc::mbar_wait(&full[s], uint32_t(armed[s]), &never);
            }
        }
    } else if (warp == 1) {
        if (lane == 0 && leader) {
            // -------------------------------------------------------- MMA issuer
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (int k = 0; k < ntiles && ok; ++k) {
                const uint32_t idesc = tc::idesc_bf16_f32(PAIR ? 2 * CM : CM, 2 * TAPS * tile(k).ngt);
                const int b = k & 1;
                const uint32_t tph = (k >> 1) & 1;
                const bool drained = PAIR ? tc::mbar_wait_cluster(&tempty[b], tph ^ 1, abort_flag)
                                          : tc::mbar_wait(&tempty[b], tph ^ 1, abort_flag);
                if (!drained) break;
                tc::fence_after_sync();
                const uint32_t d_tmem = tmem_base + uint32_t(b) * kBufCols;
                for (int kb = 0; kb < nbox; ++kb) {
                    if (!tc::mbar_wait(&full[stage], phase, abort_flag)) { ok = false; break; }
                    tc::fence_after_sync();
                    uint8_t* st = stages + size_t(stage) * stage_bytes;
                    const uint32_t a0 = tc::smem_u32(st), b0 = tc::smem_u32(st + kXBox);
#pragma unroll
                    for (int kk = 0; kk < CK / 16; ++kk) {
                        const uint64_t ad = tc::sw128_kmajor_desc(a0 + 32 * kk);
                        const uint64_t bd = tc::sw128_kmajor_desc(b0 + 32 * kk);
                        const uint32_t acc = (kb | kk) != 0 ? 1u : 0u;
                        if (PAIR) tc::mma_bf16_pair(d_tmem, ad, bd, idesc, acc);
                        else tc::mma_bf16(d_tmem, ad, bd, idesc, acc);
                    }
                    if (PAIR) tc::mma_commit_pair(&empty[stage], MC ? 0xF : 0x3);
                    else tc::mma_commit(&empty[stage]);
                    if (++stage == nstages) { stage = 0; phase ^= 1; }
                }
                if (ok) {
                    if (PAIR) tc::mma_commit_pair(&tfull[b], uint16_t(0x3u << lead_rank));
                    else tc::mma_commit(&tfull[b]);
                }
            }
            if (PAIR) tc::mma_commit_pair(mma_done, uint16_t(0x3u << lead_rank));
            else tc::mma_commit(mma_done);
            volatile int never = 0;
            tc::mbar_wait(mma_done, 0, &never);
        }
    } else {
        // ---------------------------------------------------------- epilogue
        // warps 2-9: a warp reads TMEM lanes 32 (warp % 4) ..; the two warps of a
        // lane quarter take alternate 16-column chunks of the accumulator
        const int quarter = warp & 3;
        const int half_grp = (warp - 2) >> 2;
        const int r = quarter * 32 + lane;             // TMEM lane = the tile row of this thread
        const int etid = (warp - 2) * 32 + lane;       // 0 .. 255 for the apply
        const int64_t gld = int64_t(TAPS) * a.G;       // dyn_out row length
        const uint64_t pol_out = tc::l2_policy_evict_first();
        for (int k = 0; k < ntiles; ++k) {
            const Tile tl = tile(k);
            const int mt = tl.mt, g0 = tl.g0, ngt = tl.ngt;
            const int half_t = TAPS * ngt, N_t = 2 * half_t;  // this tile's columns
            const int b = k & 1;
            const uint32_t tph = (k >> 1) & 1;
            const bool got = tc::mbar_wait(&tfull[b], tph, abort_flag);
            // one decision for the epilogue warps; also orders the previous tile's
            // reads of ds before this tile's writes
            if (tc::named_barrier_or(1, kCtcEpi, !got)) break;
            tc::fence_after_sync();
            const int64_t m0 = int64_t(mt) * CM;
            const int64_t m = m0 + r;
            const bool row_ok = m < a.P;
            const uint32_t taddr = tmem_base + (uint32_t(quarter * 32) << 16) + uint32_t(b) * kBufCols;
            float* drow = ds + size_t(r) * a.ds_ld;
            for (int c0 = 16 * half_grp; c0 < N_t; c0 += 32) {
                float v[16];
                tc::tmem_ld16(taddr + uint32_t(c0), v);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int col = c0 + 4 * q;  // four columns of one side and one tap (ngt % 4 == 0)
                    if (col < half_t) {
#pragma unroll
                        for (int e = 0; e < 4; ++e) drow[col + e] = v[4 * q + e];
                    } else if (row_ok) {
                        const int oc = col - half_t, j = oc / ngt, gl = oc - j * ngt;
                        st16_hint(a.dyn_out + m * gld + int64_t(j) * a.G + g0 + gl,
                                  make_uint4(__float_as_uint(v[4 * q]), __float_as_uint(v[4 * q + 1]),
                                             __float_as_uint(v[4 * q + 2]), __float_as_uint(v[4 * q + 3])),
                                  pol_out);
                    }
                }
            }
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) {
                // the accumulator is free for the tile after next; PAIR: CTA 0's MMA
                // thread waits for both CTAs' epilogues
                if (PAIR) tc::mbar_arrive_cluster(tc::mapa_shared(tc::smem_u32(&tempty[b]), lead_rank));
                else tc::mbar_arrive(&tempty[b]);
            }
            tc::named_barrier(1, kCtcEpi);  // every row's corrections are staged
            const int64_t left = int64_t(a.P) - m0;
            const int rows = left <= 0 ? 0 : (left < CM ? int(left) : CM);
            ctc_apply<TAPS, (TAPS <= 2)>(a, ds, m0, rows, g0, ngt, etid);
        }
    }

    tc::fence_before_sync();
    __syncthreads();
    // PAIR: CTA 0's MMAs read this CTA's shared memory and write its TMEM; neither
    // CTA frees TMEM or exits before both are done
    if (PAIR) tc::cluster_sync_all();
    if (threadIdx.x == 0 && *abort_flag && a.dev_status) atomicOr(a.dev_status, DF2_STATUS_WAIT_TIMEOUT);
    if (warp == 1) {
        tc::fence_after_sync();
        if (PAIR) tc::tmem_dealloc_pair(tmem_base, 512);
        else tc::tmem_dealloc(tmem_base, 512);
    }
}

// ------------------------------------------------------------------- host --

PFN_cuTensorMapEncodeTiled_v12000 ctc_encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

bool ctc_map(CUtensorMap* m, const void* base, int64_t rows, int64_t cols, int box_rows) {
    auto fn = ctc_encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {cuuint64_t(cols), cuuint64_t(rows)};
    cuuint64_t strides[1] = {cuuint64_t(cols) * 2};
    cuuint32_t box[2] = {cuuint32_t(CK), cuuint32_t(box_rows)};
    cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

struct CtcPlan {
    bool ok = false;
    bool pair = false;
    bool mc = false;    // clusters of two pairs sharing the W_proj boxes
    int ng = 0, n_gt = 0, n_mu = 0, units = 0, nstages = 0, ds_ld = 0;
    int n_full_rounds = 0, n_half = 0;  // the last round in half tiles (n_half > 0)
};

// The last round split into half tiles when its L tiles would leave units idle and
// 2L of them fit: the 2L units that take one then finish about as soon as a whole
// tile would, with half the MMA work each.  A half tile has ng/2 groups, which must
// still fill whole 1024-byte swizzle atoms (ng/2 a multiple of 8).
void ctc_split_last_round(CtcPlan& p, int64_t total) {
    p.n_full_rounds = 0;
    p.n_half = 0;
    if (p.units <= 0 || total <= p.units || p.ng % 16 != 0) return;
    const int64_t full = total / p.units * p.units, left = total - full;
    if (left == 0 || 2 * left > p.units) return;
    p.n_full_rounds = int(total / p.units);
    p.n_half = int(2 * left);
}

// Clusters of two pairs of this kernel that fit at once (occupancy API), cached per
// device and launch shape; 0 when the query fails.
int ctc_mc_slots(int taps, size_t smem);

// Groups per tile: a divisor of G that is a multiple of 8 (each W_proj box then
// fills whole 1024-byte swizzle atoms) with 2*taps*ng <= 256 (the MMA's N and one
// TMEM buffer), chosen by a model of the time: rounds of tiles over the units,
// times the bytes a CTA stages per tile from L2 (its 128 x rows and its W_proj
// rows; half the W_proj rows on average in clusters of two pairs, whose first pair
// loads them for both).  Measured at the training-packed shape, a tile's time
// follows those L2 bytes, not its MMA work: N = 256 ran 136 us and N = 160 161 us
// without the apply.
CtcPlan ctc_plan(int64_t P, int C, int B, int taps, int g, int num_sms) {
    CtcPlan best;
    if (taps < 1 || taps > 4 || g < 1 || C % g != 0 || C % 8 != 0 || B < 1 || CM % B != 0 || P % B != 0)
        return best;
    if (P <= 0 || P > INT32_MAX || num_sms < 2) return best;
    const int G = C / g;
    const int n_mt = int((P + CM - 1) / CM);
    const bool pair = n_mt >= 2;
    const int n_mu = pair ? (n_mt + 1) / 2 : n_mt;
    const int slots = pair ? num_sms / 2 : num_sms;
    const uint32_t budget = 227 * 1024 - 1024;
    double best_cost = 0;
    for (int ng = 8; 2 * taps * ng <= 256; ng += 8) {
        if (G % ng != 0 || (ng * g) % 8 != 0) continue;
        const int ds_ld = (taps * ng) | 1;  // odd: a row's writes land in distinct banks
        int st = 0;
        for (int s = kCtcMaxStages; s >= 3; --s)
            if (ctc_smem(s, taps, ng, pair, ds_ld) <= budget) { st = s; break; }
        if (st == 0) continue;
        const int n_gt = G / ng;
        const int64_t total = int64_t(n_mu) * n_gt;
        const int units = int(total < slots ? total : slots);
        const int64_t rounds = (total + units - 1) / units;
        const double cost = double(rounds) * (CM + double(ctc_b_rows(taps, ng, pair)));
        if (!best.ok || cost < best_cost) {
            best_cost = cost;
            best.ok = true;
            best.pair = pair;
            best.mc = false;
            best.ng = ng;
            best.n_gt = n_gt;
            best.n_mu = n_mu;
            best.units = units;
            best.nstages = st;
            best.ds_ld = ds_ld;
        }
        if (pair && n_mu % 2 == 0) {
            const int mc_slots = ctc_mc_slots(taps, ctc_smem(st, taps, ng, true, ds_ld) + 1024);
            if (mc_slots > 0) {
                const int64_t total2 = int64_t(n_mu / 2) * n_gt;
                const int units2 = int(total2 < mc_slots ? total2 : mc_slots);
                const int64_t rounds2 = (total2 + units2 - 1) / units2;
                const double cost2 = double(rounds2) * (CM + 0.5 * double(ctc_b_rows(taps, ng, true)));
                if (cost2 < best_cost) {
                    best_cost = cost2;
                    best.ok = true;
                    best.pair = true;
                    best.mc = true;
                    best.ng = ng;
                    best.n_gt = n_gt;
                    best.n_mu = n_mu;
                    best.units = units2;
                    best.nstages = st;
                    best.ds_ld = ds_ld;
                }
            }
        }
    }
    if (best.ok) {
        const int64_t total = int64_t(best.mc ? best.n_mu / 2 : best.n_mu) * best.n_gt;
        ctc_split_last_round(best, total);
    }
    return best;
}

template <int TAPS, bool PAIR, bool MC = false>
cudaError_t ctc_launch(const CUtensorMap& tx, const CUtensorMap& tw, const CUtensorMap& twh, const ConvTcArgs& a,
                       cudaStream_t stream) {
    const size_t smem = ctc_smem(a.nstages, TAPS, a.ng, PAIR, a.ds_ld) + 1024;
    auto kernel = conv_prepare_tc_kernel<TAPS, PAIR, MC>;
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned((MC ? 4 : (PAIR ? 2 : 1)) * a.n_units));
    cfg.blockDim = dim3(kCtcThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = MC ? 4u : (PAIR ? 2u : 1u);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = PAIR ? 1 : 0;
    e = cudaLaunchKernelEx(&cfg, kernel, tx, tw, twh, a);
    note_launch();
    return e;
}

template <int TAPS>
int ctc_mc_slots_t(size_t smem) {
    auto kernel = conv_prepare_tc_kernel<TAPS, true, true>;
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)) != cudaSuccess)
        return 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(4);
    cfg.blockDim = dim3(kCtcThreads);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 4;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) != cudaSuccess) return 0;
    return n;
}

int ctc_mc_slots(int taps, size_t smem) {
    static std::mutex mu;
    static std::map<std::pair<int, int64_t>, int> cache;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    const std::pair<int, int64_t> key{dev, int64_t(taps) << 32 | int64_t(smem)};
    {
        std::lock_guard<std::mutex> lock(mu);
        auto it = cache.find(key);
        if (it != cache.end()) return it->second;
    }
    int n = 0;
    switch (taps) {
        case 1: n = ctc_mc_slots_t<1>(smem); break;
        case 2: n = ctc_mc_slots_t<2>(smem); break;
        case 3: n = ctc_mc_slots_t<3>(smem); break;
        case 4: n = ctc_mc_slots_t<4>(smem); break;
        default: n = 0;
    }
    std::lock_guard<std::mutex> lock(mu);
    cache[key] = n;
    return n;
}

int ctc_num_sms() {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return 0;
    return sms;
}

}  // namespace

bool conv_prepare_tc_supported(int64_t P, int C, int B, int taps, int g) {
    return P > 0 && ctc_plan(P, C, B, taps, g, ctc_num_sms() > 0 ? ctc_num_sms() : 2).ok;
}

cudaError_t conv_prepare_tc_launch(const uint16_t* x, int64_t P, int C, int B, int taps, int g,
                                   const uint16_t* W, const float* base, uint16_t* y, float* dyn_out,
                                   int32_t* dev_status, cudaStream_t stream) {
    const int sms = ctc_num_sms();
    const CtcPlan p = ctc_plan(P, C, B, taps, g, sms);
    if (!p.ok) return cudaErrorInvalidValue;
    const int G = C / g;
    CUtensorMap tx, tw, twh;
    if (!ctc_map(&tx, x, P, C, CM) || !ctc_map(&tw, W, int64_t(2) * taps * G, C, p.ng) ||
        !ctc_map(&twh, W, int64_t(2) * taps * G, C, p.n_half > 0 ? p.ng / 2 : p.ng))
        return cudaErrorInvalidValue;
    ConvTcArgs a{};
    a.x = x;
    a.base = base;
    a.y = y;
    a.dyn_out = dyn_out;
    a.dev_status = dev_status;
    a.P = int(P);
    a.C = C;
    a.B = B;
    a.g = g;
    a.G = G;
    a.ng = p.ng;
    a.n_gt = p.n_gt;
    a.n_mu = p.n_mu;
    a.n_units = p.units;
    a.n_full_rounds = p.n_full_rounds;
    a.n_half = p.n_half;
    a.nstages = p.nstages;
    a.ds_ld = p.ds_ld;
    switch (taps) {
#define DF2_CTC(TP)                                                                    \
    case TP:                                                                           \
        if (p.mc) return ctc_launch<TP, true, true>(tx, tw, twh, a, stream);           \
        return p.pair ? ctc_launch<TP, true>(tx, tw, twh, a, stream)                   \
                      : ctc_launch<TP, false>(tx, tw, twh, a, stream);
        DF2_CTC(1)
        DF2_CTC(2)
        DF2_CTC(3)
        DF2_CTC(4)
#undef DF2_CTC
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace df2
