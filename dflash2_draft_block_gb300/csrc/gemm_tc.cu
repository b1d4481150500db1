// Many-row GEMM on the tensor cores: out[m, n] = sum_k A[m, k] * B[n, k] with
// A = positions (h, or conv activations x) and B = the weight rows (W_lm, W_H,
// W_proj), bf16 in, fp32 accumulate in TMEM (tcgen05.mma, M = 128, N = 256).
//
// Two epilogues share one TMA/MMA pipeline:
//   * STORE: fp32 tile to global, columns split between two outputs (the conv
//     projection's input-side and output-side kernels; G = H(h)).
//   * TOPK: the unary logits of the head never leave the chip.  TMEM lane m of the
//     accumulator is position m, so each epilogue thread owns one position and
//     streams its 256 logits per tile against the K-th best so far; survivors go
//     into a per-thread min-heap of the K best (root = the current K-th), kept in
//     shared memory with a [slot][thread] layout so every lane hits its own bank.
//     A CTA owns 128 positions and a contiguous vocabulary range; its per-position
//     lists go to the workspace in rank order and topk_merge_sorted_kernel folds
//     the ranges.
//
// Roles (192 threads): warp 0 lane 0 issues the TMA loads (stages of kbox
// [128 x 64] A boxes and [256 x 64] B boxes, 128-byte swizzle), warp 1 lane 0
// issues tcgen05.mma into one of two TMEM accumulators (2 x 256 columns), warps
// 2-5 drain the other accumulator with tcgen05.ld.  All waits are bounded.
#include <cudaTypedefs.h>

#include <map>
#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "tc_pair.cuh"
#include "tc_ptx.cuh"

namespace df2 {

namespace {

constexpr int WM = 128;  // rows of A per tile (MMA M, TMEM lanes)
constexpr int WK = 64;   // K elements per box (one 128-byte swizzle row)
constexpr int kWideThreads = 192;
constexpr uint32_t kABox = WM * WK * 2;  // 16 KB
// rows of B per tile (MMA N, TMEM columns): 256
constexpr int kWideMaxStages = 8;

enum { EPI_STORE = 0, EPI_TOPK = 1 };

struct WideArgs {
    int M, N, Kd;           // A rows, B rows, reduction length
    int n_mt;               // M tiles
    int n_nt;               // N tiles
    int tiles_per_cta;      // consecutive N tiles per CTA
    int m_major;            // 1: consecutive CTAs share an M tile; 0: share an N range
    int linear;             // 1 (store only): the tiles, numbered N-fastest over (M tile or
                            // pair, N tile), dealt round-robin to n_units units
    int n_units;
    int nstages, kbox;
    // STORE
    float* out0;
    int64_t ld0;
    int n_split;
    float* out1;
    int64_t ld1;
    // TOPK
    int K;
    float* part_v;          // [n_groups][M][K]
    int* part_id;
    unsigned* thr_g;        // [M] best K-th value so far over all ranges (ordered key), or null
    // TOPK: G = A . W_H^T rides along as n_gt extra store tiles (B from the third
    // tensor map), G tile j on vocabulary range g_grp0 + j of every M tile (ranges
    // with fewer N tiles than the rest, so the longest unit stays as long)
    int n_gt, g_grp0;
    float* g_out;           // [M][g_n]
    int g_n;
    int32_t* dev_status;
    unsigned* zero_words;   // [n_zero] zeroed by CTA 0 for the next kernel in the stream
    int n_zero;
};

__host__ __device__ inline uint32_t wide_stage_bytes(int kbox, int bn) {
    return uint32_t(kbox) * (kABox + uint32_t(bn) * WK * 2);
}

__host__ __device__ inline uint32_t wide_smem(int nstages, int kbox, int epi, int K, int bn) {
    uint32_t off = uint32_t(nstages) * wide_stage_bytes(kbox, bn);
    off += uint32_t(2 * nstages + 5) * 8 + 16;  // barriers, TMEM address, abort flag
    off = (off + 15) / 16 * 16;
    if (epi == EPI_TOPK) off += uint32_t(K) * 128 * 8;  // heaps [K][128] (value, id)
    return off;
}

// Min-heap by rank order kept by one thread in a [slot][thread] shared array of
// packed (value bits, id) pairs: the root is the worst of the kept entries.
// (v, i) replaces the root and sifts down.
__device__ __forceinline__ void heap_replace_root(uint2* hp, int K, int tt, float v, int i) {
    int pos = 0;
    while (true) {
        const int c1 = 2 * pos + 1;
        if (c1 >= K) break;
        int c = c1;
        uint2 ce = hp[c1 * 128 + tt];
        if (c1 + 1 < K) {
            const uint2 c2 = hp[(c1 + 1) * 128 + tt];
            if (ranks_before(__uint_as_float(ce.x), int(ce.y), __uint_as_float(c2.x), int(c2.y))) {
                c = c1 + 1;  // the worse child
                ce = c2;
            }
        }
        if (!ranks_before(v, i, __uint_as_float(ce.x), int(ce.y))) break;
        hp[pos * 128 + tt] = ce;
        pos = c;
    }
    hp[pos * 128 + tt] = make_uint2(__float_as_uint(v), unsigned(i));
}

// (v, i) added at position n of a heap of n entries (n < capacity), sifted up: while
// the heap is filling, a new entry climbs ~1-2 levels on average, where replacing a
// root above placeholder entries would sift it down through all of them.
__device__ __forceinline__ void heap_push(uint2* hp, int n, int tt, float v, int i) {
    int pos = n;
    while (pos > 0) {
        const int par = (pos - 1) >> 1;
        const uint2 pe = hp[par * 128 + tt];
        if (!ranks_before(__uint_as_float(pe.x), int(pe.y), v, i)) break;  // the parent is the worse
        hp[pos * 128 + tt] = pe;
        pos = par;
    }
    hp[pos * 128 + tt] = make_uint2(__float_as_uint(v), unsigned(i));
}

// Order-preserving map of finite floats to unsigned keys (0 = below everything).
__device__ __forceinline__ unsigned order_key(float v) {
    const unsigned u = __float_as_uint(v);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_value(unsigned k) {
    if (k < 0x00800000u) return -INFINITY;  // below the key of -inf: nothing published yet
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

}  // namespace

namespace {

// PAIR: a cluster of two CTAs shares each 256 x WN tile (cta_group::2).  CTA r
// of the pair stages A rows [128 r, 128 r + 128) of the pair's 256 and B rows
// [WN/2 r, WN/2 (r + 1)) of the tile's WN; CTA 0's MMA thread computes the whole
// tile, and each CTA's TMEM receives its own 128 rows x WN columns.  Each CTA thus
// stages half the B bytes per flop of the one-CTA tile.
// MC (with PAIR): a cluster of two pairs on consecutive M tiles of the same N
// range.  The first pair's CTAs load the B halves once, multicast to the CTA of the
// same pair rank in the other pair; a stage is free again when both pairs' MMAs
// have read it (their commits arrive on every CTA's empty barrier).  A quarter less
// data crosses from L2 to the SMs per flop.
template <int EPI, int WN, bool PAIR, bool GT, bool MC = false>
__global__ void __launch_bounds__(kWideThreads, 1)
gemm_wide_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                 const __grid_constant__ CUtensorMap tm_g, const WideArgs args) {
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte aligned, by pointer arithmetic on the shared array so that the
    // compiler keeps every access derived from it in the shared address space
    uint8_t* smem = smem_raw + ((1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u);
    constexpr int kBRows = PAIR ? WN / 2 : WN;  // B rows this CTA stages per tile
    constexpr uint32_t kBBox = kBRows * WK * 2;
    const int nstages = args.nstages, kbox = args.kbox;
    const uint32_t stage_bytes = wide_stage_bytes(kbox, kBRows);
    uint8_t* stages = smem;  // stage s: kbox A boxes, then kbox B boxes
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + size_t(nstages) * stage_bytes);
    uint64_t* empty = full + nstages;
    uint64_t* tfull = empty + nstages;
    uint64_t* tempty = tfull + 2;
    uint64_t* mma_done = tempty + 2;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(mma_done + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
    uint32_t heap_off = uint32_t(nstages) * stage_bytes + uint32_t(2 * nstages + 5) * 8 + 16;
    heap_off = (heap_off + 15) / 16 * 16;
    uint2* hp = reinterpret_cast<uint2*>(smem + heap_off);      // [K][128] (value bits, id)

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int bid = int(blockIdx.x);
    if (bid == 0)
        for (int i = threadIdx.x; i < args.n_zero; i += blockDim.x) args.zero_words[i] = 0u;
    const int n_groups = (args.n_nt + args.tiles_per_cta - 1) / args.tiles_per_cta;
    // the work unit: one M tile, or (PAIR) one pair of M tiles, times a range of N tiles
    const uint32_t crank = PAIR ? tc::cluster_ctarank() : 0u;
    const uint32_t rank = crank & 1u;         // rank inside the CTA pair
    const uint32_t lead_rank = crank & ~1u;   // cluster rank of this CTA's pair leader
    const bool leader = rank == 0;
    const int unit = PAIR ? bid >> 1 : bid;
    const int n_mu = PAIR ? (args.n_mt + 1) / 2 : args.n_mt;
    const int mu = args.m_major ? unit / n_groups : unit % n_mu;
    const int mt = PAIR ? 2 * mu + int(rank) : mu;
    const int grp = args.m_major ? unit % n_groups : unit / n_mu;
    const int nt0 = grp * args.tiles_per_cta;
    const int nt1 = min(args.n_nt, nt0 + args.tiles_per_cta);
    // this CTA's tiles k = 0 .. ntiles-1: a fixed M tile over N tiles nt0.., or (linear)
    // tiles unit, unit + n_units, ... of the N-fastest numbering.  In the linear walk a
    // unit's store epilogue overlaps its next tile's MMAs, and at every step the units
    // work on consecutive tiles, which share their A rows in L2.
    const int total = n_mu * args.n_nt;
    const int n_rng = nt1 - nt0;
    // this unit also computes G tile grp - g_grp0
    // (GT: launches with G tiles; the others compile without them)
    const bool has_g = GT && EPI == EPI_TOPK && grp >= args.g_grp0 && grp < args.g_grp0 + args.n_gt;
    const int ntiles = args.linear ? (unit < total ? (total - unit + args.n_units - 1) / args.n_units : 0)
                                   : n_rng + (has_g ? 1 : 0);
    auto tile_is_g = [&](int k) { return has_g && k == n_rng; };
    auto tile_nt = [&](int k) {
        if (tile_is_g(k)) return grp - args.g_grp0;
        return args.linear ? (unit + k * args.n_units) % args.n_nt : nt0 + k;
    };
    auto tile_mt = [&](int k) {
        if (!args.linear) return mt;
        const int mu_k = (unit + k * args.n_units) / args.n_nt;
        return PAIR ? 2 * mu_k + int(rank) : mu_k;
    };
    const int nbox = (args.Kd + WK - 1) / WK;
    const int nk = (nbox + kbox - 1) / kbox;

    if (threadIdx.x == 0) {
        for (int s = 0; s < nstages; ++s) {
            tc::mbar_init(&full[s], 1);
            tc::mbar_init(&empty[s], MC ? 2 : 1);  // MC: both pairs' MMAs release a stage
        }
        for (int b = 0; b < 2; ++b) {
            tc::mbar_init(&tfull[b], 1);
            tc::mbar_init(&tempty[b], PAIR ? 8 : 4);  // the epilogue warps of one CTA, or of both
        }
        tc::mbar_init(mma_done, 1);
        *abort_flag = 0;
        tc::fence_mbar_init();
    }
    if (EPI == EPI_TOPK && warp >= 2) {
        const int tt = (warp - 2) * 32 + lane;
        for (int k = 0; k < args.K; ++k) hp[k * 128 + tt] = make_uint2(__float_as_uint(-INFINITY), unsigned(INT_MAX));
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
        tc::prefetch_tmap(&tm_a);
        tc::prefetch_tmap(&tm_b);
        if (GT) tc::prefetch_tmap(&tm_g);
    }
    tc::fence_before_sync();
    __syncthreads();
    if (PAIR) tc::cluster_sync_all();  // the peer's barriers are initialised before any remote use
    tc::fence_after_sync();
    const uint32_t tmem_base = *tmem_holder;

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------------ TMA producer
            const uint64_t pol_a = tc::l2_policy_evict_last();
            const uint64_t pol_b = EPI == EPI_TOPK ? tc::l2_policy_evict_first() : tc::l2_policy_evict_last();
            int stage = 0;
            uint32_t phase = 0;
            int8_t armed[kWideMaxStages];
            for (int s = 0; s < kWideMaxStages; ++s) armed[s] = -1;
            bool ok = true;
            for (int k = 0; k < ntiles && ok; ++k) {
                const int nt = tile_nt(k), mtk = tile_mt(k);
                const bool gt = tile_is_g(k);
                for (int kb = 0; kb < nk; ++kb) {
                    const int nb = min(kbox, nbox - kb * kbox);
                    if (!tc::mbar_wait(&empty[stage], phase ^ 1, abort_flag)) { ok = false; break; }
                    // PAIR: CTA 0's full barrier counts the bytes both CTAs stage
                    if (leader)
                        tc::mbar_arrive_expect_tx(&full[stage], uint32_t(nb) * (kABox + kBBox) * (PAIR ? 2u : 1u));
                    uint8_t* st = stages + size_t(stage) * stage_bytes;
                    const int yb = nt * WN + int(rank) * kBRows;
                    for (int j = 0; j < nb; ++j) {
                        const int x = (kb * kbox + j) * WK;
                        uint8_t* da = st + size_t(j) * kABox;
                        uint8_t* db = st + size_t(kbox) * kABox + size_t(j) * kBBox;
                        if (PAIR) {
                            const uint32_t fb = tc::mapa_shared(tc::smem_u32(&full[stage]), lead_rank);
                            tc::tma_load_2d_pair(da, &tm_a, fb, x, mtk * WM, pol_a);
                            if (MC) {
                                // the first pair loads the B halves for both pairs
                                const uint16_t mask = uint16_t((1u << crank) | (1u << (crank + 2)));
                                if (crank < 2) tc::tma_load_2d_pair_mc(db, gt ? &tm_g : &tm_b, fb, mask, x, yb, pol_b);
                            } else if (gt) {
                                tc::tma_load_2d_pair(db, &tm_g, fb, x, yb, pol_b);
                            } else {
                                tc::tma_load_2d_pair(db, &tm_b, fb, x, yb, pol_b);
                            }
                        } else {
                            tc::tma_load_2d(da, &tm_a, &full[stage], x, mtk * WM, pol_a);
                            if (gt) tc::tma_load_2d(db, &tm_g, &full[stage], x, yb, pol_b);
                            else tc::tma_load_2d(db, &tm_b, &full[stage], x, yb, pol_b);
                        }
                    }
                    armed[stage] = int8_t(phase);
                    if (++stage == nstages) { stage = 0; phase ^= 1; }
                }
            }
            if (!ok && leader) {
                // wait (bounded) for the copies in flight; PAIR: CTA 1's copies complete on
                // CTA 0's barriers too, and CTA 1 leaves only after the closing cluster
                // barrier, which CTA 0 reaches after this
                volatile int never = 0;
                for (int s = 0; s < nstages; ++s)
                    if (armed[s] >= 0) tc::mbar_wait(&full[s], uint32_t(armed[s]), &never);
            }
        }
    } else if (warp == 1) {
        if (lane == 0 && leader) {
            // -------------------------------------------------------- MMA issuer
            constexpr uint32_t idesc = tc::idesc_bf16_f32(PAIR ? 2 * WM : WM, WN);
            int stage = 0;
            uint32_t phase = 0;
            int it = 0;
            bool ok = true;
            for (int k = 0; k < ntiles && ok; ++k, ++it) {
                const int b = it & 1;
                const uint32_t tph = (it >> 1) & 1;
                const bool drained = PAIR ? tc::mbar_wait_cluster(&tempty[b], tph ^ 1, abort_flag)
                                          : tc::mbar_wait(&tempty[b], tph ^ 1, abort_flag);
                if (!drained) break;
                tc::fence_after_sync();
                const uint32_t d_tmem = tmem_base + uint32_t(b * WN);
                for (int kb = 0; kb < nk; ++kb) {
                    if (!tc::mbar_wait(&full[stage], phase, abort_flag)) { ok = false; break; }
                    tc::fence_after_sync();
                    const int nb = min(kbox, nbox - kb * kbox);
                    uint8_t* st = stages + size_t(stage) * stage_bytes;
                    for (int j = 0; j < nb; ++j) {
                        const uint32_t a0 = tc::smem_u32(st + size_t(j) * kABox);
                        const uint32_t b0 = tc::smem_u32(st + size_t(kbox) * kABox + size_t(j) * kBBox);
#pragma unroll
                        for (int k = 0; k < WK / 16; ++k) {
                            const uint64_t ad = tc::sw128_kmajor_desc(a0 + 32 * k);
                            const uint64_t bd = tc::sw128_kmajor_desc(b0 + 32 * k);
                            const uint32_t acc = (kb | j | k) != 0 ? 1u : 0u;
                            if (PAIR) tc::mma_bf16_pair(d_tmem, ad, bd, idesc, acc);
                            else tc::mma_bf16(d_tmem, ad, bd, idesc, acc);
                        }
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
        const int quarter = warp & 3;
        const int tt = (warp - 2) * 32 + lane;      // heap column
        const int m = mt * WM + quarter * 32 + lane;  // A row (position) of this thread
        const bool row_ok = m < args.M;
        float tv = -INFINITY;                       // heap root: the K-th best so far
        int tid = INT_MAX;
        int hn = 0;                                 // entries in the heap (K once it is full)
        // Best K-th value any vocabulary range has reached for this position: a
        // logit strictly below it cannot be in the global top-K.
        float gthr = -INFINITY;
        int it = 0;
        for (int k = 0; k < ntiles; ++k, ++it) {
            const int nt = tile_nt(k);
            const bool gt = tile_is_g(k);
            const int b = it & 1;
            const uint32_t tph = (it >> 1) & 1;
            const bool got = tc::mbar_wait(&tfull[b], tph, abort_flag);
            if (!__all_sync(kFull, got)) break;
            tc::fence_after_sync();
            const uint32_t taddr = tmem_base + (uint32_t(quarter * 32) << 16) + uint32_t(b * WN);
            if (EPI == EPI_STORE || gt) {
                // the store epilogue's row for this tile (the top-K epilogue's is fixed)
                const int ms = tile_mt(k) * WM + quarter * 32 + lane;
                const bool ms_ok = ms < args.M;
                // where a store tile goes: the store launch's outputs, or (top-K) G
                float* so0 = EPI == EPI_STORE ? args.out0 : args.g_out;
                float* so1 = EPI == EPI_STORE ? args.out1 : nullptr;
                const int64_t sl0 = EPI == EPI_STORE ? args.ld0 : args.g_n;
                const int64_t sl1 = EPI == EPI_STORE ? args.ld1 : 0;
                const int sns = EPI == EPI_STORE ? args.n_split : args.g_n;
                const int sN = EPI == EPI_STORE ? args.N : args.g_n;
                for (int c0 = 0; c0 < WN; c0 += 16) {
                    float v[16];
                    tc::tmem_ld16(taddr + uint32_t(c0), v);
                    const int n0 = nt * WN + c0;
                    if (ms_ok && n0 < sN) {
                        const bool whole = n0 + 16 <= sN;
                        const bool side0 = n0 + 16 <= sns, side1 = n0 >= sns;
                        float* dst = nullptr;
                        if (side0) dst = so0 + int64_t(ms) * sl0 + n0;
                        else if (side1) dst = so1 + int64_t(ms) * sl1 + (n0 - sns);
                        if (whole && dst && (reinterpret_cast<uintptr_t>(dst) & 15) == 0) {
#pragma unroll
                            for (int q = 0; q < 4; ++q)
                                reinterpret_cast<float4*>(dst)[q] =
                                    make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
                        } else {
#pragma unroll
                            for (int e = 0; e < 16; ++e) {
                                const int n = n0 + e;
                                if (n >= sN) break;
                                if (n < sns) so0[int64_t(ms) * sl0 + n] = v[e];
                                else so1[int64_t(ms) * sl1 + (n - sns)] = v[e];
                            }
                        }
                    }
                }
            } else {
                for (int c0 = 0; c0 < WN; c0 += 16) {
                    float v[16];
                    tc::tmem_ld16(taddr + uint32_t(c0), v);
                    const int n0 = nt * WN + c0;
                    // the chunk's candidates that beat the current K-th, as a bit mask;
                    // the warp then inserts them in rounds, one per lane per round, so
                    // the cost is the largest per-lane count, not one round per column
                    unsigned mask = 0;
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const int n = n0 + e;
                        if (row_ok && n < args.N && v[e] >= gthr && ranks_before(v[e], n, tv, tid))
                            mask |= 1u << e;
                    }
                    while (__any_sync(kFull, mask != 0)) {
                        if (mask) {
                            const int j = __ffs(mask) - 1;
                            mask &= mask - 1;
                            float cv = v[0];
#pragma unroll
                            for (int e = 1; e < 16; ++e) cv = (j == e) ? v[e] : cv;
                            const int n = n0 + j;
                            if (ranks_before(cv, n, tv, tid)) {
                                if (hn < args.K) {
                                    heap_push(hp, hn, tt, cv, n);
                                    if (++hn == args.K) {  // full: its root is the K-th best
                                        const uint2 root = hp[tt];
                                        tv = __uint_as_float(root.x);
                                        tid = int(root.y);
                                    }
                                } else {
                                    heap_replace_root(hp, args.K, tt, cv, n);
                                    const uint2 root = hp[tt];
                                    tv = __uint_as_float(root.x);
                                    tid = int(root.y);
                                }
                            }
                        }
                    }
                }
            }
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) {
                // PAIR: CTA 0's MMA thread waits for both CTAs' epilogues
                if (PAIR) tc::mbar_arrive_cluster(tc::mapa_shared(tc::smem_u32(&tempty[b]), lead_rank));
                else tc::mbar_arrive(&tempty[b]);
            }
            if (EPI == EPI_TOPK && !gt && args.thr_g && row_ok) {
                unsigned k = 0;
                if (tid != INT_MAX) k = order_key(tv);  // heap full: publish its K-th value
                const unsigned old = atomicMax(args.thr_g + m, k);
                gthr = key_value(old > k ? old : k);
            }
        }
        if (EPI == EPI_TOPK && row_ok) {
            // heap -> rank order (repeatedly move the worst to the end), then write; the
            // slots past the hn entries still hold their (-inf, no id) placeholders
            const int K = args.K;
            for (int end = hn - 1; end > 0; --end) {
                const uint2 root = hp[tt], last = hp[end * 128 + tt];
                hp[end * 128 + tt] = root;
                heap_replace_root(hp, end, tt, __uint_as_float(last.x), int(last.y));
            }
            const size_t base = (size_t(grp) * args.M + m) * K;
            for (int k = 0; k < K; ++k) {
                const uint2 en = hp[k * 128 + tt];
                const bool ok_k = int(en.y) != INT_MAX;
                args.part_v[base + k] = ok_k ? __uint_as_float(en.x) : -INFINITY;
                args.part_id[base + k] = ok_k ? int(en.y) : -1;
            }
        }
    }

    tc::fence_before_sync();
    __syncthreads();
    // PAIR: CTA 0's MMAs read this CTA's shared memory and write its TMEM; neither
    // CTA frees TMEM or exits before both are done
    if (PAIR) tc::cluster_sync_all();
    if (threadIdx.x == 0 && *abort_flag && args.dev_status) atomicOr(args.dev_status, DF2_STATUS_WAIT_TIMEOUT);
    if (warp == 1) {
        tc::fence_after_sync();
        if (PAIR) tc::tmem_dealloc_pair(tmem_base, 512);
        else tc::tmem_dealloc(tmem_base, 512);
    }
}

}  // namespace

// ------------------------------------------------------------------- host --

namespace {

PFN_cuTensorMapEncodeTiled_v12000 wide_encode_fn() {
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

bool wide_map(CUtensorMap* m, const void* base, int64_t rows, int64_t cols, int box_rows) {
    auto fn = wide_encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {cuuint64_t(cols), cuuint64_t(rows)};
    cuuint64_t strides[1] = {cuuint64_t(cols) * 2};
    cuuint32_t box[2] = {cuuint32_t(WK), cuuint32_t(box_rows)};
    cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 256 columns for every K: an N = 192 MMA ran at ~79% of the N = 256 rate, which
// cost more than the fourth pipeline stage the 64-entry heaps displace
int wide_bn(int epi, int K) {
    (void)epi;
    (void)K;
    return 256;
}

// Pipeline stages that fit beside the epilogue's heaps: a stage holds one 64-wide
// K slice of A (128 rows) and of the B rows the CTA stages (256, or 128 in a pair).
int wide_stages(int epi, int K, bool pair) {
    const uint32_t budget = 227 * 1024 - 1024;
    const int brows = pair ? wide_bn(epi, K) / 2 : wide_bn(epi, K);
    for (int s = pair ? 6 : 4; s >= 2; --s)
        if (wide_smem(s, 1, epi, K, brows) <= budget) return s;
    return 0;
}

// Vocabulary ranges per M tile for the top-K epilogue: enough CTAs to fill whole
// waves of the SMs (at least 90% of the last wave busy).
int wide_groups(int n_mt, int n_nt, int num_sms) {
    for (int w = 1; w <= 16; ++w) {
        int S = (w * num_sms) / n_mt;
        if (S < 1) continue;
        if (S > n_nt) S = n_nt;
        if (double(n_mt) * S >= 0.9 * w * num_sms || S == n_nt) {
            const int tpc = (n_nt + S - 1) / S;
            return (n_nt + tpc - 1) / tpc;
        }
    }
    return n_nt < num_sms ? n_nt : num_sms;
}

// The tiling of one launch: a CTA per 128-row M tile, or, with two or more M
// tiles, a CTA pair per two M tiles (the last pair's second tile may lie past M;
// its CTA still stages its half of every B tile).
struct WidePlan {
    bool pair;
    bool mc;            // top-K: clusters of two pairs sharing the W_lm tiles
    bool linear;        // store: units take runs of the M-fastest tile order
    int n_mt, n_nt;     // 128-row M tiles, 256-row N tiles
    int n_mu;           // work units along M: tiles, or pairs of tiles
    int tiles_per_cta;  // tiles per unit (consecutive N tiles, or a run of the linear order)
    int n_groups;       // N ranges per unit (top-K)
    int units;          // units launched (each one CTA or one CTA pair)
    int nstages;
};

// Clusters of two CTA pairs (four SMs of one GPC) that can run at once with the
// top-K kernel's shared memory, from the occupancy API, once per device and shape
// class; 0 when the query fails.
int mc_cluster_slots(int K, int nstages);

WidePlan wide_plan(int epi, int64_t M, int64_t N, int K, int num_sms, bool persistent) {
    WidePlan p{};
    const int bn = wide_bn(epi, K);
    p.n_mt = int((M + WM - 1) / WM);
    p.n_nt = int((N + bn - 1) / bn);
    p.pair = p.n_mt >= 2 && wide_stages(epi, K, true) >= 2;
    p.n_mu = p.pair ? (p.n_mt + 1) / 2 : p.n_mt;
    p.nstages = wide_stages(epi, K, p.pair);
    const int slots = p.pair ? num_sms / 2 : num_sms;
    if (persistent) {
        const int groups = wide_groups(p.n_mu, p.n_nt, slots);
        p.tiles_per_cta = (p.n_nt + groups - 1) / groups;
        p.n_groups = (p.n_nt + p.tiles_per_cta - 1) / p.tiles_per_cta;
        p.units = p.n_mu * p.n_groups;
        if (epi == EPI_TOPK && p.pair && p.n_mu % 2 == 0) {
            // the same with clusters of two pairs: fewer of them fit at once (four SMs
            // of one GPC each), but a tile moves a quarter fewer bytes from L2, which
            // feeds this kernel.  Cost: waves x tiles per unit x relative tile time.
            const int mc_slots = 2 * mc_cluster_slots(K, p.nstages);
            if (mc_slots >= 2) {
                const int g2 = wide_groups(p.n_mu, p.n_nt, mc_slots);
                const int tpc2 = (p.n_nt + g2 - 1) / g2;
                const int ng2 = (p.n_nt + tpc2 - 1) / tpc2;
                const int units2 = p.n_mu * ng2;
                const double cost_pair = double((p.units + slots - 1) / slots) * p.tiles_per_cta;
                const double cost_mc = double((units2 + mc_slots - 1) / mc_slots) * tpc2 * 0.85;
                if (cost_mc < cost_pair) {
                    p.mc = true;
                    p.tiles_per_cta = tpc2;
                    p.n_groups = ng2;
                    p.units = units2;
                }
            }
        }
    } else {
        // one wave of units dealt the tiles round-robin
        const int total = p.n_mu * p.n_nt;
        p.linear = true;
        p.units = total < slots ? total : slots;
        p.tiles_per_cta = (total + p.units - 1) / p.units;
        p.n_groups = p.n_nt;
    }
    return p;
}

template <int EPI, int BN, bool PAIR, bool GT, bool MC = false>
cudaError_t launch_wide(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tg, const WideArgs& a,
                        int grid, cudaStream_t stream) {
    const int brows = PAIR ? BN / 2 : BN;
    const size_t smem = wide_smem(a.nstages, a.kbox, EPI, a.K, brows) + 1024;
    auto kernel = gemm_wide_kernel<EPI, BN, PAIR, GT, MC>;
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(grid));
    cfg.blockDim = dim3(kWideThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = MC ? 4u : (PAIR ? 2u : 1u);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = PAIR ? 1 : 0;
    e = cudaLaunchKernelEx(&cfg, kernel, ta, tb, tg, a);
    note_launch();
    return e;
}

template <int EPI>
cudaError_t launch_plan(const WidePlan& p, const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tg,
                        const WideArgs& a, cudaStream_t stream) {
    const int grid = (p.pair ? 2 : 1) * p.units;
    if constexpr (EPI == EPI_TOPK) {
        // clusters of two pairs on consecutive position tiles of one vocabulary range
        // (the units of a range are consecutive: an even number of pairs keeps every
        // cluster inside one range)
        const bool mc = p.mc;
        if (a.n_gt > 0) {
            if (mc) return launch_wide<EPI, 256, true, true, true>(ta, tb, tg, a, grid, stream);
            return p.pair ? launch_wide<EPI, 256, true, true>(ta, tb, tg, a, grid, stream)
                          : launch_wide<EPI, 256, false, true>(ta, tb, tg, a, grid, stream);
        }
        if (mc) return launch_wide<EPI, 256, true, false, true>(ta, tb, tg, a, grid, stream);
    }
    return p.pair ? launch_wide<EPI, 256, true, false>(ta, tb, tg, a, grid, stream)
                  : launch_wide<EPI, 256, false, false>(ta, tb, tg, a, grid, stream);
}

int mc_cluster_slots(int K, int nstages) {
    static std::mutex mu;
    static std::map<std::pair<int, int>, int> cache;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    const std::pair<int, int> key{dev, (K << 8) | nstages};
    {
        std::lock_guard<std::mutex> lock(mu);
        auto it = cache.find(key);
        if (it != cache.end()) return it->second;
    }
    const size_t smem = wide_smem(nstages, 1, EPI_TOPK, K, 128) + 1024;
    auto kernel = gemm_wide_kernel<EPI_TOPK, 256, true, false, true>;
    int n = 0;
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)) == cudaSuccess) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(4);
        cfg.blockDim = dim3(kWideThreads);
        cfg.dynamicSmemBytes = smem;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 4;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) != cudaSuccess) n = 0;
    }
    std::lock_guard<std::mutex> lock(mu);
    cache[key] = n;
    return n;
}

}  // namespace

bool wide_supported(int64_t M, int64_t N, int64_t Kd, int K) {
    return M >= 1 && N >= 1 && Kd >= 1 && Kd % 8 == 0 && M <= INT32_MAX && N <= INT32_MAX &&
           Kd <= INT32_MAX && K <= 64 && wide_stages(EPI_TOPK, K < 1 ? 1 : K, false) >= 2;
}

size_t wide_topk_workspace(int64_t M, int64_t N, int K, int num_sms) {
    const WidePlan p = wide_plan(EPI_TOPK, M, N, K, num_sms, true);
    return size_t(p.n_groups) * size_t(M) * size_t(K) * 8 + size_t(M) * 4;
}

cudaError_t wide_store_launch(const uint16_t* A, int64_t M, const uint16_t* B, int64_t N, int64_t Kd,
                              float* out0, int64_t ld0, int64_t n_split, float* out1, int64_t ld1,
                              int32_t* dev_status, cudaStream_t stream) {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
        return cudaErrorInvalidValue;
    const WidePlan p = wide_plan(EPI_STORE, M, N, 0, sms, false);
    CUtensorMap ta, tb;
    if (!wide_map(&ta, A, M, Kd, WM) || !wide_map(&tb, B, N, Kd, p.pair ? 128 : 256))
        return cudaErrorInvalidValue;
    WideArgs a{};
    a.M = int(M); a.N = int(N); a.Kd = int(Kd);
    a.n_mt = p.n_mt;
    a.n_nt = p.n_nt;
    a.tiles_per_cta = p.tiles_per_cta;
    a.m_major = 1;
    a.linear = p.linear ? 1 : 0;
    a.n_units = p.units;
    a.nstages = p.nstages;
    a.kbox = 1;
    a.out0 = out0; a.ld0 = ld0; a.n_split = int(n_split); a.out1 = out1; a.ld1 = ld1;
    a.K = 0;
    a.dev_status = dev_status;
    return launch_plan<EPI_STORE>(p, ta, tb, tb, a, stream);
}

cudaError_t wide_topk_launch(const uint16_t* A, int64_t M, const uint16_t* B, int64_t N, int64_t Kd, int K,
                             int32_t* ids, float* vals, void* ws, int32_t* dev_status, int num_sms,
                             cudaStream_t stream, TopkParts* parts_out, unsigned* zero_words, int n_zero,
                             const uint16_t* W_H, int64_t r, float* G) {
    const WidePlan p = wide_plan(EPI_TOPK, M, N, K, num_sms, true);
    const int bn = wide_bn(EPI_TOPK, K);
    CUtensorMap ta, tb, tg;
    if (!wide_map(&ta, A, M, Kd, WM) || !wide_map(&tb, B, N, Kd, p.pair ? bn / 2 : bn))
        return cudaErrorInvalidValue;
    // G = A . W_H^T: inside this launch when it fits on the short last vocabulary
    // range (one 256-column tile, and that range has fewer tiles than the others),
    // else as a store launch of its own after it
    const bool want_g = W_H && G && r > 0;
    const int last_rng = p.n_nt - (p.n_groups - 1) * p.tiles_per_cta;
    const bool fold_g = want_g && r <= 256 && last_rng < p.tiles_per_cta;
    tg = tb;
    if (fold_g && !wide_map(&tg, W_H, r, Kd, p.pair ? bn / 2 : bn)) return cudaErrorInvalidValue;
    WideArgs a{};
    a.M = int(M); a.N = int(N); a.Kd = int(Kd);
    a.n_mt = p.n_mt;
    a.n_nt = p.n_nt;
    a.tiles_per_cta = p.tiles_per_cta;
    const int n_groups = p.n_groups;
    a.m_major = 0;
    a.nstages = p.nstages;
    a.kbox = 1;
    a.K = K;
    a.part_v = static_cast<float*>(ws);
    a.part_id = reinterpret_cast<int*>(a.part_v + size_t(n_groups) * M * K);
    a.thr_g = reinterpret_cast<unsigned*>(a.part_id + size_t(n_groups) * M * K);
    a.dev_status = dev_status;
    a.zero_words = zero_words;
    a.n_zero = n_zero;
    if (fold_g) {
        a.n_gt = 1;
        a.g_grp0 = n_groups - 1;
        a.g_out = G;
        a.g_n = int(r);
    }
    cudaError_t e = cudaMemsetAsync(a.thr_g, 0, size_t(M) * 4, stream);
    if (e != cudaSuccess) return e;
    e = launch_plan<EPI_TOPK>(p, ta, tb, tg, a, stream);
    if (e != cudaSuccess) return e;
    if (want_g && !fold_g) {
        e = wide_store_launch(A, M, W_H, r, Kd, G, r, r, G, r, dev_status, stream);
        if (e != cudaSuccess) return e;
    }
    if (parts_out) {  // the caller folds the per-range lists itself
        *parts_out = TopkParts{a.part_v, a.part_id, n_groups};
        return cudaSuccess;
    }
    return topk_merge_sorted_launch(a.part_v, a.part_id, n_groups, M, K, ids, vals, stream, LogitMap{},
                                    Refine{A, B, Kd});
}

}  // namespace df2
