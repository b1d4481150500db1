// Unary logits + top-K + hidden projection on the tensor cores (tcgen05, TMEM,
// TMA), for few positions per call (the batch-1 / small-batch latency case).
//
// U[p, v] = h[p, :] . W_lm[v, :] over the full vocabulary ("DFlash2", vLLM
// Speculators guide, "Candidate Selector"); top-K per position; G = h W_H^T
// (verl-SpeCo PR #62, "What DFlash2 adds": H projects the hidden state).
//
// At this size the head is a stream of the whole LM head from HBM, so the
// kernel is built around that stream:
//   * the vocabulary is cut into tiles of at most 128 rows (plus ceil(r/128)
//     tiles of W_H); one persistent CTA per SM walks tiles blockIdx.x,
//     +gridDim.x, ...  The first n_hi vocabulary tiles have bm_hi rows and the
//     rest bm_lo (both multiples of 8), chosen on the host so that every CTA
//     walks the same number of tiles and the busiest streams as few rows as it
//     can; a short tile's spare MMA rows hold stale shared memory and are never
//     read out;
//   * warp 0 (one lane) streams each tile with TMA in stages of `kbox` [128 x 64]
//     bf16 boxes (so every W row contributes 64*kbox contiguous elements per
//     stage), 128-byte swizzled, evict-first in L2, into a ring of `nstages`
//     slots, together with the matching [N x 64] boxes of h (rows past P read 0);
//   * two issuing lanes (warps 1 and 6) issue tcgen05.mma M=128 (vocab rows) x N
//     (positions, 16 or 32) x K=16 into TMEM, alternating k-steps, each into its
//     own partial accumulator (at N = 16 an MMA is a few cycles of tensor work,
//     while this loop's per-MMA work in the issuing lane -- descriptors, the
//     accumulator choice -- came to ~150 cycles, as long as the W stream; two
//     lanes halve it); two tile accumulators alternate so the next tile's MMAs
//     overlap the epilogue of this one;
//   * warps 2-5 read the accumulator (warp w owns TMEM lanes 32*(w%4)..+31, i.e.
//     32 vocab rows) and keep, per position, a top-K list in registers across
//     their 32 lanes (topk_warp.cuh): a ballot against the list's K-th entry
//     drops a tile's 32 candidates unless one of them enters the list, so after
//     the first tiles almost every tile costs one compare per position; W_H
//     tiles store G instead.
// The logits never reach global memory.  At the end the four warps' lists of a
// position are folded into one, written to the workspace in rank order, and
// topk_merge_sorted_kernel folds the CTAs' lists into the final top-K.
#include <cudaTypedefs.h>

#include "common.cuh"
#include "head_tc.h"
#include "kernels.h"
#include "tc_ptx.cuh"
#include "topk_warp.cuh"

namespace df2 {

namespace {

constexpr int BM = 128;          // vocab rows per tile (MMA M)
constexpr int BK = 64;           // K elements per stage (one 128-byte swizzle row)
constexpr int kEpiWarps = 4;
constexpr int kIssuers = 2;                        // MMA-issuing lanes: warps 1 and kIssuerWarp2
constexpr int kIssuerWarp2 = 2 + kEpiWarps;
constexpr int kThreads = 64 + 32 * kEpiWarps + 32;
constexpr uint32_t kWBytes = BM * BK * 2;
constexpr int kMaxK = 64;
constexpr int kMaxStages = 16;

struct SmemLayout {
    uint32_t w_off, h_off, bar_off, misc_off, xch_off, total, stage_w, stage_h;
};

// xch: the four epilogue warps' lists, exchanged through shared memory at the
// end.  It aliases the start of the W stage ring: the epilogue only uses it after
// the last tile's accumulator is complete, i.e. after every MMA has read its
// operands and every TMA load has landed.
__host__ __device__ inline SmemLayout smem_layout(int N, int R, int nstages, int kbox) {
    SmemLayout L;
    L.stage_w = uint32_t(kbox) * kWBytes;
    L.stage_h = uint32_t(kbox) * uint32_t(N) * BK * 2;
    L.w_off = 0;
    L.h_off = L.w_off + uint32_t(nstages) * L.stage_w;
    L.bar_off = L.h_off + uint32_t(nstages) * L.stage_h;               // 1024-aligned
    L.misc_off = L.bar_off + uint32_t(2 * nstages + 6) * 8;
    L.xch_off = 0;
    const uint32_t xch_bytes = uint32_t(kEpiWarps * N * R * 32) * 8;
    const uint32_t end = L.misc_off + 16;
    L.total = end > xch_bytes ? end : xch_bytes;
    return L;
}

template <int N, int R>
__global__ void __launch_bounds__(kThreads, 1)
head_skinny_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_w2,
                   const __grid_constant__ CUtensorMap tm_h, const __grid_constant__ CUtensorMap tm_wh, int P,
                   int D, int V, int K, int r, int n_vtiles, int n_hi, int bm_hi, int bm_lo, int n_tiles,
                   int nstages, int kbox, int pf_stages, int nacc,
                   float* __restrict__ part_v, int* __restrict__ part_id, float* __restrict__ G,
                   int32_t* __restrict__ dev_status, int stall_stage, unsigned* __restrict__ zero_words,
                   int n_zero) {
    // TMEM: two tile buffers (the epilogue drains one while the MMAs fill the
    // other), each holding nacc partial accumulators of N columns.  Successive
    // k-steps of a tile rotate over the partial accumulators; partial a belongs to
    // issuer a % kIssuers, so the issuers never write the same accumulator; the
    // epilogue adds the partials.
    const uint32_t buf_cols = uint32_t(nacc) * N;
    uint32_t tmem_cols = 32;
    while (tmem_cols < 2 * buf_cols) tmem_cols *= 2;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const SmemLayout L = smem_layout(N, R, nstages, kbox);
    uint8_t* sW = smem + L.w_off;
    uint8_t* sH = smem + L.h_off;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bar_off);
    uint64_t* empty = full + nstages;
    uint64_t* tfull = empty + nstages;
    uint64_t* tempty = tfull + 2;
    uint64_t* mma_done = tempty + 2;  // [kIssuers]
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + L.misc_off);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L.misc_off + 4);
    float* xch_v = reinterpret_cast<float*>(smem + L.xch_off);                 // [4][N][R*32]
    int* xch_id = reinterpret_cast<int*>(xch_v + kEpiWarps * N * R * 32);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nbox = (D + BK - 1) / BK;            // 64-wide boxes along D
    // counters the kernel after this one expects to start at zero
    if (blockIdx.x == 0)
        for (int i = threadIdx.x; i < n_zero; i += blockDim.x) zero_words[i] = 0u;
    const int nk = (nbox + kbox - 1) / kbox;       // stages per tile
    const uint32_t h_box_bytes = uint32_t(N) * BK * 2;
    // tile t: its first row, its row count, and the tensor map whose box it is
    auto tile_row0 = [&](int t) {
        if (t >= n_vtiles) return (t - n_vtiles) * BM;
        return t < n_hi ? t * bm_hi : n_hi * bm_hi + (t - n_hi) * bm_lo;
    };
    auto tile_rows = [&](int t) { return t >= n_vtiles ? BM : (t < n_hi ? bm_hi : bm_lo); };
    auto tile_map = [&](int t) { return t >= n_vtiles ? &tm_wh : (t < n_hi ? &tm_w : &tm_w2); };

    if (threadIdx.x == 0) {
        for (int s = 0; s < nstages; ++s) {
            tc::mbar_init(&full[s], 1);
            tc::mbar_init(&empty[s], kIssuers);  // a commit from each issuer
        }
        for (int b = 0; b < 2; ++b) {
            tc::mbar_init(&tfull[b], kIssuers);
            tc::mbar_init(&tempty[b], kEpiWarps);
        }
        for (int i = 0; i < kIssuers; ++i) tc::mbar_init(&mma_done[i], 1);
        abort_flag[0] = 0;
        tc::fence_mbar_init();
    }
    if (warp == 1) {
        tc::tmem_alloc(tmem_holder, tmem_cols);
        tc::tmem_relinquish();
    }
    if (warp == 0 && lane == 0) {
        tc::prefetch_tmap(&tm_w);
        if (n_hi < n_vtiles) tc::prefetch_tmap(&tm_w2);
        tc::prefetch_tmap(&tm_h);
        if (n_tiles > n_vtiles) tc::prefetch_tmap(&tm_wh);
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem_base = *tmem_holder;

    if (warp == 0) {
        if (lane == 0) {
            // ---------------------------------------------------- TMA producer
            const uint64_t pol_w = tc::l2_policy_evict_first();
            const uint64_t pol_h = tc::l2_policy_evict_last();
            const int my_tiles = n_tiles > int(blockIdx.x) ? (n_tiles - 1 - int(blockIdx.x)) / int(gridDim.x) + 1 : 0;
            const int total = my_tiles * nk;
            // L2 prefetch of the first pf_stages stages of this CTA's stream
            for (int g = 0; g < pf_stages && g < total; ++g) {
                const int t = int(blockIdx.x) + (g / nk) * int(gridDim.x);
                const int kb = g % nk;
                for (int j = 0; j < kbox && kb * kbox + j < nbox; ++j)
                    tc::tma_prefetch_2d(tile_map(t), (kb * kbox + j) * BK, tile_row0(t));
            }
            int stage = 0;
            uint32_t phase = 0;
            int8_t armed[kMaxStages];
            for (int s = 0; s < kMaxStages; ++s) armed[s] = -1;
            bool ok = true;
            for (int g = 0; g < total && ok; ++g) {
                const int t = int(blockIdx.x) + (g / nk) * int(gridDim.x);
                const int kb = g % nk;
                const CUtensorMap* mw = tile_map(t);
                const int row0 = tile_row0(t);
                const uint32_t w_box_bytes = uint32_t(tile_rows(t)) * BK * 2;
                const int nb = min(kbox, nbox - kb * kbox);
                if (!tc::mbar_wait(&empty[stage], phase ^ 1, abort_flag)) { ok = false; break; }
                tc::mbar_arrive_expect_tx(&full[stage], uint32_t(nb) * (w_box_bytes + h_box_bytes));
                // self-test only: a stage whose copies are never issued, so the
                // consumer's bounded wait must give up and report a timeout
                for (int j = 0; j < nb && g != stall_stage; ++j) {
                    tc::tma_load_2d(sW + size_t(stage) * L.stage_w + size_t(j) * kWBytes, mw, &full[stage],
                                    (kb * kbox + j) * BK, row0, pol_w);
                    tc::tma_load_2d(sH + size_t(stage) * L.stage_h + size_t(j) * h_box_bytes, &tm_h,
                                    &full[stage], (kb * kbox + j) * BK, 0, pol_h);
                }
                armed[stage] = int8_t(phase);
                if (++stage == nstages) { stage = 0; phase ^= 1; }
                const int gp = g + pf_stages;
                if (pf_stages > 0 && gp < total) {
                    const int tp = int(blockIdx.x) + (gp / nk) * int(gridDim.x);
                    const int kbp = gp % nk;
                    for (int j = 0; j < kbox && kbp * kbox + j < nbox; ++j)
                        tc::tma_prefetch_2d(tile_map(tp), (kbp * kbox + j) * BK, tile_row0(tp));
                }
            }
            if (!ok) {
                // drain: every copy this thread started lands before the CTA exits
                volatile int never = 0;
                for (int s = 0; s < nstages; ++s)
                    if (armed[s] >= 0) tc::mbar_wait(&full[s], uint32_t(armed[s]), &never);
            }
        }
    } else if (warp == 1 || warp == kIssuerWarp2) {
        if (lane == 0) {
            // ----------------------------------------------------- MMA issuers
            const int who = warp == 1 ? 0 : 1;
            constexpr uint32_t idesc = tc::idesc_bf16_f32(BM, N);
            int stage = 0;
            uint32_t phase = 0;
            int it = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < n_tiles && ok; t += gridDim.x, ++it) {
                const int b = it & 1;
                const uint32_t tph = (it >> 1) & 1;
                if (!tc::mbar_wait(&tempty[b], tph ^ 1, abort_flag)) break;
                tc::fence_after_sync();
                const uint32_t d_tmem = tmem_base + uint32_t(b) * buf_cols;
                int ks = 0;  // k-step (16 elements of D) within the tile
                for (int kb = 0; kb < nk; ++kb) {
                    if (!tc::mbar_wait(&full[stage], phase, abort_flag)) { ok = false; break; }
                    tc::fence_after_sync();
                    const int nb = min(kbox, nbox - kb * kbox);
                    for (int j = 0; j < nb; ++j) {
                        const uint32_t a0 = tc::smem_u32(sW + size_t(stage) * L.stage_w + size_t(j) * kWBytes);
                        const uint32_t b0 = tc::smem_u32(sH + size_t(stage) * L.stage_h + size_t(j) * h_box_bytes);
#pragma unroll
                        for (int k = 0; k < BK / 16; ++k, ++ks) {
                            const int a = ks % nacc;
                            if (a % kIssuers != who) continue;
                            tc::mma_bf16(d_tmem + uint32_t(a * N), tc::sw128_kmajor_desc(a0 + 32 * k),
                                         tc::sw128_kmajor_desc(b0 + 32 * k), idesc,
                                         ks >= nacc ? 1u : 0u);
                        }
                    }
                    tc::mma_commit(&empty[stage]);
                    if (++stage == nstages) { stage = 0; phase ^= 1; }
                }
                if (ok) tc::mma_commit(&tfull[b]);
            }
            // every MMA this thread issued is complete before TMEM is released
            tc::mma_commit(&mma_done[who]);
            volatile int never = 0;
            tc::mbar_wait(&mma_done[who], 0, &never);
        }
    } else if (warp < 2 + kEpiWarps) {
        // ---------------------------------------------------------- epilogue
        const int e = warp - 2;
        const int quarter = warp & 3;
        const int nacc_used = min(nacc, 4 * nbox);  // partials a tile actually wrote
        wtk::List<R> lists[N];
#pragma unroll
        for (int p = 0; p < N; ++p) lists[p].clear();
        int it = 0;
        for (int t = blockIdx.x; t < n_tiles; t += gridDim.x, ++it) {
            const int b = it & 1;
            const uint32_t tph = (it >> 1) & 1;
            const bool got = tc::mbar_wait(&tfull[b], tph, abort_flag);
            if (!__all_sync(kFull, got)) break;
            tc::fence_after_sync();
            float acc[N];
            const uint32_t taddr = tmem_base + (uint32_t(quarter * 32) << 16) + uint32_t(b) * buf_cols;
            tc::tmem_ld16(taddr, acc);
            if constexpr (N == 32) tc::tmem_ld16(taddr + 16, acc + 16);
            for (int a = 1; a < nacc_used; ++a) {
                float part[N];
                tc::tmem_ld16(taddr + uint32_t(a * N), part);
                if constexpr (N == 32) tc::tmem_ld16(taddr + uint32_t(a * N) + 16, part + 16);
#pragma unroll
                for (int p = 0; p < N; ++p) acc[p] += part[p];
            }
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&tempty[b]);

            const bool is_wh = t >= n_vtiles;
            const int lr = quarter * 32 + lane;  // the tile's row of this lane
            const int row = tile_row0(t) + lr;
            if (is_wh) {
                if (row < r) {
#pragma unroll
                    for (int p = 0; p < N; ++p)
                        if (p < P) G[size_t(p) * r + row] = acc[p];
                }
            } else {
                const bool valid = lr < tile_rows(t) && row < V;
#pragma unroll
                for (int p = 0; p < N; ++p)
                    if (p < P) lists[p].offer(acc[p], valid ? row : wtk::kEmptyId, K, lane);
            }
        }
        // the four warps' lists of a position -> one list -> workspace (partial blockIdx.x)
#pragma unroll
        for (int p = 0; p < N; ++p) {
            if (p < P) {
#pragma unroll
                for (int rr = 0; rr < R; ++rr) {
                    const int at = ((e * N + p) * R + rr) * 32 + lane;
                    xch_v[at] = lists[p].v[rr];
                    xch_id[at] = lists[p].id[rr];
                }
            }
        }
        tc::named_barrier(1, 32 * kEpiWarps);
        for (int p = e; p < P; p += kEpiWarps) {
            wtk::List<R> m;
#pragma unroll
            for (int rr = 0; rr < R; ++rr) {
                m.v[rr] = xch_v[((0 * N + p) * R + rr) * 32 + lane];
                m.id[rr] = xch_id[((0 * N + p) * R + rr) * 32 + lane];
            }
            for (int src = 1; src < kEpiWarps; ++src) {
#pragma unroll
                for (int rr = 0; rr < R; ++rr) {
                    const int at = ((src * N + p) * R + rr) * 32 + lane;
                    m.offer_sorted(xch_v[at], xch_id[at], K, lane);
                }
            }
            const size_t base = (size_t(blockIdx.x) * P + p) * K;
#pragma unroll
            for (int rr = 0; rr < R; ++rr) {
                const int k = rr * 32 + lane;
                if (k < K) {
                    part_v[base + k] = m.id[rr] != wtk::kEmptyId ? m.v[rr] : -INFINITY;
                    part_id[base + k] = m.id[rr] != wtk::kEmptyId ? m.id[rr] : -1;
                }
            }
        }
    }

    tc::fence_before_sync();
    __syncthreads();
    if (threadIdx.x == 0 && *abort_flag && dev_status) atomicOr(dev_status, DF2_STATUS_WAIT_TIMEOUT);
    if (warp == 1) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem_base, tmem_cols);
    }
}

// ---------------------------------------------------------------- host --

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

// Row-major bf16 [rows, cols] tensor, box {64 cols, box_rows}, 128-byte swizzle.
bool make_map(CUtensorMap* m, const void* base, int64_t rows, int64_t cols, int box_rows) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {cuuint64_t(cols), cuuint64_t(rows)};
    cuuint64_t strides[1] = {cuuint64_t(cols) * 2};
    cuuint32_t box[2] = {cuuint32_t(BK), cuuint32_t(box_rows)};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
                    estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

int pick_n(int64_t P) { return P <= 16 ? 16 : 32; }

#ifndef DF2_HEAD_KBOX
#define DF2_HEAD_KBOX 4  // 64-wide boxes per pipeline stage: 512 contiguous bytes per W row
#endif
#ifndef DF2_HEAD_PF
#define DF2_HEAD_PF 0    // stages prefetched into L2 ahead of the TMA loads
#endif
#ifndef DF2_HEAD_NACC
#define DF2_HEAD_NACC 2  // partial accumulators per tile: a multiple of the issuers
#endif
static_assert(DF2_HEAD_NACC % kIssuers == 0, "every issuer owns whole partial accumulators");

struct Plan {
    int N, R, nstages, kbox;
};

Plan pick_plan(int64_t P, int K) {
    Plan pl{pick_n(P), K <= 32 ? 1 : 2, 0, DF2_HEAD_KBOX};
    const int budget = 227 * 1024 - 1024;
    for (int kb = pl.kbox; kb >= 1; kb /= 2) {
        for (int s = kMaxStages; s >= 2; --s)
            if (int(smem_layout(pl.N, pl.R, s, kb).total) <= budget && s * kb <= 4 * kMaxStages) {
                if (s * kb >= 6 || kb == 1) { pl.nstages = s; pl.kbox = kb; return pl; }
                break;
            }
    }
    return pl;
}

// The vocabulary tiles: at 128 rows each CTA would walk `per` tiles (W_H's
// included), and that stays so with n_vtiles = per * grid - n_wh tiles of the two
// multiples of 8 around V / n_vtiles.  Round-robin then deals every CTA nearly the
// same number of long tiles (V 151936, 152 CTAs: 782 of 128 rows, 432 of 120, so
// the busiest CTA streams 1008 rows instead of 1024).
struct VTiling {
    int n_vtiles, n_hi, bm_hi, bm_lo;
};
VTiling v_tiling(int64_t V, int n_wh, int grid) {
    const int64_t t128 = (V + BM - 1) / BM;
    const VTiling uniform{int(t128), int(t128), BM, BM};
    const int64_t per = (t128 + n_wh + grid - 1) / grid;
    const int64_t slots = per * grid - n_wh;
    if (slots < t128) return uniform;
    const int64_t lo = V / slots / 8 * 8;
    if (lo < 8 || lo >= BM) return uniform;
    const int64_t n_hi = (V - slots * lo + 7) / 8;  // tiles of lo + 8 rows; the rest lo
    if (n_hi < 0 || n_hi > slots) return uniform;
    return VTiling{int(slots), int(n_hi), int(lo + 8), int(lo)};
}

}  // namespace

bool head_tc_supported(int64_t P, int64_t D, int64_t V, int K) {
    // register lists: N positions x R rows per epilogue lane; 32 x 2 would not fit
    return P >= 1 && P <= 32 && K <= kMaxK && (P <= 16 || K <= 32) && D % 8 == 0 &&
           D <= (int64_t(1) << 30) && V <= INT32_MAX && pick_plan(P, K).nstages >= 2;
}

size_t head_tc_workspace(int64_t P, int64_t D, int64_t V, int K, int num_sms) {
    (void)D;
    const int64_t n_tiles = (V + BM - 1) / BM;
    const int64_t grid = n_tiles < num_sms ? n_tiles : num_sms;
    return size_t(grid) * size_t(P) * size_t(K) * 8;
}

int head_tc_launch(const uint16_t* h, int64_t P, int64_t D, const uint16_t* W, int64_t V, int K,
                   const uint16_t* W_H, int r, float* G, int32_t* ids, float* vals, void* ws,
                   int32_t* dev_status, int num_sms, cudaStream_t stream, int stall_stage,
                   TopkParts* parts_out, unsigned* zero_words, int n_zero) {
    const Plan pl = pick_plan(P, K);
    const int N = pl.N;
    const bool has_wh = W_H != nullptr;
    const int n_v128 = int((V + BM - 1) / BM);
    const int grid = n_v128 < num_sms ? n_v128 : num_sms;
    const int n_wh = has_wh ? (r + BM - 1) / BM : 0;
    const VTiling vt = v_tiling(V, n_wh, grid);
    CUtensorMap tm_w, tm_w2, tm_h, tm_wh;
    if (!make_map(&tm_w, W, V, D, vt.bm_hi) || !make_map(&tm_h, h, P, D, N)) return DF2_ERR_CUDA;
    if (vt.n_hi < vt.n_vtiles) {
        if (!make_map(&tm_w2, W, V, D, vt.bm_lo)) return DF2_ERR_CUDA;
    } else {
        tm_w2 = tm_w;
    }
    if (has_wh) {
        if (!make_map(&tm_wh, W_H, r, D, BM)) return DF2_ERR_CUDA;
    } else {
        tm_wh = tm_w;
    }
    const int n_vtiles = vt.n_vtiles;
    const int n_tiles = n_vtiles + n_wh;
    const size_t parts = size_t(grid);
    float* part_v = static_cast<float*>(ws);
    int* part_id = reinterpret_cast<int*>(part_v + parts * P * K);
    const size_t smem = smem_layout(N, pl.R, pl.nstages, pl.kbox).total + 1024;
    cudaError_t e = cudaSuccess;
#define DF2_HEAD(NV, RV)                                                                          \
    do {                                                                                          \
        e = cudaFuncSetAttribute(head_skinny_kernel<NV, RV>,                                      \
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));         \
        if (e != cudaSuccess) return DF2_ERR_CUDA;                                                \
        head_skinny_kernel<NV, RV><<<grid, kThreads, smem, stream>>>(                             \
            tm_w, tm_w2, tm_h, tm_wh, int(P), int(D), int(V), K, r, n_vtiles, vt.n_hi, vt.bm_hi,   \
            vt.bm_lo, n_tiles, pl.nstages,                                                        \
            pl.kbox, DF2_HEAD_PF, DF2_HEAD_NACC, part_v, part_id, G, dev_status, stall_stage,     \
            zero_words, n_zero);                                                                  \
    } while (0)
    if (N == 16 && pl.R == 1) DF2_HEAD(16, 1);
    else if (N == 16) DF2_HEAD(16, 2);
    else DF2_HEAD(32, 1);
#undef DF2_HEAD
    note_launch();
    if (cudaGetLastError() != cudaSuccess) return DF2_ERR_CUDA;
    if (parts_out) {  // the caller folds the per-CTA lists itself
        *parts_out = TopkParts{part_v, part_id, int(parts)};
        return DF2_OK;
    }
    e = topk_merge_sorted_launch(part_v, part_id, int(parts), P, K, ids, vals, stream, LogitMap{},
                                 Refine{h, W, D});
    return e == cudaSuccess ? DF2_OK : DF2_ERR_CUDA;
}

}  // namespace df2
