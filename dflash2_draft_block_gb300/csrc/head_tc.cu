// Unary logits + top-K + hidden projection on the tensor cores (tcgen05, TMEM,
// TMA), for few positions per call (the batch-1 / small-batch latency case).
//
// U[p, v] = h[p, :] . W_lm[v, :] over the full vocabulary ("DFlash2", vLLM
// Speculators guide, "Candidate Selector"); top-K per position; G = h W_H^T
// (verl-SpeCo PR #62, "What DFlash2 adds": H projects the hidden state).
//
// At this size the head is a stream of the whole LM head from HBM, so the
// kernel is built around that stream:
//   * the vocabulary is cut into 128-row tiles (plus ceil(r/128) tiles of W_H);
//     one persistent CTA per SM walks tiles blockIdx.x, +gridDim.x, ...
//   * warp 0 (one lane) streams [128 x 64] bf16 boxes of the tile with TMA,
//     128-byte swizzled, evict-first in L2, into a ring of `nstages` slots,
//     together with the matching [N x 64] box of h (rows past P read as zero);
//   * warp 1 (one lane) issues tcgen05.mma M=128 (vocab rows) x N (positions,
//     16 or 32) x K=16, accumulating the tile's logits in TMEM; the two TMEM
//     accumulators alternate so the next tile's MMAs overlap the epilogue;
//   * warps 2-5 read the accumulator (warp w owns TMEM lanes 32*(w%4)..+31,
//     i.e. 32 vocab rows) and fold each position's 32 logits into a per-warp
//     top-K list in shared memory (a ballot against the list's worst entry
//     rejects nearly everything once the list is full), or store G for W_H tiles.
// The logits never reach global memory.  Each epilogue warp's lists go to the
// workspace and topk_merge_kernel reduces them to the sorted top-K.
#include <cudaTypedefs.h>

#include "common.cuh"
#include "head_tc.h"
#include "kernels.h"
#include "tc_ptx.cuh"

namespace df2 {

namespace {

constexpr int BM = 128;          // vocab rows per tile (MMA M)
constexpr int BK = 64;           // K elements per stage (one 128-byte swizzle row)
constexpr int kEpiWarps = 4;
constexpr int kThreads = 64 + 32 * kEpiWarps;
constexpr uint32_t kWBytes = BM * BK * 2;
constexpr int kMaxK = 64;
constexpr int kMaxStages = 16;

// Top-K list state kept in shared memory; operated on by one warp.
struct ListState {
    int n;
    float wv;
    int wid;
    int wpos;
};

__device__ __forceinline__ void list_find_worst(ListState* st, const float* v, const int* id, int K,
                                                int lane) {
    float bv = 0.f;
    int bi = 0, bp = -1;
    for (int i = lane; i < K; i += 32) {
        const float vv = v[i];
        const int ii = id[i];
        if (bp < 0 || ranks_before(bv, bi, vv, ii)) { bv = vv; bi = ii; bp = i; }
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) {
        const float ov = __shfl_xor_sync(kFull, bv, o);
        const int oi = __shfl_xor_sync(kFull, bi, o);
        const int op = __shfl_xor_sync(kFull, bp, o);
        if (op >= 0 && (bp < 0 || ranks_before(bv, bi, ov, oi))) { bv = ov; bi = oi; bp = op; }
    }
    if (lane == 0) { st->wv = bv; st->wid = bi; st->wpos = bp; }
    __syncwarp();
}

// Offer one candidate per lane to the list.
__device__ __forceinline__ void list_offer(ListState* st, float* v, int* id, int K, bool valid,
                                           float cv, int cid, int lane) {
    int n = st->n;
    float wv = st->wv;
    int wid = st->wid;
    unsigned m = __ballot_sync(kFull, valid && (n < K || ranks_before(cv, cid, wv, wid)));
    while (m) {
        const int src = __ffs(m) - 1;
        m &= m - 1;
        const float sv = __shfl_sync(kFull, cv, src);
        const int si = __shfl_sync(kFull, cid, src);
        if (n < K) {
            if (lane == 0) { v[n] = sv; id[n] = si; st->n = n + 1; }
            ++n;
            __syncwarp();
            if (n == K) list_find_worst(st, v, id, K, lane);
        } else if (ranks_before(sv, si, wv, wid)) {
            if (lane == 0) { v[st->wpos] = sv; id[st->wpos] = si; }
            __syncwarp();
            list_find_worst(st, v, id, K, lane);
        }
        wv = st->wv;
        wid = st->wid;
    }
}

struct SmemLayout {
    uint32_t w_off, h_off, bar_off, misc_off, state_off, lv_off, lid_off, total;
};

__host__ __device__ inline SmemLayout smem_layout(int N, int K, int nstages) {
    SmemLayout L;
    const uint32_t h_bytes = uint32_t(N) * BK * 2;
    L.w_off = 0;
    L.h_off = L.w_off + uint32_t(nstages) * kWBytes;
    L.bar_off = L.h_off + uint32_t(nstages) * h_bytes;                 // 1024-aligned
    L.misc_off = L.bar_off + uint32_t(2 * nstages + 5) * 8;
    L.state_off = (L.misc_off + 16 + 15) / 16 * 16;
    L.lv_off = L.state_off + uint32_t(kEpiWarps * N) * sizeof(ListState);
    L.lid_off = L.lv_off + uint32_t(kEpiWarps * N * K) * 4;
    L.total = L.lid_off + uint32_t(kEpiWarps * N * K) * 4;
    return L;
}

template <int N>
__global__ void __launch_bounds__(kThreads, 1)
head_skinny_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_h,
                   const __grid_constant__ CUtensorMap tm_wh, int P, int D, int V, int K, int r,
                   int n_vtiles, int n_tiles, int nstages, float* __restrict__ part_v,
                   int* __restrict__ part_id, float* __restrict__ G, int32_t* __restrict__ dev_status) {
    constexpr uint32_t kHBytes = N * BK * 2;
    constexpr uint32_t kTmemCols = 2 * N;  // 32 or 64: two accumulators
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const SmemLayout L = smem_layout(N, K, nstages);
    uint8_t* sW = smem + L.w_off;
    uint8_t* sH = smem + L.h_off;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bar_off);
    uint64_t* empty = full + nstages;
    uint64_t* tfull = empty + nstages;
    uint64_t* tempty = tfull + 2;
    uint64_t* mma_done = tempty + 2;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + L.misc_off);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L.misc_off + 4);
    ListState* states = reinterpret_cast<ListState*>(smem + L.state_off);
    float* lv = reinterpret_cast<float*>(smem + L.lv_off);
    int* lid = reinterpret_cast<int*>(smem + L.lid_off);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nk = (D + BK - 1) / BK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < nstages; ++s) {
            tc::mbar_init(&full[s], 1);
            tc::mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            tc::mbar_init(&tfull[b], 1);
            tc::mbar_init(&tempty[b], kEpiWarps);
        }
        tc::mbar_init(mma_done, 1);
        *abort_flag = 0;
        tc::fence_mbar_init();
    }
    if (warp >= 2) {
        const int e = warp - 2;
        for (int i = lane; i < N; i += 32) {
            ListState* st = &states[e * N + i];
            st->n = 0; st->wv = -INFINITY; st->wid = INT_MAX; st->wpos = 0;
        }
    }
    if (warp == 1) {
        tc::tmem_alloc(tmem_holder, kTmemCols);
        tc::tmem_relinquish();
    }
    if (warp == 0 && lane == 0) {
        tc::prefetch_tmap(&tm_w);
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
            int stage = 0;
            uint32_t phase = 0;
            int8_t armed[kMaxStages];
            for (int s = 0; s < kMaxStages; ++s) armed[s] = -1;
            bool ok = true;
            for (int t = blockIdx.x; t < n_tiles && ok; t += gridDim.x) {
                const bool is_wh = t >= n_vtiles;
                const CUtensorMap* mw = is_wh ? &tm_wh : &tm_w;
                const int row0 = (is_wh ? t - n_vtiles : t) * BM;
                for (int kb = 0; kb < nk; ++kb) {
                    if (!tc::mbar_wait(&empty[stage], phase ^ 1, abort_flag)) { ok = false; break; }
                    tc::mbar_arrive_expect_tx(&full[stage], kWBytes + kHBytes);
                    tc::tma_load_2d(sW + size_t(stage) * kWBytes, mw, &full[stage], kb * BK, row0, pol_w);
                    tc::tma_load_2d(sH + size_t(stage) * kHBytes, &tm_h, &full[stage], kb * BK, 0, pol_h);
                    armed[stage] = int8_t(phase);
                    if (++stage == nstages) { stage = 0; phase ^= 1; }
                }
            }
            if (!ok) {
                // drain: every copy this thread started lands before the CTA exits
                volatile int never = 0;
                for (int s = 0; s < nstages; ++s)
                    if (armed[s] >= 0) tc::mbar_wait(&full[s], uint32_t(armed[s]), &never);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ------------------------------------------------------ MMA issuer
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
                const uint32_t d_tmem = tmem_base + uint32_t(b * N);
                for (int kb = 0; kb < nk; ++kb) {
                    if (!tc::mbar_wait(&full[stage], phase, abort_flag)) { ok = false; break; }
                    tc::fence_after_sync();
                    const uint32_t a0 = tc::smem_u32(sW + size_t(stage) * kWBytes);
                    const uint32_t b0 = tc::smem_u32(sH + size_t(stage) * kHBytes);
#pragma unroll
                    for (int k = 0; k < BK / 16; ++k)
                        tc::mma_bf16(d_tmem, tc::sw128_kmajor_desc(a0 + 32 * k),
                                     tc::sw128_kmajor_desc(b0 + 32 * k), idesc,
                                     (kb | k) != 0 ? 1u : 0u);
                    tc::mma_commit(&empty[stage]);
                    if (++stage == nstages) { stage = 0; phase ^= 1; }
                }
                if (ok) tc::mma_commit(&tfull[b]);
            }
            // every MMA this thread issued is complete before TMEM is released
            tc::mma_commit(mma_done);
            volatile int never = 0;
            tc::mbar_wait(mma_done, 0, &never);
        }
    } else {
        // ---------------------------------------------------------- epilogue
        const int e = warp - 2;
        const int quarter = warp & 3;
        int it = 0;
        for (int t = blockIdx.x; t < n_tiles; t += gridDim.x, ++it) {
            const int b = it & 1;
            const uint32_t tph = (it >> 1) & 1;
            const bool got = tc::mbar_wait(&tfull[b], tph, abort_flag);
            if (!__all_sync(kFull, got)) break;
            tc::fence_after_sync();
            float acc[N];
            const uint32_t taddr = tmem_base + (uint32_t(quarter * 32) << 16) + uint32_t(b * N);
            tc::tmem_ld16(taddr, acc);
            if constexpr (N == 32) tc::tmem_ld16(taddr + 16, acc + 16);
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&tempty[b]);

            const bool is_wh = t >= n_vtiles;
            const int row = (is_wh ? t - n_vtiles : t) * BM + quarter * 32 + lane;
            if (is_wh) {
                if (row < r) {
#pragma unroll
                    for (int p = 0; p < N; ++p)
                        if (p < P) G[size_t(p) * r + row] = acc[p];
                }
            } else {
                const bool valid = row < V;
#pragma unroll
                for (int p = 0; p < N; ++p) {
                    if (p < P) {
                        const int li = e * N + p;
                        list_offer(&states[li], lv + size_t(li) * K, lid + size_t(li) * K, K, valid,
                                   acc[p], row, lane);
                    }
                }
            }
        }
        // this warp's lists -> workspace partial (blockIdx.x * 4 + e)
        const size_t s = size_t(blockIdx.x) * kEpiWarps + e;
        for (int p = 0; p < P; ++p) {
            const int li = e * N + p;
            const int n = states[li].n;
            for (int k = lane; k < K; k += 32) {
                const size_t at = (s * P + p) * K + k;
                part_v[at] = k < n ? lv[size_t(li) * K + k] : -INFINITY;
                part_id[at] = k < n ? lid[size_t(li) * K + k] : -1;
            }
        }
    }

    tc::fence_before_sync();
    __syncthreads();
    if (threadIdx.x == 0 && *abort_flag && dev_status) atomicOr(dev_status, DF2_STATUS_WAIT_TIMEOUT);
    if (warp == 1) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem_base, kTmemCols);
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

int pick_stages(int N, int K) {
    const int budget = 227 * 1024 - 1024;
    for (int s = kMaxStages; s >= 2; --s)
        if (int(smem_layout(N, K, s).total) <= budget) return s;
    return 0;
}

}  // namespace

bool head_tc_supported(int64_t P, int64_t D, int64_t V, int K) {
    return P >= 1 && P <= 32 && K <= kMaxK && D % 8 == 0 && D <= (int64_t(1) << 30) &&
           V <= INT32_MAX && pick_stages(pick_n(P), K) >= 2;
}

size_t head_tc_workspace(int64_t P, int64_t D, int64_t V, int K, int num_sms) {
    (void)D;
    const int64_t n_tiles = (V + BM - 1) / BM;
    const int64_t grid = n_tiles < num_sms ? n_tiles : num_sms;
    return size_t(grid) * kEpiWarps * size_t(P) * size_t(K) * 8;
}

int head_tc_launch(const uint16_t* h, int64_t P, int64_t D, const uint16_t* W, int64_t V, int K,
                   const uint16_t* W_H, int r, float* G, int32_t* ids, float* vals, void* ws,
                   int32_t* dev_status, int num_sms, cudaStream_t stream) {
    const int N = pick_n(P);
    const int nstages = pick_stages(N, K);
    CUtensorMap tm_w, tm_h, tm_wh;
    if (!make_map(&tm_w, W, V, D, BM) || !make_map(&tm_h, h, P, D, N)) return DF2_ERR_CUDA;
    const bool has_wh = W_H != nullptr;
    if (has_wh) {
        if (!make_map(&tm_wh, W_H, r, D, BM)) return DF2_ERR_CUDA;
    } else {
        tm_wh = tm_w;
    }
    const int n_vtiles = int((V + BM - 1) / BM);
    const int n_tiles = n_vtiles + (has_wh ? (r + BM - 1) / BM : 0);
    const int grid = n_vtiles < num_sms ? n_vtiles : num_sms;
    const size_t parts = size_t(grid) * kEpiWarps;
    float* part_v = static_cast<float*>(ws);
    int* part_id = reinterpret_cast<int*>(part_v + parts * P * K);
    const size_t smem = smem_layout(N, K, nstages).total + 1024;
    cudaError_t e;
    if (N == 16) {
        e = cudaFuncSetAttribute(head_skinny_kernel<16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 int(smem));
        if (e != cudaSuccess) return DF2_ERR_CUDA;
        head_skinny_kernel<16><<<grid, kThreads, smem, stream>>>(
            tm_w, tm_h, tm_wh, int(P), int(D), int(V), K, r, n_vtiles, n_tiles, nstages, part_v,
            part_id, G, dev_status);
    } else {
        e = cudaFuncSetAttribute(head_skinny_kernel<32>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 int(smem));
        if (e != cudaSuccess) return DF2_ERR_CUDA;
        head_skinny_kernel<32><<<grid, kThreads, smem, stream>>>(
            tm_w, tm_h, tm_wh, int(P), int(D), int(V), K, r, n_vtiles, n_tiles, nstages, part_v,
            part_id, G, dev_status);
    }
    if (cudaGetLastError() != cudaSuccess) return DF2_ERR_CUDA;
    e = topk_merge_launch(part_v, part_id, int(parts), P, K, ids, vals, stream);
    return e == cudaSuccess ? DF2_OK : DF2_ERR_CUDA;
}

}  // namespace df2
