// Candidate selector: greedy walk and teacher-forced pair scores.
//
// Pair score S_t(a, b) = U_t(b) + < A(a) (.) H(h_t), B(b) > (verl-SpeCo PR #62,
// "What DFlash2 adds"; "DFlash 2 Explanation", "Problem 1").  The walk starts at
// the anchor and feeds each position's best successor in as the next
// predecessor (vLLM Speculators "DFlash2" guide, "Candidate Selector"); the
// teacher-forced scorer takes the predecessor as given (PR #62, "Selector
// training objective").
//
// The walk runs one CTA per request with its gathers staged in shared memory
// (walk_request_cta, selector_dev.cuh) when they fit, else one warp per request;
// the teacher-forced scores run one warp per (row, group of 8 candidates).  Lane
// l owns rank elements [8l, 8l+8) of every 256-wide chunk: the gate
// q = A[a] (.) G_t is formed once per position in registers, each candidate's B
// row is read with one 16-byte load per lane per chunk, and a shuffle tree sums
// the lanes.  The warp walk's candidate loop is unrolled by 4 so that four B-row
// gathers are in flight.
#include "common.cuh"
#include "kernels.h"
#include "selector_dev.cuh"

namespace df2 {

namespace {

using namespace sel;

constexpr int kWarpsPerBlock = 4;

// Scores of candidates [j0, j0+4) of one row against gate q; ids are in range.
template <int NCH>
__device__ __forceinline__ void score4(const int32_t* __restrict__ ids_row,
                                       const float* __restrict__ vals_row, int K, int j0,
                                       const uint16_t* __restrict__ Bc, int r, int lane,
                                       const float q[NCH][8], float s[4], int b[4]) {
    float part[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        b[u] = (j0 + u < K) ? __ldg(ids_row + j0 + u) : 0;
        part[u] = (j0 + u < K) ? dot_lane<NCH>(Bc, b[u], r, lane, q) : 0.f;
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const float d = warp_sum(part[u]);
        s[u] = (j0 + u < K) ? __ldg(vals_row + j0 + u) + d : -INFINITY;
    }
}

template <int NCH>
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
walk_kernel(const int32_t* __restrict__ anchors, int R, int B, const int32_t* __restrict__ ids,
            const float* __restrict__ vals, const float* __restrict__ G,
            const uint16_t* __restrict__ A, const uint16_t* __restrict__ Bc, int64_t V, int K, int r,
            int32_t* __restrict__ path, float* __restrict__ path_scores,
            int32_t* __restrict__ dev_status) {
    const int lane = threadIdx.x & 31;
    const int q = blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
    if (q >= R) return;
    const int T = B - 1;

    int32_t a = __ldg(anchors + q);
    bool ok = a >= 0 && a < V;
    for (int64_t e = lane; e < int64_t(T) * K; e += 32) {
        const int32_t b = __ldg(ids + (int64_t(q) * B + 1) * K + e);
        ok = ok && b >= 0 && b < V;
    }
    if (!__all_sync(kFull, ok)) {
        for (int t = lane; t < T; t += 32) {
            path[int64_t(q) * T + t] = -1;
            path_scores[int64_t(q) * T + t] = __int_as_float(0x7fc00000);
        }
        if (lane == 0 && dev_status) atomicOr(dev_status, DF2_STATUS_ID_OUT_OF_RANGE);
        return;
    }

    for (int t = 1; t < B; ++t) {
        const int64_t row = int64_t(q) * B + t;
        float qv[NCH][8];
        load_gate<NCH>(A, a, r, G + row * r, lane, qv);
        float best = -INFINITY;
        int best_id = -1;
        for (int j0 = 0; j0 < K; j0 += 4) {
            float s[4];
            int b[4];
            score4<NCH>(ids + row * K, vals + row * K, K, j0, Bc, r, lane, qv, s, b);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                if (j0 + u < K && (best_id < 0 || ranks_before(s[u], b[u], best, best_id))) {
                    best = s[u];
                    best_id = b[u];
                }
            }
        }
        if (lane == 0) {
            path[int64_t(q) * T + (t - 1)] = best_id;
            path_scores[int64_t(q) * T + (t - 1)] = best;
        }
        a = best_id;
    }
}

// One warp per (row, group of kPairGroup candidates): the gate and the group's
// B rows are independent loads, so a warp waits for about two memory latencies.
constexpr int kPairGroup = 8;

template <int NCH>
__global__ void __launch_bounds__(256)
pair_scores_kernel(const int32_t* __restrict__ pred, int64_t P, const int32_t* __restrict__ ids,
                   const float* __restrict__ vals, const float* __restrict__ G,
                   const uint16_t* __restrict__ A, const uint16_t* __restrict__ Bc, int64_t V, int K,
                   int r, float* __restrict__ scores, int32_t* __restrict__ dev_status) {
    const int lane = threadIdx.x & 31;
    const int ngroups = (K + kPairGroup - 1) / kPairGroup;
    const int64_t w = int64_t(blockIdx.x) * 8 + (threadIdx.x >> 5);
    if (w >= P * ngroups) return;
    const int64_t p = w / ngroups;
    const int j0 = int(w - p * ngroups) * kPairGroup;
    const float nan = __int_as_float(0x7fc00000);
    const int32_t a = __ldg(pred + p);
    bool bad = false;
    if (a < 0 || a >= V) {
        if (lane < kPairGroup && j0 + lane < K) scores[p * K + j0 + lane] = nan;
        bad = true;
    } else {
        float qv[NCH][8];
        load_gate<NCH>(A, a, r, G + p * r, lane, qv);
        float part[kPairGroup];
        int32_t b[kPairGroup];
        bool inr[kPairGroup];
#pragma unroll
        for (int u = 0; u < kPairGroup; ++u) {
            b[u] = (j0 + u < K) ? __ldg(ids + p * K + j0 + u) : 0;
            inr[u] = b[u] >= 0 && b[u] < V;
            part[u] = (j0 + u < K && inr[u]) ? dot_lane<NCH>(Bc, b[u], r, lane, qv) : 0.f;
        }
#pragma unroll
        for (int u = 0; u < kPairGroup; ++u) {
            const float d = warp_sum(part[u]);
            if (j0 + u < K && lane == 0)
                scores[p * K + j0 + u] = inr[u] ? __ldg(vals + p * K + j0 + u) + d : nan;
            bad = bad || (j0 + u < K && !inr[u]);
        }
    }
    if (bad && lane == 0 && dev_status) atomicOr(dev_status, DF2_STATUS_ID_OUT_OF_RANGE);
}

template <int NCH>
__global__ void __launch_bounds__(kWalkThreads, 1)
walk_cta_kernel(const int32_t* __restrict__ anchors, int B, const int32_t* __restrict__ ids,
                const float* __restrict__ vals, const float* __restrict__ G,
                const uint16_t* __restrict__ A, const uint16_t* __restrict__ Bc, int64_t V, int K,
                int r, int32_t* __restrict__ path, float* __restrict__ path_scores,
                int32_t* __restrict__ dev_status) {
    extern __shared__ __align__(16) uint8_t smem[];
    walk_request_cta<NCH, false>(blockIdx.x, anchors, B, ids, vals, G, A, Bc, V, K, r, path, path_scores,
                                 dev_status, smem);
}

}  // namespace

cudaError_t walk_launch(const int32_t* anchors, int R, int B, const int32_t* ids, const float* vals,
                        const float* G, const uint16_t* A, const uint16_t* Bc, int64_t V, int K,
                        int r, int32_t* path, float* scores, int32_t* dev_status,
                        cudaStream_t stream) {
    const int nch = (r + 255) / 256;
    const size_t smem = walk_cta_smem(B, K, r);
    if (smem <= 200 * 1024) {
#define DF2_WALK_CTA(N)                                                                             \
    do {                                                                                            \
        cudaError_t e = cudaFuncSetAttribute(walk_cta_kernel<N>,                                    \
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)); \
        if (e != cudaSuccess) return e;                                                             \
        walk_cta_kernel<N><<<unsigned(R), kWalkThreads, smem, stream>>>(anchors, B, ids, vals, G, A,  \
                                                                        Bc, V, K, r, path, scores,   \
                                                                        dev_status);                 \
    } while (0)
        if (nch <= 1) DF2_WALK_CTA(1);
        else if (nch <= 2) DF2_WALK_CTA(2);
        else if (nch <= 4) DF2_WALK_CTA(4);
        else if (nch <= 8) DF2_WALK_CTA(8);
        else DF2_WALK_CTA(16);
#undef DF2_WALK_CTA
        note_launch();
        return cudaGetLastError();
    }
    const unsigned grid = unsigned((R + kWarpsPerBlock - 1) / kWarpsPerBlock);
#define DF2_WALK(N)                                                                            \
    walk_kernel<N><<<grid, kWarpsPerBlock * 32, 0, stream>>>(anchors, R, B, ids, vals, G, A,  \
                                                             Bc, V, K, r, path, scores,       \
                                                             dev_status)
    if (nch <= 1) DF2_WALK(1);
    else if (nch <= 2) DF2_WALK(2);
    else if (nch <= 4) DF2_WALK(4);
    else if (nch <= 8) DF2_WALK(8);
    else DF2_WALK(16);
#undef DF2_WALK
    note_launch();
    return cudaGetLastError();
}

cudaError_t pair_scores_launch(const int32_t* pred, int64_t P, const int32_t* ids,
                               const float* vals, const float* G, const uint16_t* A,
                               const uint16_t* Bc, int64_t V, int K, int r, float* scores,
                               int32_t* dev_status, cudaStream_t stream) {
    const int64_t warps = P * ((K + kPairGroup - 1) / kPairGroup);
    const unsigned grid = unsigned((warps + 7) / 8);
    const int nch = (r + 255) / 256;
#define DF2_PAIR(N)                                                                            \
    pair_scores_kernel<N><<<grid, 256, 0, stream>>>(pred, P, ids, vals, G, A, Bc, V, K, r,    \
                                                    scores, dev_status)
    if (nch <= 1) DF2_PAIR(1);
    else if (nch <= 2) DF2_PAIR(2);
    else if (nch <= 4) DF2_PAIR(4);
    else if (nch <= 8) DF2_PAIR(8);
    else DF2_PAIR(16);
#undef DF2_PAIR
    note_launch();
    return cudaGetLastError();
}

}  // namespace df2
