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

// Walk for requests whose gathers do not all fit in shared memory: one CTA per
// request streams the steps.  The B rows and G row of step t+1 do not depend on
// the choice at step t, so they are copied (cp.async, two buffers) while step t
// runs, and the A rows of step t's candidates -- the possible predecessors at
// step t+1 -- are prefetched into L2.  Warp w scores candidates w, w+8, ... with
// the lane slicing and shuffle tree of the other walk kernels (bit-identical
// scores); the warps' bests meet in shared memory.
constexpr int kStreamThreads = 256;
constexpr int kStreamWarps = kStreamThreads / 32;

__host__ __device__ inline size_t walk_stream_smem(int K, int r) {
    return 2 * (size_t(K) * r * 2 + size_t(r) * 4) + kStreamWarps * 16 + 64;
}

template <int NCH>
__global__ void __launch_bounds__(kStreamThreads, 1)
walk_stream_kernel(const int32_t* __restrict__ anchors, int B, const int32_t* __restrict__ ids,
                   const float* __restrict__ vals, const float* __restrict__ G,
                   const uint16_t* __restrict__ A, const uint16_t* __restrict__ Bc, int64_t V, int K,
                   int r, int32_t* __restrict__ path, float* __restrict__ path_scores,
                   int32_t* __restrict__ dev_status) {
    extern __shared__ __align__(16) uint8_t smem[];
    __shared__ int bad;
    const int T = B - 1;
    const int q = blockIdx.x;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const size_t stage_bytes = size_t(K) * r * 2 + size_t(r) * 4;
    float* wv = reinterpret_cast<float*>(smem + 2 * stage_bytes);  // [warps] best value
    int* wi = reinterpret_cast<int*>(wv + kStreamWarps);           // [warps] best id
    int* wj = wi + kStreamWarps;                                   // [warps] best column
    const int64_t row1 = int64_t(q) * B + 1;
    const int32_t a0 = __ldg(anchors + q);
    if (tid == 0) bad = (a0 < 0 || a0 >= V) ? 1 : 0;
    __syncthreads();
    for (int e = tid; e < T * K; e += kStreamThreads) {
        const int32_t b = __ldg(ids + row1 * K + e);
        if (b < 0 || b >= V) bad = 1;
    }
    __syncthreads();
    if (bad) {
        for (int t = tid; t < T; t += kStreamThreads) {
            path[int64_t(q) * T + t] = -1;
            path_scores[int64_t(q) * T + t] = __int_as_float(0x7fc00000);
        }
        if (tid == 0 && dev_status) atomicOr(dev_status, DF2_STATUS_ID_OUT_OF_RANGE);
        return;
    }
    const int cpr = r / 8;
    // stage t (1-based) into buffer t & 1: position t's B rows [K][r] and G row [r]
    auto issue = [&](int t) {
        uint16_t* Bs = reinterpret_cast<uint16_t*>(smem + (t & 1) * stage_bytes);
        float* Gs = reinterpret_cast<float*>(Bs + size_t(K) * r);
        const int64_t row = row1 + t - 1;
        for (int j = warp; j < K; j += kStreamWarps) {
            const uint16_t* src = Bc + int64_t(__ldg(ids + row * K + j)) * r;
            for (int c = lane; c < cpr; c += 32) cp_async16(Bs + size_t(j) * r + c * 8, src + c * 8);
        }
        for (int c = tid; c < r / 4; c += kStreamThreads) cp_async16(Gs + c * 4, G + row * r + c * 4);
        asm volatile("cp.async.commit_group;" ::: "memory");
        if (t < T) {  // position t's candidates are the predecessors at step t+1
            const int lines = (r * 2 + 127) / 128;
            for (int e = tid; e < K * lines; e += kStreamThreads)
                asm volatile("prefetch.global.L2 [%0];" ::"l"(A + int64_t(__ldg(ids + row * K + e / lines)) * r +
                                                              (e % lines) * 64));
        }
    };
    issue(1);
    int32_t a = a0;
    for (int t = 1; t <= T; ++t) {
        if (t < T) issue(t + 1);
        // the gate A[a] (.) G_t: this warp's lane slices (A from L2, G once staged)
        float af[NCH][8];
#pragma unroll
        for (int c = 0; c < NCH; ++c) {
            const int i0 = c * 256 + lane * 8;
            if (i0 < r) unpack8(__ldg(reinterpret_cast<const uint4*>(A + int64_t(a) * r + i0)), af[c]);
            else
#pragma unroll
                for (int e = 0; e < 8; ++e) af[c][e] = 0.f;
        }
        if (t < T) asm volatile("cp.async.wait_group 1;" ::: "memory");
        else asm volatile("cp.async.wait_group 0;" ::: "memory");
        __syncthreads();
        const uint16_t* Bs = reinterpret_cast<const uint16_t*>(smem + (t & 1) * stage_bytes);
        const float* Gs = reinterpret_cast<const float*>(Bs + size_t(K) * r);
        float qv[NCH][8];
#pragma unroll
        for (int c = 0; c < NCH; ++c) {
            float gc[1][8];
            load_gslice<1>(Gs + c * 256, r - c * 256, lane, gc);
#pragma unroll
            for (int e = 0; e < 8; ++e) qv[c][e] = af[c][e] * gc[0][e];
        }
        const int64_t row = row1 + t - 1;
        float bv = -INFINITY;
        int bid = INT_MAX, bj = -1;
        for (int j0 = warp; j0 < K; j0 += 4 * kStreamWarps) {
            float part[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int j = j0 + u * kStreamWarps;
                part[u] = 0.f;
                if (j < K) {
#pragma unroll
                    for (int c = 0; c < NCH; ++c) {
                        float bf[1][8];
                        load_bslice<1>(Bs + size_t(j) * r + c * 256, r - c * 256, lane, true, bf);
#pragma unroll
                        for (int e = 0; e < 8; ++e) part[u] = fmaf(qv[c][e], bf[0][e], part[u]);
                    }
                }
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int j = j0 + u * kStreamWarps;
                const float d = warp_sum(part[u]);
                if (j < K) {
                    const float sj = __ldg(vals + row * K + j) + d;
                    const int idj = __ldg(ids + row * K + j);
                    if (bj < 0 || ranks_before(sj, idj, bv, bid)) {
                        bv = sj;
                        bid = idj;
                        bj = j;
                    }
                }
            }
        }
        if (lane == 0) {
            wv[warp] = bv;
            wi[warp] = bid;
            wj[warp] = bj;
        }
        __syncthreads();
        // every thread reduces the warps' bests in the same order
        float best = -INFINITY;
        int best_id = INT_MAX, best_j = -1;
        for (int w = 0; w < kStreamWarps; ++w) {
            const int j = wj[w];
            if (j >= 0 && (best_j < 0 || ranks_before(wv[w], wi[w], best, best_id) ||
                           (wv[w] == best && wi[w] == best_id && j < best_j))) {
                best = wv[w];
                best_id = wi[w];
                best_j = j;
            }
        }
        if (tid == 0) {
            path[int64_t(q) * T + (t - 1)] = best_id;
            path_scores[int64_t(q) * T + (t - 1)] = best;
        }
        a = best_id;
        __syncthreads();  // buffer t & 1 and the warps' bests are free again
    }
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
    const size_t ssmem = walk_stream_smem(K, r);
    if (ssmem <= 200 * 1024) {
#define DF2_WALK_STREAM(N)                                                                          \
    do {                                                                                            \
        cudaError_t e = cudaFuncSetAttribute(walk_stream_kernel<N>,                                 \
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, int(ssmem)); \
        if (e != cudaSuccess) return e;                                                             \
        walk_stream_kernel<N><<<unsigned(R), kStreamThreads, ssmem, stream>>>(anchors, B, ids, vals, G, \
                                                                              A, Bc, V, K, r, path,   \
                                                                              scores, dev_status);    \
    } while (0)
        if (nch <= 1) DF2_WALK_STREAM(1);
        else if (nch <= 2) DF2_WALK_STREAM(2);
        else if (nch <= 4) DF2_WALK_STREAM(4);
        else if (nch <= 8) DF2_WALK_STREAM(8);
        else DF2_WALK_STREAM(16);
#undef DF2_WALK_STREAM
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
