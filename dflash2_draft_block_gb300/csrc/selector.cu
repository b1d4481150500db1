// Candidate selector: greedy walk and teacher-forced pair scores.
//
// Pair score S_t(a, b) = U_t(b) + < A(a) (.) H(h_t), B(b) > (verl-SpeCo PR #62,
// "What DFlash2 adds"; "DFlash 2 Explanation", "Problem 1").  The walk starts at
// the anchor and feeds each position's best successor in as the next
// predecessor (vLLM Speculators "DFlash2" guide, "Candidate Selector"); the
// teacher-forced scorer takes the predecessor as given (PR #62, "Selector
// training objective").
//
// The walk runs one CTA per request: with its gathers staged in shared memory
// (walk_request_cta, selector_dev.cuh) when they fit, else reading them from L2
// one step after they were prefetched (walk_l2_kernel).  The teacher-forced scores
// run one warp per (row, group of 8 candidates).  Lane l owns rank elements
// [8l, 8l+8) of every 256-wide chunk: the gate q = A[a] (.) G_t is formed once per
// position in registers, each candidate's B row is read with one 16-byte load per
// lane per chunk, and a shuffle tree sums the lanes.
#include "common.cuh"
#include "kernels.h"
#include "selector_dev.cuh"

namespace df2 {

namespace {

using namespace sel;

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

constexpr int kStreamThreads = 256;
constexpr int kStreamWarps = kStreamThreads / 32;

// Walk for requests whose gathers do not fit in shared memory, with nothing staged:
// one CTA per request reads the candidates' B rows and the G row straight from L2,
// where they were prefetched one step ahead (they do not depend on the choice), and
// the first kPredPrefetch candidates' A rows -- the likeliest predecessors, the
// candidates being sorted by unary value -- are prefetched too; any other
// predecessor's A row is read on demand.  With a few hundred bytes of shared memory
// every request is resident at once, so the steps' latencies overlap across
// requests instead of running in waves.  Warp w scores candidates w, w+8, ... with
// the lane slicing, fmaf chains and shuffle trees of the other walk kernels, and the
// warps' bests meet in shared memory in a fixed order: bit-identical scores.
constexpr int kPredPrefetch = 8;

template <int NCH>
__global__ void __launch_bounds__(kStreamThreads, NCH <= 8 ? 2 : 1)
walk_l2_kernel(const int32_t* __restrict__ anchors, int B, const int32_t* __restrict__ ids,
               const float* __restrict__ vals, const float* __restrict__ G, const uint16_t* __restrict__ A,
               const uint16_t* __restrict__ Bc, int64_t V, int K, int r, int32_t* __restrict__ path,
               float* __restrict__ path_scores, int32_t* __restrict__ dev_status) {
    __shared__ float wv[kStreamWarps];
    __shared__ int wi[kStreamWarps], wj[kStreamWarps];
    __shared__ int bad;
    const int T = B - 1;
    const int q = blockIdx.x;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
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
    const int lines = (r * 2 + 127) / 128;   // 128-byte lines of a codebook row
    const int glines = (r * 4 + 127) / 128;  // of a G row
    // position t's candidates' B rows and G row, and its likeliest candidates' A rows
    // (the predecessors at step t+1), into L2
    auto prefetch = [&](int t) {
        const int64_t row = row1 + t - 1;
        for (int e = tid; e < K * lines; e += kStreamThreads)
            asm volatile("prefetch.global.L2 [%0];" ::"l"(Bc + int64_t(__ldg(ids + row * K + e / lines)) * r +
                                                          (e % lines) * 64));
        for (int e = tid; e < glines; e += kStreamThreads)
            asm volatile("prefetch.global.L2 [%0];" ::"l"(G + row * r + e * 32));
        if (t < T) {
            const int np = K < kPredPrefetch ? K : kPredPrefetch;
            for (int e = tid; e < np * lines; e += kStreamThreads)
                asm volatile("prefetch.global.L2 [%0];" ::"l"(A + int64_t(__ldg(ids + row * K + e / lines)) * r +
                                                              (e % lines) * 64));
        }
    };
    prefetch(1);
    int32_t a = a0;
    for (int t = 1; t <= T; ++t) {
        if (t < T) prefetch(t + 1);
        const int64_t row = row1 + t - 1;
        // the gate A[a] (.) G_t on this warp's lane slices
        float af[NCH][8];
#pragma unroll
        for (int c = 0; c < NCH; ++c) {
            const int i0 = c * 256 + lane * 8;
            if (i0 < r) unpack8(__ldg(reinterpret_cast<const uint4*>(A + int64_t(a) * r + i0)), af[c]);
            else
#pragma unroll
                for (int e = 0; e < 8; ++e) af[c][e] = 0.f;
        }
        float qv[NCH][8];
#pragma unroll
        for (int c = 0; c < NCH; ++c) {
            float gc[1][8];
            load_gslice<1>(G + row * r + c * 256, r - c * 256, lane, gc);
#pragma unroll
            for (int e = 0; e < 8; ++e) qv[c][e] = af[c][e] * gc[0][e];
        }
        float bv = -INFINITY;
        int bid = INT_MAX, bj = -1;
        for (int j0 = warp; j0 < K; j0 += 4 * kStreamWarps) {
            float part[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int j = j0 + u * kStreamWarps;
                part[u] = 0.f;
                if (j < K) {
                    const uint16_t* brow = Bc + int64_t(__ldg(ids + row * K + j)) * r;
#pragma unroll
                    for (int c = 0; c < NCH; ++c) {
                        float bf[1][8];
                        load_bslice<1>(brow + c * 256, r - c * 256, lane, true, bf);
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
        __syncthreads();  // the warps' bests are free again
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
#define DF2_WALK_L2(N)                                                                                \
    walk_l2_kernel<N><<<unsigned(R), kStreamThreads, 0, stream>>>(anchors, B, ids, vals, G, A, Bc, V, K, r, \
                                                                  path, scores, dev_status)
    if (nch <= 1) DF2_WALK_L2(1);
    else if (nch <= 2) DF2_WALK_L2(2);
    else if (nch <= 4) DF2_WALK_L2(4);
    else if (nch <= 8) DF2_WALK_L2(8);
    else DF2_WALK_L2(16);
#undef DF2_WALK_L2
    note_launch();
    return cudaGetLastError();
}

namespace {

// The selector's K-way cross-entropy ([PR62] "Selector training objective"): one
// warp per row.  The lanes stride the row's K scores for its maximum and the first
// column holding the target, then sum exp(score - maximum); lane 0 writes
// loss = log(sum) + maximum - score[label].  Rows whose target is not a candidate
// (or is negative) get label -1 and NaN.
constexpr int kCeWarps = 8;

__global__ void __launch_bounds__(kCeWarps * 32)
selector_ce_kernel(const float* __restrict__ scores, const int32_t* __restrict__ ids,
                   const int32_t* __restrict__ targets, int64_t P, int K, int64_t V, float* __restrict__ loss,
                   int32_t* __restrict__ label_idx, int32_t* __restrict__ dev_status) {
    const int64_t p = int64_t(blockIdx.x) * kCeWarps + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (p >= P) return;
    const int32_t y = __ldg(targets + p);
    const bool has = y >= 0 && y < V;
    if (y >= V && lane == 0 && dev_status) atomicOr(dev_status, DF2_STATUS_ID_OUT_OF_RANGE);
    const float* s = scores + p * K;
    const int32_t* id = ids + p * K;
    float m = -INFINITY;
    int js = INT_MAX;
    for (int j = lane; j < K; j += 32) {
        m = fmaxf(m, __ldg(s + j));
        if (has && __ldg(id + j) == y && j < js) js = j;
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) {
        m = fmaxf(m, __shfl_xor_sync(kFull, m, o));
        js = min(js, __shfl_xor_sync(kFull, js, o));
    }
    if (js == INT_MAX) {
        if (lane == 0) {
            loss[p] = __int_as_float(0x7fc00000);
            if (label_idx) label_idx[p] = -1;
        }
        return;
    }
    float sum = 0.f;
    for (int j = lane; j < K; j += 32) sum += expf(__ldg(s + j) - m);
#pragma unroll
    for (int o = 16; o; o >>= 1) sum += __shfl_xor_sync(kFull, sum, o);
    if (lane == 0) {
        loss[p] = logf(sum) + m - __ldg(s + js);
        if (label_idx) label_idx[p] = js;
    }
}

}  // namespace

cudaError_t selector_ce_launch(const float* scores, const int32_t* ids, const int32_t* targets, int64_t P,
                               int K, int64_t V, float* loss, int32_t* label_idx, int32_t* dev_status,
                               cudaStream_t stream) {
    const unsigned grid = unsigned((P + kCeWarps - 1) / kCeWarps);
    selector_ce_kernel<<<grid, kCeWarps * 32, 0, stream>>>(scores, ids, targets, P, K, V, loss, label_idx,
                                                           dev_status);
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
