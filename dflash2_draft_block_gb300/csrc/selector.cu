// Candidate selector: greedy walk and teacher-forced pair scores.
//
// Pair score S_t(a, b) = U_t(b) + < A(a) (.) H(h_t), B(b) > (verl-SpeCo PR #62,
// "What DFlash2 adds"; "DFlash 2 Explanation", "Problem 1").  The walk starts at
// the anchor and feeds each position's best successor in as the next
// predecessor (vLLM Speculators "DFlash2" guide, "Candidate Selector"); the
// teacher-forced scorer takes the predecessor as given (PR #62, "Selector
// training objective").
//
// One warp per request (walk) or per row (pair scores).  Lane l owns rank
// elements [8l, 8l+8) of every 256-wide chunk: the gate q = A[a] (.) G_t is
// formed once per position in registers, each candidate's B row is read with one
// 16-byte load per lane per chunk, and a shuffle tree sums the lanes.  The
// candidate loop is unrolled by 4 so that four B-row gathers are in flight.
#include "common.cuh"
#include "kernels.h"

namespace df2 {

namespace {

constexpr int kWarpsPerBlock = 4;

// q[c][e] = A[a, 256c + 8l + e] * G[256c + 8l + e] for the lane's slice (NCH chunks).
template <int NCH>
__device__ __forceinline__ void load_gate(const uint16_t* __restrict__ A, int64_t a, int r,
                                          const float* __restrict__ Grow, int lane,
                                          float q[NCH][8]) {
#pragma unroll
    for (int c = 0; c < NCH; ++c) {
        const int i0 = c * 256 + lane * 8;
        if (i0 < r) {
            float af[8];
            unpack8(__ldg(reinterpret_cast<const uint4*>(A + a * r + i0)), af);
            const float4 g0 = __ldg(reinterpret_cast<const float4*>(Grow + i0));
            const float4 g1 = __ldg(reinterpret_cast<const float4*>(Grow + i0 + 4));
            q[c][0] = af[0] * g0.x; q[c][1] = af[1] * g0.y; q[c][2] = af[2] * g0.z; q[c][3] = af[3] * g0.w;
            q[c][4] = af[4] * g1.x; q[c][5] = af[5] * g1.y; q[c][6] = af[6] * g1.z; q[c][7] = af[7] * g1.w;
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) q[c][e] = 0.f;
        }
    }
}

template <int NCH>
__device__ __forceinline__ float dot_lane(const uint16_t* __restrict__ Bc, int64_t b, int r, int lane,
                                          const float q[NCH][8]) {
    float s = 0.f;
#pragma unroll
    for (int c = 0; c < NCH; ++c) {
        const int i0 = c * 256 + lane * 8;
        if (i0 < r) {
            float bf[8];
            unpack8(__ldg(reinterpret_cast<const uint4*>(Bc + b * r + i0)), bf);
#pragma unroll
            for (int e = 0; e < 8; ++e) s = fmaf(q[c][e], bf[e], s);
        }
    }
    return s;
}

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

__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gmem_src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(
                     static_cast<uint32_t>(__cvta_generic_to_shared(smem_dst))),
                 "l"(gmem_src)
                 : "memory");
}

// Walk with everything it can read gathered into shared memory first: the B rows
// of every candidate of rows 1..B-1, the A rows of the anchor and of every
// candidate of rows 1..B-2 (the only possible predecessors), and the G rows.
// The gathers are independent, so they are all in flight at once; the B-1
// sequential steps then touch shared memory only and are run by one warp with
// no block-wide barrier.  One CTA per request (8 warps issue the gathers).
constexpr int kWalkThreads = 256;

// Sum 16 per-lane values over the warp at once: at each butterfly level a lane
// keeps half of its values and adds its partner's copy of them, so 16 shuffles in
// 5 levels replace 16 separate 5-level reductions.  Returns u = (lane >> 1) & 15:
// on return v[0] of this lane is the warp-wide sum of the lanes' v[u].
__device__ __forceinline__ int reduce16_transpose(float v[16], int lane) {
#pragma unroll
    for (int m = 16, h = 8; m >= 2; m >>= 1, h >>= 1) {
        const bool upper = (lane & m) != 0;
#pragma unroll
        for (int i = 0; i < h; ++i) {
            const float send = upper ? v[i] : v[i + h];
            const float keep = upper ? v[i + h] : v[i];
            v[i] = keep + __shfl_xor_sync(kFull, send, m);
        }
    }
    v[0] += __shfl_xor_sync(kFull, v[0], 1);
    return (lane >> 1) & 15;
}

__host__ __device__ inline size_t walk_cta_smem(int B, int K, int r) {
    const size_t T = size_t(B) - 1;
    return T * K * r * 2 + ((T - 1) * K + 1) * r * 2 + T * r * 4 + T * K * 8 + 64;
}

template <int NCH>
__global__ void __launch_bounds__(kWalkThreads)
walk_cta_kernel(const int32_t* __restrict__ anchors, int B, const int32_t* __restrict__ ids,
                const float* __restrict__ vals, const float* __restrict__ G,
                const uint16_t* __restrict__ A, const uint16_t* __restrict__ Bc, int64_t V, int K,
                int r, int32_t* __restrict__ path, float* __restrict__ path_scores,
                int32_t* __restrict__ dev_status) {
    extern __shared__ __align__(16) uint8_t smem[];
    const int T = B - 1;
    const int q = blockIdx.x;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    uint16_t* Bs = reinterpret_cast<uint16_t*>(smem);                     // [T*K][r]
    uint16_t* As = Bs + size_t(T) * K * r;                                // [(T-1)*K + 1][r]
    float* Gs = reinterpret_cast<float*>(As + (size_t(T - 1) * K + 1) * r);  // [T][r]
    float* vs = Gs + size_t(T) * r;                                       // [T*K]
    int* is = reinterpret_cast<int*>(vs + size_t(T) * K);                 // [T*K]
    int* bad = is + size_t(T) * K;

    const int64_t row1 = int64_t(q) * B + 1;  // first drafted row of the request
    const int32_t a0 = __ldg(anchors + q);
    if (tid == 0) *bad = (a0 < 0 || a0 >= V) ? 1 : 0;
    __syncthreads();
    for (int e = tid; e < T * K; e += kWalkThreads) {
        const int32_t b = __ldg(ids + row1 * K + e);
        is[e] = b;
        vs[e] = __ldg(vals + row1 * K + e);
        if (b < 0 || b >= V) *bad = 1;
    }
    __syncthreads();
    if (*bad) {
        for (int t = tid; t < T; t += kWalkThreads) {
            path[int64_t(q) * T + t] = -1;
            path_scores[int64_t(q) * T + t] = __int_as_float(0x7fc00000);
        }
        if (tid == 0 && dev_status) atomicOr(dev_status, DF2_STATUS_ID_OUT_OF_RANGE);
        return;
    }

    const int cpr = r / 8;  // 16-byte chunks per bf16 row
    for (int i = tid; i < T * K * cpr; i += kWalkThreads) {
        const int row = i / cpr, c = i - row * cpr;
        cp_async16(Bs + size_t(row) * r + c * 8, Bc + int64_t(is[row]) * r + c * 8);
    }
    const int na = (T - 1) * K + 1;
    for (int i = tid; i < na * cpr; i += kWalkThreads) {
        const int arow = i / cpr, c = i - arow * cpr;
        const int64_t a = arow == 0 ? a0 : is[arow - 1];
        cp_async16(As + size_t(arow) * r + c * 8, A + a * r + c * 8);
    }
    const int gpr = r / 4;  // 16-byte chunks per fp32 row
    for (int i = tid; i < T * gpr; i += kWalkThreads) {
        const int t = i / gpr, c = i - t * gpr;
        cp_async16(Gs + size_t(t) * r + c * 4, G + (row1 + t) * r + c * 4);
    }
    asm volatile("cp.async.commit_group;\n\tcp.async.wait_all;" ::: "memory");
    __syncthreads();
    if (warp != 0) return;

    // The sequential part, one warp, shared memory only.  Lane l owns rank
    // elements [256c + 8l, 256c + 8l + 8) of the gate and of every B row.
    int arow = 0;  // As row of the current predecessor
    for (int t = 1; t <= T; ++t) {
        float qv[NCH][8];
#pragma unroll
        for (int c = 0; c < NCH; ++c) {
            const int i0 = c * 256 + lane * 8;
            if (i0 < r) {
                float af[8];
                unpack8(*reinterpret_cast<const uint4*>(As + size_t(arow) * r + i0), af);
                const float* g = Gs + size_t(t - 1) * r + i0;
#pragma unroll
                for (int e = 0; e < 8; ++e) qv[c][e] = af[e] * g[e];
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e) qv[c][e] = 0.f;
            }
        }
        float best = -INFINITY;
        int best_id = -1, best_j = 0;
        for (int j0 = 0; j0 < K; j0 += 16) {
            // 16 candidates' lane partials, summed across the warp together
            float part[16];
#pragma unroll
            for (int u = 0; u < 16; ++u) {
                part[u] = 0.f;
                if (j0 + u < K) {
                    const uint16_t* brow = Bs + (size_t(t - 1) * K + j0 + u) * r;
#pragma unroll
                    for (int c = 0; c < NCH; ++c) {
                        const int i0 = c * 256 + lane * 8;
                        if (i0 < r) {
                            float bf[8];
                            unpack8(*reinterpret_cast<const uint4*>(brow + i0), bf);
#pragma unroll
                            for (int e = 0; e < 8; ++e) part[u] = fmaf(qv[c][e], bf[e], part[u]);
                        }
                    }
                }
            }
            // lanes 2u and 2u+1 end up holding candidate j0+u's full sum
            const int u = reduce16_transpose(part, lane);
            float sj = -INFINITY;
            int idj = INT_MAX, jj = -1;
            if (j0 + u < K) {
                sj = vs[(t - 1) * K + j0 + u] + part[0];
                idj = is[(t - 1) * K + j0 + u];
                jj = j0 + u;
            }
#pragma unroll
            for (int o = 16; o; o >>= 1) {
                const float ov = __shfl_xor_sync(kFull, sj, o);
                const int oi = __shfl_xor_sync(kFull, idj, o);
                const int oj = __shfl_xor_sync(kFull, jj, o);
                if (oj >= 0 && (jj < 0 || ranks_before(ov, oi, sj, idj))) { sj = ov; idj = oi; jj = oj; }
            }
            if (jj >= 0 && (best_id < 0 || ranks_before(sj, idj, best, best_id))) {
                best = sj;
                best_id = idj;
                best_j = jj;
            }
        }
        if (lane == 0) {
            path[int64_t(q) * T + (t - 1)] = best_id;
            path_scores[int64_t(q) * T + (t - 1)] = best;
        }
        arow = 1 + (t - 1) * K + best_j;
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
