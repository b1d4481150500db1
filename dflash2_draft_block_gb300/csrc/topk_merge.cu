// Cross-CTA merge of sorted per-CTA top-K lists (K <= 64) into the final top-K.
//
// One CTA per position.  All lists of the position are first copied to shared
// memory in one round of independent loads; each of the 8 warps then folds every
// 8th CTA list into a register-resident list (topk_warp.cuh): a list row is a
// batch already in rank order, and one ballot against the running K-th entry
// drops it unless it improves the list.  Warp 0 then folds the other warps' lists and writes the
// K best in rank order.
#include "common.cuh"
#include "kernels.h"
#include "topk_warp.cuh"

namespace df2 {

namespace {

constexpr int kWarps = 8;

template <int R>
__global__ void __launch_bounds__(kWarps * 32)
topk_merge_sorted_kernel(const float* __restrict__ part_v, const int* __restrict__ part_id, int S,
                         int64_t P, int K, int32_t* __restrict__ out_ids,
                         float* __restrict__ out_vals) {
    extern __shared__ __align__(16) uint8_t smem[];
    float* cv = reinterpret_cast<float*>(smem);        // [S*K] this position's candidates
    int* ci = reinterpret_cast<int*>(cv + S * K);
    __shared__ float xv[kWarps][R * 32];
    __shared__ int xi[kWarps][R * 32];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t p = blockIdx.x;
    // one round of independent, coalesced loads of every list of this position
    for (int i = threadIdx.x; i < S * K; i += kWarps * 32) {
        const int s = i / K, k = i - s * K;
        const size_t at = (size_t(s) * P + p) * K + k;
        cv[i] = __ldg(part_v + at);
        ci[i] = __ldg(part_id + at);
    }
    __syncthreads();
    wtk::List<R> m;
    m.clear();
    for (int s = warp; s < S; s += kWarps) {
#pragma unroll
        for (int rr = 0; rr < R; ++rr) {
            const int k = rr * 32 + lane;
            float v = -INFINITY;
            int id = wtk::kEmptyId;
            if (k < K && ci[s * K + k] >= 0) {
                v = cv[s * K + k];
                id = ci[s * K + k];
            }
            m.offer_sorted(v, id, K, lane);
        }
    }
#pragma unroll
    for (int rr = 0; rr < R; ++rr) {
        xv[warp][rr * 32 + lane] = m.v[rr];
        xi[warp][rr * 32 + lane] = m.id[rr];
    }
    __syncthreads();
    if (warp != 0) return;
    for (int w = 1; w < kWarps; ++w)
#pragma unroll
        for (int rr = 0; rr < R; ++rr) m.offer_sorted(xv[w][rr * 32 + lane], xi[w][rr * 32 + lane], K, lane);
#pragma unroll
    for (int rr = 0; rr < R; ++rr) {
        const int k = rr * 32 + lane;
        if (k < K) {
            const bool ok = m.id[rr] != wtk::kEmptyId;
            out_ids[p * K + k] = ok ? m.id[rr] : -1;
            out_vals[p * K + k] = ok ? m.v[rr] : -INFINITY;
        }
    }
}

}  // namespace

cudaError_t topk_merge_sorted_launch(const float* part_v, const int* part_id, int S, int64_t P, int K,
                                     int32_t* ids, float* vals, cudaStream_t stream) {
    const size_t smem = size_t(S) * K * 8;
    cudaError_t e;
    if (K <= 32) {
        e = cudaFuncSetAttribute(topk_merge_sorted_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 int(smem));
        if (e != cudaSuccess) return e;
        topk_merge_sorted_kernel<1><<<unsigned(P), kWarps * 32, smem, stream>>>(part_v, part_id, S, P, K,
                                                                                ids, vals);
    } else {
        e = cudaFuncSetAttribute(topk_merge_sorted_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 int(smem));
        if (e != cudaSuccess) return e;
        topk_merge_sorted_kernel<2><<<unsigned(P), kWarps * 32, smem, stream>>>(part_v, part_id, S, P, K,
                                                                                ids, vals);
    }
    note_launch();
    return cudaGetLastError();
}

}  // namespace df2
