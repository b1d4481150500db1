// The merge kernel: one CTA per position folds the sorted per-CTA lists of the
// head kernels into the final top-K (merge_position, topk_merge_dev.cuh).
#include "common.cuh"
#include "kernels.h"
#include "topk_merge_dev.cuh"

namespace df2 {

namespace {

using namespace mrg;

// Six CTAs per SM (40 registers): the merge runs one short CTA per position, so
// occupancy hides its load latencies; the rare exact recomputes may spill a few
// values to local memory instead.
template <int R>
__global__ void __launch_bounds__(kMergeThreads, 6)
topk_merge_sorted_kernel(const float* __restrict__ part_v, const int* __restrict__ part_id, int S,
                         int64_t P, int K, int32_t* __restrict__ out_ids,
                         float* __restrict__ out_vals, LogitMap lm, Refine rf) {
    extern __shared__ __align__(16) uint8_t smem[];
    merge_position<R>(part_v, part_id, S, P, K, blockIdx.x, out_ids, out_vals, smem, lm, rf);
}

template <int R>
cudaError_t launch_merge(const float* part_v, const int* part_id, int S, int64_t P, int K, int32_t* ids,
                         float* vals, cudaStream_t stream, LogitMap lm, Refine rf) {
    const size_t smem = merge_smem(S, K);
    const cudaError_t e = cudaFuncSetAttribute(topk_merge_sorted_kernel<R>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (e != cudaSuccess) return e;
    topk_merge_sorted_kernel<R><<<unsigned(P), kWarps * 32, smem, stream>>>(part_v, part_id, S, P, K, ids, vals,
                                                                           lm, rf);
    return cudaSuccess;
}

}  // namespace

cudaError_t topk_merge_sorted_launch(const float* part_v, const int* part_id, int S, int64_t P, int K,
                                     int32_t* ids, float* vals, cudaStream_t stream, LogitMap lm, Refine rf) {
    const cudaError_t e = K <= 32 ? launch_merge<1>(part_v, part_id, S, P, K, ids, vals, stream, lm, rf)
                                  : launch_merge<2>(part_v, part_id, S, P, K, ids, vals, stream, lm, rf);
    if (e != cudaSuccess) return e;
    note_launch();
    return cudaGetLastError();
}

}  // namespace df2
