// The fused tail of the draft head: after the head kernel has left its sorted
// per-CTA (or per-range) top-K lists in the workspace, one launch finishes the
// selector's part of the cycle.  CTA p
//   1. folds position p's lists into its top-K (merge_position),
//   2. scores position p's candidates after the teacher-forced predecessor
//      pred[p] (pair_row_cta; verl-SpeCo PR #62, "Selector training objective"),
//   3. takes a ticket for its request; the CTA that completes a request's block
//      walks it (walk_request_cta; vLLM Speculators "DFlash2" guide, "Candidate
//      Selector": start at the anchor, feed each best successor in as the next
//      predecessor).
// The results are the ones the separate merge, walk and teacher-forced kernels
// give (the same arithmetic, in the same order); only the launches and the
// waiting between them go.  Every CTA must be resident at once for the tickets
// to be taken in one wave, so the launch is used for P <= the SM count.
#include "common.cuh"
#include "kernels.h"
#include "selector_dev.cuh"
#include "topk_merge_dev.cuh"

namespace df2 {

namespace {

constexpr int kTailThreads = 256;
static_assert(kTailThreads == mrg::kMergeThreads && kTailThreads == sel::kWalkThreads,
              "the three phases share one CTA shape");

size_t tail_smem(int B, int K, int r, int S) {
    const size_t a = mrg::merge_smem(S, K), b = sel::walk_cta_smem(B, K, r);
    return a > b ? a : b;
}

template <int R, int NCH>
__global__ void __launch_bounds__(kTailThreads, 1)
draft_tail_kernel(const float* __restrict__ part_v, const int* __restrict__ part_id, int S, int64_t P,
                  int K, int32_t* __restrict__ ids, float* __restrict__ vals,
                  const int32_t* __restrict__ anchors, int B, const float* __restrict__ G,
                  const uint16_t* __restrict__ A, const uint16_t* __restrict__ Bc, int64_t V, int r,
                  int32_t* __restrict__ path, float* __restrict__ path_scores,
                  const int32_t* __restrict__ pred, float* __restrict__ pair_scores,
                  unsigned* __restrict__ tickets, int32_t* __restrict__ dev_status) {
    extern __shared__ __align__(16) uint8_t smem[];
    __shared__ int last;
    const int64_t p = blockIdx.x;
    const int q = int(p / B);

    mrg::merge_position<R>(part_v, part_id, S, P, K, p, ids, vals, smem);
    __syncthreads();  // row p's list is written (by warp 0) before anyone reads it
    if (pred) sel::pair_row_cta<NCH, true>(p, pred, ids, vals, G, A, Bc, V, K, r, pair_scores, dev_status);

    // publish row p, then count it towards request q
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) last = atomicAdd(tickets + q, 1u) == unsigned(B - 1);
    __syncthreads();
    if (!last) return;
    __threadfence();  // the other rows of request q, published before their tickets
    sel::walk_request_cta<NCH, true>(q, anchors, B, ids, vals, G, A, Bc, V, K, r, path, path_scores,
                                     dev_status, smem);
}

}  // namespace

bool draft_tail_supported(int64_t P, int B, int K, int r, int S, int num_sms) {
    return P >= 1 && P <= num_sms && K <= 64 && r <= 4096 && P % B == 0 &&
           tail_smem(B, K, r, S) <= 200 * 1024;
}

cudaError_t draft_tail_launch(const TopkParts& parts, int64_t P, int K, int32_t* ids, float* vals,
                              const int32_t* anchors, int B, const float* G, const uint16_t* A,
                              const uint16_t* Bc, int64_t V, int r, int32_t* path, float* path_scores,
                              const int32_t* pred, float* pair_scores, unsigned* tickets,
                              int32_t* dev_status, cudaStream_t stream) {
    const size_t smem = tail_smem(B, K, r, parts.S);
    const int nch = (r + 255) / 256;
    cudaError_t e = cudaSuccess;
#define DF2_TAIL(RV, N)                                                                                 \
    do {                                                                                                \
        e = cudaFuncSetAttribute(draft_tail_kernel<RV, N>, cudaFuncAttributeMaxDynamicSharedMemorySize,  \
                                 int(smem));                                                            \
        if (e != cudaSuccess) return e;                                                                 \
        draft_tail_kernel<RV, N><<<unsigned(P), kTailThreads, smem, stream>>>(                           \
            parts.v, parts.id, parts.S, P, K, ids, vals, anchors, B, G, A, Bc, V, r, path, path_scores,  \
            pred, pair_scores, tickets, dev_status);                                                    \
    } while (0)
#define DF2_TAIL_N(RV)                        \
    do {                                      \
        if (nch <= 1) DF2_TAIL(RV, 1);        \
        else if (nch <= 2) DF2_TAIL(RV, 2);   \
        else if (nch <= 4) DF2_TAIL(RV, 4);   \
        else if (nch <= 8) DF2_TAIL(RV, 8);   \
        else DF2_TAIL(RV, 16);                \
    } while (0)
    if (K <= 32) DF2_TAIL_N(1);
    else DF2_TAIL_N(2);
#undef DF2_TAIL_N
#undef DF2_TAIL
    note_launch();
    return cudaGetLastError();
}

}  // namespace df2
