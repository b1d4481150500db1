// Internal launchers of libdflash2 (not part of the C-ABI).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace df2 {

// The unary logits' output multiplier and final softcap: u -> cap * tanh(mul * u / cap),
// or mul * u when cap == 0 (the defaults leave every value bit for bit as it is).
// With mul > 0 the map is non-decreasing, so the kernels select on the raw logits
// and map only the K values they keep; where rounding maps neighbours to one
// value (a saturating cap), the kept list is re-ranked by (mapped value, lower id).
struct LogitMap {
    float mul = 1.f;
    float cap = 0.f;
    __host__ __device__ __forceinline__ bool identity() const { return mul == 1.f && cap == 0.f; }
    __device__ __forceinline__ float operator()(float u) const {
        const float x = mul * u;
        return cap > 0.f ? cap * tanhf(x / cap) : x;
    }
};

// ---- unary logits + top-K on the CUDA cores (any D % 8 == 0, K <= DF2_MAX_TOPK)
bool head_simple_supported(int64_t D, int K);
size_t head_simple_workspace(int64_t P, int64_t D, int64_t V, int K, int num_sms);
cudaError_t head_simple_launch(const uint16_t* h, int64_t P, int64_t D, const uint16_t* W, int64_t V,
                               int K, int32_t* ids, float* vals, void* ws, int num_sms,
                               cudaStream_t stream, LogitMap lm = LogitMap{});

// ---- S unsorted partial lists [S][P][K] (id -1 = empty slot) -> sorted top-K [P][K],
//      the kept values mapped by lm
cudaError_t topk_merge_launch(const float* part_v, const int* part_id, int S, int64_t P, int K,
                              int32_t* ids, float* vals, cudaStream_t stream, LogitMap lm = LogitMap{});

// Where the top-K merges find the logits' operands to recompute near-tied
// neighbours exactly (h == null: no recompute).
struct Refine {
    const uint16_t* h;   // [P][D] bf16
    const uint16_t* W;   // [V][D] bf16
    int64_t D;           // D % 8 == 0, rows 16-byte aligned
};

// ---- S partial lists [S][P][K], each in rank order (id -1 = empty), K <= 64 -> top-K [P][K];
//      with rf, near-tied neighbours (the K-th/(K+1)-th boundary included) recomputed exactly
struct TopkParts {
    const float* v;
    const int* id;
    int S;
};
cudaError_t topk_merge_sorted_launch(const float* part_v, const int* part_id, int S, int64_t P, int K,
                                     int32_t* ids, float* vals, cudaStream_t stream,
                                     LogitMap lm = LogitMap{}, Refine rf = Refine{nullptr, nullptr, 0});

// ---- out = X . W^T on the CUDA cores, columns split between two outputs
cudaError_t gemm_simple_launch(const void* X, bool x_f32, const uint16_t* W, int64_t M, int64_t N,
                               int64_t Kd, float* out0, int64_t ld0, int64_t n_split, float* out1,
                               int64_t ld1, cudaStream_t stream);

// ---- the same for few rows of X (one warp per output column, X in shared memory);
//      needs Kd % 8 == 0
cudaError_t gemm_rows_launch(const void* X, bool x_f32, const uint16_t* W, int64_t M, int64_t N,
                             int64_t Kd, float* out0, int64_t ld0, int64_t n_split, float* out1,
                             int64_t ld1, int num_sms, cudaStream_t stream);

// ---- many-row tensor-core GEMM (gemm_tc.cu): A [M, Kd] x B [N, Kd]^T, bf16
bool wide_supported(int64_t M, int64_t N, int64_t Kd, int K);
size_t wide_topk_workspace(int64_t M, int64_t N, int K, int num_sms);
// fp32 out, columns n < n_split to out0 (row stride ld0), the rest to out1
cudaError_t wide_store_launch(const uint16_t* A, int64_t M, const uint16_t* B, int64_t N, int64_t Kd,
                              float* out0, int64_t ld0, int64_t n_split, float* out1, int64_t ld1,
                              int32_t* dev_status, cudaStream_t stream);
// per-row top-K of A B^T (ids = B row indices), merged into ids/vals [M][K]; with
// parts_out the sorted per-range lists are left for the caller to fold instead,
// and zero_words[0 .. n_zero) are zeroed for the next kernel in the stream.  With
// W_H, also G = A W_H^T [M][r] (fp32), in the same launch where it fits
cudaError_t wide_topk_launch(const uint16_t* A, int64_t M, const uint16_t* B, int64_t N, int64_t Kd, int K,
                             int32_t* ids, float* vals, void* ws, int32_t* dev_status, int num_sms,
                             cudaStream_t stream, TopkParts* parts_out = nullptr,
                             unsigned* zero_words = nullptr, int n_zero = 0,
                             const uint16_t* W_H = nullptr, int64_t r = 0, float* G = nullptr);

// ---- selector
cudaError_t walk_launch(const int32_t* anchors, int R, int B, const int32_t* ids, const float* vals,
                        const float* G, const uint16_t* A, const uint16_t* Bc, int64_t V, int K,
                        int r, int32_t* path, float* scores, int32_t* dev_status,
                        cudaStream_t stream);
cudaError_t pair_scores_launch(const int32_t* pred, int64_t P, const int32_t* ids,
                               const float* vals, const float* G, const uint16_t* A,
                               const uint16_t* Bc, int64_t V, int K, int r, float* scores,
                               int32_t* dev_status, cudaStream_t stream);
cudaError_t selector_ce_launch(const float* scores, const int32_t* ids, const int32_t* targets, int64_t P,
                               int K, int64_t V, float* loss, int32_t* label_idx, int32_t* dev_status,
                               cudaStream_t stream);

// ---- lattice: L[q][t-1][i][j] = S_t(i-th predecessor, j-th candidate), then a walk over it
cudaError_t lattice_launch(const int32_t* anchors, int R, int B, const int32_t* ids, const float* vals,
                           const float* G, const uint16_t* A, const uint16_t* Bc, int64_t V, int K,
                           int r, float* lattice, int32_t* dev_status, cudaStream_t stream);
cudaError_t lattice_walk_launch(const float* lattice, const int32_t* ids, int R, int B, int K, int64_t V,
                                const float* uniforms, float temperature, int32_t* path,
                                float* path_scores, int32_t* dev_status, cudaStream_t stream);

// ---- the fused tail of the draft head: one thread-block cluster per request
// folds its rows' sorted lists, scores the teacher-forced pairs (pred nullable)
// and the lattice slots, and walks the request
bool draft_tail_supported(int64_t P, int B, int K, int r, int S, int num_sms);
cudaError_t draft_tail_launch(const TopkParts& parts, int64_t P, int K, int32_t* ids, float* vals,
                              const int32_t* anchors, int B, const float* G, const uint16_t* A,
                              const uint16_t* Bc, int64_t V, int r, int32_t* path, float* path_scores,
                              const int32_t* pred, float* pair_scores, int32_t* dev_status,
                              cudaStream_t stream, LogitMap lm = LogitMap{},
                              Refine rf = Refine{nullptr, nullptr, 0});

// ---- conv: y = sum_{j<taps, t-j>=0} (base[j] + dyn[p, j, c/g]) * x[p-j]
// ---- conv prepare for few rows (P <= 64, B <= 16): projection and apply fused
bool conv_prepare_rows_supported(int64_t P, int C, int B, bool f32);
cudaError_t conv_prepare_rows_launch(const void* x, bool f32, int64_t P, int C, int B, int taps, int g,
                                     const uint16_t* W, const float* base, void* y, float* dyn_out,
                                     cudaStream_t stream);
// ---- conv prepare for many bf16 rows, fused on the tensor cores (conv_tc.cu): the
//      projection, dyn_out and the conv applied in one kernel; needs 128 % B == 0,
//      taps <= 4 and a multiple of 8 groups dividing C / g
bool conv_prepare_tc_supported(int64_t P, int C, int B, int taps, int g);
cudaError_t conv_prepare_tc_launch(const uint16_t* x, int64_t P, int C, int B, int taps, int g,
                                   const uint16_t* W, const float* base, uint16_t* y, float* dyn_out,
                                   int32_t* dev_status, cudaStream_t stream);
cudaError_t conv_apply_launch(const void* x, bool f32, int64_t P, int C, int B, int taps, int g,
                              const float* base_io, const float* dyn, int64_t dyn_ld, void* y,
                              cudaStream_t stream, const void* res = nullptr);

}  // namespace df2
