// out[m, n] = sum_k X[m, k] * W[n, k] on the CUDA cores, fp32 accumulation.
//
// Used for the hidden projection G = H(h) when the tensor-core head does not
// take the shape, and for the conv kernel projection with fp32 activations.  The
// epilogue splits the columns: n < n_split goes to out0 (row stride ld0), the
// rest to out1 (row stride ld1) — the conv projection's input-side and
// output-side kernels land in separate buffers this way.
#include "common.cuh"
#include "kernels.h"

namespace df2 {

namespace {

constexpr int BM = 64, BN = 64, BK = 16;

template <typename TX>
__device__ __forceinline__ float load_x(const TX* p);
template <>
__device__ __forceinline__ float load_x<float>(const float* p) { return __ldg(p); }
template <>
__device__ __forceinline__ float load_x<uint16_t>(const uint16_t* p) { return bf16_to_f32(__ldg(p)); }

template <typename TX>
__global__ void __launch_bounds__(256)
gemm_nt_simple(const TX* __restrict__ X, const uint16_t* __restrict__ W, int64_t M, int64_t N,
               int64_t Kd, float* __restrict__ out0, int64_t ld0, int64_t n_split,
               float* __restrict__ out1, int64_t ld1) {
    __shared__ float As[BK][BM + 4];
    __shared__ float Bs[BK][BN + 4];
    const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
    const int64_t m0 = int64_t(blockIdx.y) * BM, n0 = int64_t(blockIdx.x) * BN;
    float acc[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;

    for (int64_t k0 = 0; k0 < Kd; k0 += BK) {
        for (int e = threadIdx.x; e < BM * BK; e += 256) {
            const int r = e / BK, c = e % BK;
            const int64_t gm = m0 + r, gk = k0 + c;
            As[c][r] = (gm < M && gk < Kd) ? load_x<TX>(X + gm * Kd + gk) : 0.f;
            const int64_t gn = n0 + r;
            Bs[c][r] = (gn < N && gk < Kd) ? bf16_to_f32(__ldg(W + gn * Kd + gk)) : 0.f;
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < BK; ++kk) {
            float a[4], b[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) a[i] = As[kk][ty * 4 + i];
#pragma unroll
            for (int j = 0; j < 4; ++j) b[j] = Bs[kk][tx * 4 + j];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int64_t gm = m0 + ty * 4 + i;
        if (gm >= M) continue;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int64_t gn = n0 + tx * 4 + j;
            if (gn >= N) continue;
            if (gn < n_split) out0[gm * ld0 + gn] = acc[i][j];
            else out1[gm * ld1 + (gn - n_split)] = acc[i][j];
        }
    }
}

}  // namespace

cudaError_t gemm_simple_launch(const void* X, bool x_f32, const uint16_t* W, int64_t M, int64_t N,
                               int64_t Kd, float* out0, int64_t ld0, int64_t n_split, float* out1,
                               int64_t ld1, cudaStream_t stream) {
    if (M <= 0 || N <= 0) return cudaSuccess;
    dim3 grid(unsigned((N + BN - 1) / BN), unsigned((M + BM - 1) / BM));
    if (x_f32)
        gemm_nt_simple<float><<<grid, 256, 0, stream>>>(static_cast<const float*>(X), W, M, N, Kd,
                                                        out0, ld0, n_split, out1, ld1);
    else
        gemm_nt_simple<uint16_t><<<grid, 256, 0, stream>>>(static_cast<const uint16_t*>(X), W, M, N,
                                                           Kd, out0, ld0, n_split, out1, ld1);
    return cudaGetLastError();
}

}  // namespace df2
