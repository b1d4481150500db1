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

// Few rows of X: one warp per output column n (one row of W, read once with
// 16-byte loads), the PG rows of X copied to shared memory in their own dtype
// with one round of cp.async (every copy in flight at once).  Used when M is
// small, where the tiled kernel above would leave most SMs idle.
__device__ __forceinline__ void cp_async16_g(void* smem_dst, const void* gmem_src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(
                     static_cast<uint32_t>(__cvta_generic_to_shared(smem_dst))),
                 "l"(gmem_src)
                 : "memory");
}

__device__ __forceinline__ void load8(const uint16_t* p, float f[8]) {
    unpack8(*reinterpret_cast<const uint4*>(p), f);
}
__device__ __forceinline__ void load8(const float* p, float f[8]) {
    const float4 a = *reinterpret_cast<const float4*>(p);
    const float4 b = *reinterpret_cast<const float4*>(p + 4);
    f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
    f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
}

template <int PG, typename TX>
__global__ void __launch_bounds__(256)
gemm_rows_kernel(const TX* __restrict__ X, const uint16_t* __restrict__ W, int64_t M, int64_t N,
                 int64_t Kd, float* __restrict__ out0, int64_t ld0, int64_t n_split,
                 float* __restrict__ out1, int64_t ld1) {
    extern __shared__ __align__(16) uint8_t xs_raw[];
    TX* xs = reinterpret_cast<TX*>(xs_raw);  // [PG][Kd]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t m0 = int64_t(blockIdx.y) * PG;
    const int nm = int(dmin<int64_t>(PG, M - m0));
    constexpr int kPer16 = 16 / int(sizeof(TX));  // elements per 16-byte chunk
    const int64_t cpr = Kd / kPer16;               // chunks per row
    for (int64_t i = threadIdx.x; i < int64_t(nm) * cpr; i += 256) {
        const int p = int(i / cpr);
        const int64_t c = i - int64_t(p) * cpr;
        cp_async16_g(xs + size_t(p) * Kd + c * kPer16, X + (m0 + p) * Kd + c * kPer16);
    }
    for (int64_t i = int64_t(nm) * cpr + threadIdx.x; i < int64_t(PG) * cpr; i += 256)
        reinterpret_cast<uint4*>(xs)[i] = make_uint4(0, 0, 0, 0);
    asm volatile("cp.async.commit_group;\n\tcp.async.wait_all;" ::: "memory");
    __syncthreads();
    const int64_t k8 = Kd / 8;
    for (int64_t n = int64_t(blockIdx.x) * 8 + warp; n < N; n += int64_t(gridDim.x) * 8) {
        float acc[PG];
#pragma unroll
        for (int p = 0; p < PG; ++p) acc[p] = 0.f;
        const uint4* wrow = reinterpret_cast<const uint4*>(W + n * Kd);
#pragma unroll 8
        for (int64_t c = lane; c < k8; c += 32) {
            float wf[8];
            unpack8(__ldg(wrow + c), wf);
#pragma unroll
            for (int p = 0; p < PG; ++p) {
                float xf[8];
                load8(xs + size_t(p) * Kd + c * 8, xf);
#pragma unroll
                for (int e = 0; e < 8; ++e) acc[p] = fmaf(wf[e], xf[e], acc[p]);
            }
        }
        float mine = 0.f;
#pragma unroll
        for (int p = 0; p < PG; ++p) {
            const float s = warp_sum(acc[p]);
            if (lane == p) mine = s;
        }
        if (lane < nm) {
            const int64_t gm = m0 + lane;
            if (n < n_split) out0[gm * ld0 + n] = mine;
            else out1[gm * ld1 + (n - n_split)] = mine;
        }
    }
}

}  // namespace

cudaError_t gemm_rows_launch(const void* X, bool x_f32, const uint16_t* W, int64_t M, int64_t N,
                             int64_t Kd, float* out0, int64_t ld0, int64_t n_split, float* out1,
                             int64_t ld1, int num_sms, cudaStream_t stream) {
    if (M <= 0 || N <= 0) return cudaSuccess;
    const size_t esz = x_f32 ? 4 : 2;
    int pg = 8;
    while (pg > 1 && size_t(pg) * Kd * esz > 160 * 1024) pg /= 2;
    const size_t smem = size_t(pg) * Kd * esz;
    const int64_t groups = (M + pg - 1) / pg;
    int64_t gx = (N + 7) / 8;
    const int64_t want = (4LL * num_sms + groups - 1) / groups;
    if (gx > want) gx = want < 1 ? 1 : want;
    const dim3 grid = dim3(static_cast<unsigned>(gx), static_cast<unsigned>(groups));
    cudaError_t e = cudaSuccess;
#define DF2_ROWS(PGV, T)                                                                            \
    e = cudaFuncSetAttribute(gemm_rows_kernel<PGV, T>, cudaFuncAttributeMaxDynamicSharedMemorySize, \
                             int(smem));                                                            \
    if (e != cudaSuccess) return e;                                                                 \
    gemm_rows_kernel<PGV, T><<<grid, 256, smem, stream>>>(static_cast<const T*>(X), W, M, N, Kd,    \
                                                           out0, ld0, n_split, out1, ld1)
    if (x_f32) {
        if (pg == 8) { DF2_ROWS(8, float); } else if (pg == 4) { DF2_ROWS(4, float); }
        else if (pg == 2) { DF2_ROWS(2, float); } else { DF2_ROWS(1, float); }
    } else {
        if (pg == 8) { DF2_ROWS(8, uint16_t); } else if (pg == 4) { DF2_ROWS(4, uint16_t); }
        else if (pg == 2) { DF2_ROWS(2, uint16_t); } else { DF2_ROWS(1, uint16_t); }
    }
#undef DF2_ROWS
    note_launch();
    return cudaGetLastError();
}

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
    note_launch();
    return cudaGetLastError();
}

}  // namespace df2
