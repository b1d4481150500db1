// Grouped dynamic causal conv, applied inside anchor blocks.
//
//   y[p, c] = sum_{j < taps, t-j >= 0} (base[j, c] + dyn[p, j, c/g]) * x[p-j, c],  t = p mod B
//
// (verl-SpeCo PR #62, "What DFlash2 adds": Conv_k(x)_t = k_{t,0} x_t + k_{t,1} x_{t-1},
// static per-channel kernel plus a correction shared by conv_group_size channels;
// "Two deltas", item 1: no tap crosses an anchor-block boundary.)
//
// One thread owns 16 bytes of channels (8 bf16 or 4 fp32) of one anchor block and
// walks the block's B rows in order, keeping the last `taps` rows of x in
// registers, so every x element is read from HBM once and every load/store is a
// coalesced 16-byte access (consecutive threads take consecutive channel chunks
// of the same row).  The rows are loaded eight at a time so each thread has
// eight loads in flight.  The base kernel for the thread's channels is loaded once.
#include "common.cuh"
#include "kernels.h"

namespace df2 {

namespace {

template <typename T>
struct Vec;
template <>
struct Vec<uint16_t> {
    static constexpr int N = 8;
    using Raw = uint4;
    static __device__ __forceinline__ Raw load_raw(const uint16_t* p) {
        return __ldg(reinterpret_cast<const uint4*>(p));
    }
    static __device__ __forceinline__ void widen(const Raw& r, float f[8]) { unpack8(r, f); }
    static __device__ __forceinline__ void load(const uint16_t* p, float f[8]) {
        unpack8(__ldg(reinterpret_cast<const uint4*>(p)), f);
    }
    static __device__ __forceinline__ void store(uint16_t* p, const float f[8]) {
        uint4 w;
        w.x = uint32_t(f32_to_bf16_rn(f[0])) | (uint32_t(f32_to_bf16_rn(f[1])) << 16);
        w.y = uint32_t(f32_to_bf16_rn(f[2])) | (uint32_t(f32_to_bf16_rn(f[3])) << 16);
        w.z = uint32_t(f32_to_bf16_rn(f[4])) | (uint32_t(f32_to_bf16_rn(f[5])) << 16);
        w.w = uint32_t(f32_to_bf16_rn(f[6])) | (uint32_t(f32_to_bf16_rn(f[7])) << 16);
        *reinterpret_cast<uint4*>(p) = w;
    }
};
template <>
struct Vec<float> {
    static constexpr int N = 4;
    using Raw = float4;
    static __device__ __forceinline__ Raw load_raw(const float* p) {
        return __ldg(reinterpret_cast<const float4*>(p));
    }
    static __device__ __forceinline__ void widen(const Raw& r, float f[4]) {
        f[0] = r.x; f[1] = r.y; f[2] = r.z; f[3] = r.w;
    }
    static __device__ __forceinline__ void load(const float* p, float f[4]) {
        const float4 v = __ldg(reinterpret_cast<const float4*>(p));
        f[0] = v.x; f[1] = v.y; f[2] = v.z; f[3] = v.w;
    }
    static __device__ __forceinline__ void store(float* p, const float f[4]) {
        *reinterpret_cast<float4*>(p) = make_float4(f[0], f[1], f[2], f[3]);
    }
};

// TAPS > 0: taps known at compile time, history in registers.  TAPS == 0: any
// taps; earlier rows are re-read through L1/L2.
template <typename T, int TAPS>
__global__ void __launch_bounds__(256)
conv_apply_kernel(const T* __restrict__ x, int64_t nblocks, int C, int B, int taps, int g, int G,
                  const float* __restrict__ base, const float* __restrict__ dyn, int64_t dyn_ld,
                  T* __restrict__ y) {
    constexpr int N = Vec<T>::N;
    const int chunks = C / N;
    const int64_t idx = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
    if (idx >= nblocks * chunks) return;
    const int64_t nb = idx / chunks;
    const int c0 = int(idx % chunks) * N;
    const bool shared_group = (g % N) == 0;  // all N channels in one group
    const int grp0 = c0 / g;

    constexpr int TR = TAPS > 0 ? TAPS : 1;
    float kb[TR][N];
    float hist[TR][N];
    if (TAPS > 0) {
#pragma unroll
        for (int j = 0; j < TR; ++j)
#pragma unroll
            for (int e = 0; e < N; ++e) {
                kb[j][e] = __ldg(base + int64_t(j) * C + c0 + e);
                hist[j][e] = 0.f;
            }
    }

    if (TAPS > 0) {
        // Rows are taken kGroup at a time: all of a group's loads (x and the dynamic
        // corrections) are issued before any is used, so each thread keeps kGroup
        // 16-byte loads in flight instead of one.
        constexpr int kGroup = 8;
        for (int t0 = 0; t0 < B; t0 += kGroup) {
            typename Vec<T>::Raw cur[kGroup];
            float dg[kGroup][TR];
#pragma unroll
            for (int u = 0; u < kGroup; ++u) {
                if (t0 + u < B) {
                    const int64_t p = nb * B + t0 + u;
                    cur[u] = Vec<T>::load_raw(x + p * C + c0);
                    if (shared_group) {
#pragma unroll
                        for (int j = 0; j < TR; ++j) dg[u][j] = __ldg(dyn + p * dyn_ld + j * G + grp0);
                    }
                }
            }
#pragma unroll
            for (int u = 0; u < kGroup; ++u) {
                const int t = t0 + u;
                if (t >= B) break;
                const int64_t p = nb * B + t;
                const float* drow = dyn + p * dyn_ld;
                float acc[N];
#pragma unroll
                for (int e = 0; e < N; ++e) acc[e] = 0.f;
#pragma unroll
                for (int j = TR - 1; j > 0; --j)
#pragma unroll
                    for (int e = 0; e < N; ++e) hist[j][e] = hist[j - 1][e];
                Vec<T>::widen(cur[u], hist[0]);
#pragma unroll
                for (int j = 0; j < TR; ++j) {
                    if (j > t) break;
                    if (shared_group) {
#pragma unroll
                        for (int e = 0; e < N; ++e) acc[e] = fmaf(kb[j][e] + dg[u][j], hist[j][e], acc[e]);
                    } else {
#pragma unroll
                        for (int e = 0; e < N; ++e) {
                            const float d = __ldg(drow + j * G + (c0 + e) / g);
                            acc[e] = fmaf(kb[j][e] + d, hist[j][e], acc[e]);
                        }
                    }
                }
                Vec<T>::store(y + p * C + c0, acc);
            }
        }
        return;
    }

    for (int t = 0; t < B; ++t) {
        const int64_t p = nb * B + t;
        float cur[N], acc[N];
        Vec<T>::load(x + p * C + c0, cur);
#pragma unroll
        for (int e = 0; e < N; ++e) acc[e] = 0.f;
        const float* drow = dyn + p * dyn_ld;
        for (int j = 0; j < taps && j <= t; ++j) {
            float xv[N];
            if (j == 0) {
#pragma unroll
                for (int e = 0; e < N; ++e) xv[e] = cur[e];
            } else {
                Vec<T>::load(x + (p - j) * C + c0, xv);
            }
#pragma unroll
            for (int e = 0; e < N; ++e) {
                const float d = __ldg(drow + j * G + (c0 + e) / g);
                const float k = __ldg(base + int64_t(j) * C + c0 + e) + d;
                acc[e] = fmaf(k, xv[e], acc[e]);
            }
        }
        Vec<T>::store(y + p * C + c0, acc);
    }
}

__device__ __forceinline__ void cp_async16_c(void* smem_dst, const void* gmem_src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(
                     static_cast<uint32_t>(__cvta_generic_to_shared(smem_dst))),
                 "l"(gmem_src)
                 : "memory");
}
__device__ __forceinline__ void cp_async4_c(void* smem_dst, const void* gmem_src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(
                     static_cast<uint32_t>(__cvta_generic_to_shared(smem_dst))),
                 "l"(gmem_src)
                 : "memory");
}

// Same arithmetic as conv_apply_kernel, but every thread first starts cp.async
// copies of its 16-byte chunk of all B rows (and, when a chunk lies inside one
// group, of its B x taps dynamic corrections) into its own shared-memory slots,
// then waits for them: the whole block's loads are in flight at once without
// holding registers.  A thread reads back only what it copied, so no barrier
// is needed.  Shared memory per CTA: B x threads x (16 + taps x 4) bytes; long
// blocks launch fewer threads per CTA so that several CTAs still fit on an SM.
constexpr int kAsyncThreads = 256;
constexpr size_t kAsyncSmemMax = 96 * 1024;

template <typename T, int TAPS>
__global__ void __launch_bounds__(kAsyncThreads)
conv_apply_async_kernel(const T* __restrict__ x, int64_t nblocks, int C, int B, int g, int G, int strips,
                        const float* __restrict__ base, const float* __restrict__ dyn, int64_t dyn_ld,
                        T* __restrict__ y) {
    constexpr int N = Vec<T>::N;
    extern __shared__ __align__(16) uint8_t smem[];
    const int nt = blockDim.x;
    uint8_t* xs = smem;                                                // [B][nt][16 B]
    float* ds = reinterpret_cast<float*>(smem + size_t(B) * nt * 16);  // [B][TAPS][nt]
    const int tid = threadIdx.x;
    const int64_t nb = blockIdx.x / strips;
    const int strip = int(blockIdx.x % strips);
    const int c0 = (strip * nt + tid) * N;
    if (nb >= nblocks || c0 >= C) return;
    const bool shared_group = (g % N) == 0;
    const int grp0 = c0 / g;
    for (int t = 0; t < B; ++t) {
        const int64_t p = nb * B + t;
        cp_async16_c(xs + (size_t(t) * nt + tid) * 16, x + p * C + c0);
        if (shared_group) {
#pragma unroll
            for (int j = 0; j < TAPS; ++j)
                cp_async4_c(ds + (size_t(t) * TAPS + j) * nt + tid, dyn + p * dyn_ld + j * G + grp0);
        }
    }
    asm volatile("cp.async.commit_group;\n\tcp.async.wait_all;" ::: "memory");

    float kb[TAPS][N], hist[TAPS][N];
#pragma unroll
    for (int j = 0; j < TAPS; ++j)
#pragma unroll
        for (int e = 0; e < N; ++e) {
            kb[j][e] = __ldg(base + int64_t(j) * C + c0 + e);
            hist[j][e] = 0.f;
        }
    for (int t = 0; t < B; ++t) {
        const int64_t p = nb * B + t;
#pragma unroll
        for (int j = TAPS - 1; j > 0; --j)
#pragma unroll
            for (int e = 0; e < N; ++e) hist[j][e] = hist[j - 1][e];
        Vec<T>::widen(*reinterpret_cast<const typename Vec<T>::Raw*>(xs + (size_t(t) * nt + tid) * 16), hist[0]);
        float acc[N];
#pragma unroll
        for (int e = 0; e < N; ++e) acc[e] = 0.f;
#pragma unroll
        for (int j = 0; j < TAPS; ++j) {
            if (j > t) break;
            if (shared_group) {
                const float d = ds[(size_t(t) * TAPS + j) * nt + tid];
#pragma unroll
                for (int e = 0; e < N; ++e) acc[e] = fmaf(kb[j][e] + d, hist[j][e], acc[e]);
            } else {
#pragma unroll
                for (int e = 0; e < N; ++e) {
                    const float d = __ldg(dyn + p * dyn_ld + j * G + (c0 + e) / g);
                    acc[e] = fmaf(kb[j][e] + d, hist[j][e], acc[e]);
                }
            }
        }
        Vec<T>::store(y + p * C + c0, acc);
    }
}

// Few rows: one thread per (row, 16-byte channel chunk); the taps re-read the
// previous rows (from L1/L2) so every thread has at most `taps` independent loads.
template <typename T>
__global__ void __launch_bounds__(256)
conv_apply_rows_kernel(const T* __restrict__ x, int64_t P, int C, int B, int taps, int g, int G,
                       const float* __restrict__ base, const float* __restrict__ dyn, int64_t dyn_ld,
                       T* __restrict__ y) {
    constexpr int N = Vec<T>::N;
    const int chunks = C / N;
    const int64_t idx = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
    if (idx >= P * chunks) return;
    const int64_t p = idx / chunks;
    const int c0 = int(idx % chunks) * N;
    const int t = int(p % B);
    const float* drow = dyn + p * dyn_ld;
    float acc[N];
#pragma unroll
    for (int e = 0; e < N; ++e) acc[e] = 0.f;
    for (int j = 0; j < taps && j <= t; ++j) {
        float xv[N];
        Vec<T>::load(x + (p - j) * C + c0, xv);
#pragma unroll
        for (int e = 0; e < N; ++e) {
            const float k = __ldg(base + int64_t(j) * C + c0 + e) + __ldg(drow + j * G + (c0 + e) / g);
            acc[e] = fmaf(k, xv[e], acc[e]);
        }
    }
    Vec<T>::store(y + p * C + c0, acc);
}

template <typename T>
cudaError_t launch_t(const T* x, int64_t P, int C, int B, int taps, int g, const float* base,
                     const float* dyn, int64_t dyn_ld, T* y, cudaStream_t stream) {
    const int64_t nblocks = P / B;
    const int64_t total = nblocks * (C / Vec<T>::N);
    if (total == 0) return cudaSuccess;
    const int G = C / g;
    if (total < 32768) {
        // too few (block, chunk) pairs to fill the GPU: spread the rows instead
        const int64_t rows_total = P * (C / Vec<T>::N);
        conv_apply_rows_kernel<T><<<unsigned((rows_total + 255) / 256), 256, 0, stream>>>(
            x, P, C, B, taps, g, G, base, dyn, dyn_ld, y);
        note_launch();
        return cudaGetLastError();
    }
    int nt = kAsyncThreads;
    const size_t slot = size_t(B) * (16 + size_t(taps) * 4);  // bytes per thread
    while (nt > 64 && slot * nt > kAsyncSmemMax) nt /= 2;
    const size_t async_smem = slot * nt;
    if (taps <= 4 && async_smem <= kAsyncSmemMax) {
        const int strips = (C / Vec<T>::N + nt - 1) / nt;
        const unsigned agrid = unsigned(nblocks * strips);
        cudaError_t e = cudaSuccess;
#define DF2_CONVA(TP)                                                                                       \
    do {                                                                                                    \
        e = cudaFuncSetAttribute(conv_apply_async_kernel<T, TP>, cudaFuncAttributeMaxDynamicSharedMemorySize, \
                                 int(async_smem));                                                         \
        if (e != cudaSuccess) return e;                                                                    \
        conv_apply_async_kernel<T, TP><<<agrid, nt, async_smem, stream>>>(                                  \
            x, nblocks, C, B, g, G, strips, base, dyn, dyn_ld, y);                                         \
    } while (0)
        switch (taps) {
            case 1: DF2_CONVA(1); break;
            case 2: DF2_CONVA(2); break;
            case 3: DF2_CONVA(3); break;
            default: DF2_CONVA(4); break;
        }
#undef DF2_CONVA
        note_launch();
        return cudaGetLastError();
    }
    const unsigned grid = unsigned((total + 255) / 256);
#define DF2_CONV(TP)                                                                               \
    conv_apply_kernel<T, TP><<<grid, 256, 0, stream>>>(x, nblocks, C, B, taps, g, G, base, dyn,    \
                                                       dyn_ld, y)
    switch (taps) {
        case 1: DF2_CONV(1); break;
        case 2: DF2_CONV(2); break;
        case 3: DF2_CONV(3); break;
        case 4: DF2_CONV(4); break;
        default: DF2_CONV(0); break;
    }
#undef DF2_CONV
    note_launch();
    return cudaGetLastError();
}

}  // namespace

cudaError_t conv_apply_launch(const void* x, bool f32, int64_t P, int C, int B, int taps, int g,
                              const float* base_io, const float* dyn, int64_t dyn_ld, void* y,
                              cudaStream_t stream) {
    if (f32)
        return launch_t<float>(static_cast<const float*>(x), P, C, B, taps, g, base_io, dyn, dyn_ld,
                               static_cast<float*>(y), stream);
    return launch_t<uint16_t>(static_cast<const uint16_t*>(x), P, C, B, taps, g, base_io, dyn,
                              dyn_ld, static_cast<uint16_t*>(y), stream);
}

}  // namespace df2
