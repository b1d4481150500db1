// Grouped dynamic causal conv, applied inside anchor blocks.
//
//   y[p, c] = sum_{j < taps, t-j >= 0} (base[j, c] + dyn[p, j, c/g]) * x[p-j, c],  t = p mod B
//
// (verl-SpeCo PR #62, "What DFlash2 adds": Conv_k(x)_t = k_{t,0} x_t + k_{t,1} x_{t-1},
// a fixed kernel per channel with a correction common to a group of conv_group_size
// channels added;
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
#include "tc_ptx.cuh"

namespace df2 {

namespace {

// Two floats to a packed bf16x2 (lo in the low half), rounded to nearest even by the
// hardware conversion: the same bits as f32_to_bf16_rn for finite values, in one
// instruction for two elements.
__device__ __forceinline__ uint32_t pack_bf16x2_rn(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

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
    static __device__ __forceinline__ float round(float f) { return bf16_to_f32(f32_to_bf16_rn(f)); }
    static __device__ __forceinline__ void store(uint16_t* p, const float f[8]) {
        uint4 w;
        w.x = pack_bf16x2_rn(f[0], f[1]);
        w.y = pack_bf16x2_rn(f[2], f[3]);
        w.z = pack_bf16x2_rn(f[4], f[5]);
        w.w = pack_bf16x2_rn(f[6], f[7]);
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
    static __device__ __forceinline__ float round(float f) { return f; }
    static __device__ __forceinline__ void store(float* p, const float f[4]) {
        *reinterpret_cast<float4*>(p) = make_float4(f[0], f[1], f[2], f[3]);
    }
};

// The residual stream added to a conv output: the output rounded to T first, the
// sum rounded again by the store, so the result equals the conv's stored output
// followed by a separate elementwise add in T.
template <typename T>
__device__ __forceinline__ void add_residual_raw(float acc[], const typename Vec<T>::Raw& raw) {
    constexpr int N = Vec<T>::N;
    float rv[N];
    Vec<T>::widen(raw, rv);
#pragma unroll
    for (int e = 0; e < N; ++e) acc[e] = Vec<T>::round(acc[e]) + rv[e];
}
template <typename T>
__device__ __forceinline__ void add_residual(float acc[], const T* __restrict__ res) {
    add_residual_raw<T>(acc, Vec<T>::load_raw(res));
}

// TAPS > 0: taps known at compile time, history in registers.  TAPS == 0: any
// taps; earlier rows are re-read through L1/L2.
template <typename T, int TAPS>
__global__ void __launch_bounds__(256)
conv_apply_kernel(const T* __restrict__ x, int64_t nblocks, int C, int B, int taps, int g, int G,
                  const float* __restrict__ base, const float* __restrict__ dyn, int64_t dyn_ld,
                  const T* __restrict__ res, T* __restrict__ y) {
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

    if constexpr (TAPS > 0) {
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
                if (res) add_residual<T>(acc, res + p * C + c0);
                Vec<T>::store(y + p * C + c0, acc);
            }
        }
    } else {
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
            if (res) add_residual<T>(acc, res + p * C + c0);
            Vec<T>::store(y + p * C + c0, acc);
        }
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

template <typename T, int TAPS, bool RES>
__global__ void __launch_bounds__(kAsyncThreads)
conv_apply_async_kernel(const T* __restrict__ x, int64_t nblocks, int C, int B, int g, int G, int strips,
                        const float* __restrict__ base, const float* __restrict__ dyn, int64_t dyn_ld,
                        const T* __restrict__ res, T* __restrict__ y) {
    constexpr int N = Vec<T>::N;
    using Raw = typename Vec<T>::Raw;
    extern __shared__ __align__(16) uint8_t smem[];
    const int nt = blockDim.x;
    uint8_t* xs = smem;                                                // [B][nt][16 B]
    uint8_t* rs = smem + size_t(B) * nt * 16;                          // RES: [B][nt][16 B]
    float* ds = reinterpret_cast<float*>(rs + (RES ? size_t(B) * nt * 16 : 0));  // [B][TAPS][nt]
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
        if (RES) cp_async16_c(rs + (size_t(t) * nt + tid) * 16, res + p * C + c0);
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
        Vec<T>::widen(*reinterpret_cast<const Raw*>(xs + (size_t(t) * nt + tid) * 16), hist[0]);
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
        if (RES) add_residual_raw<T>(acc, *reinterpret_cast<const Raw*>(rs + (size_t(t) * nt + tid) * 16));
        Vec<T>::store(y + p * C + c0, acc);
    }
}

// Pipelined apply for many rows.  An item is one anchor block times one strip of
// nt 16-byte channel chunks (a chunk inside one group).  Persistent CTAs take items
// blockIdx.x, + gridDim.x, ... through a ring of `stages` shared buffers.  A
// producer warp (the CTA's last) fetches an item's B rows of x (and of the
// residual) and the strip's corrections of every row and tap with 1-D bulk copies,
// a few large copies per item shared among its lanes and completing on the
// buffer's full barrier; the nt compute threads wait only for that barrier,
// compute the item with conv_apply_async_kernel's arithmetic, and release the
// buffer on its empty barrier.  No barrier spans the CTA inside the loop, so a
// slow thread holds up no other.  Every wait is bounded: a thread that gives up
// raises the CTA's abort flag and stops; the producer then waits, again bounded,
// for the copies it still has in flight.
struct BulkPlan {
    int nt = 0;         // compute threads per CTA (chunks per strip)
    int strips = 0;
    int stages = 0;
    uint32_t buf = 0;   // bytes per buffer
    uint32_t smem = 0;  // the buffers and their barriers
};

constexpr int kBulkMaxStages = 4;

template <typename T>
BulkPlan bulk_plan(int C, int B, int taps, int g, int G, int64_t dyn_ld, bool res) {
    BulkPlan pl;
    constexpr int N = Vec<T>::N;
    const int chunks = C / N;
    if (taps > 4 || g % N != 0 || G % 4 != 0 || dyn_ld % 4 != 0) return pl;
    // a strip of at least 128 chunks if one fits (up to 256, dividing the row), with
    // a ring of four to two buffers that fits twice on an SM, preferring more
    // buffers; narrower strips only when no such strip fits
    for (int min_nt : {128, 64})
    for (int stages = kBulkMaxStages; stages >= 2; --stages)
        for (int nt = 256; nt >= min_nt; nt -= 32) {
            if (chunks % nt != 0) continue;
            const int ngrp = nt * N / g;
            if (ngrp % 4 != 0) continue;
            const uint32_t row = uint32_t(nt) * 16;
            const uint32_t buf =
                (uint32_t(B) * row * (res ? 2u : 1u) + uint32_t(B) * taps * ngrp * 4 + 127) / 128 * 128;
            if (stages * buf + 128 > 110 * 1024) continue;
            pl.nt = nt;
            pl.strips = chunks / nt;
            pl.stages = stages;
            pl.buf = buf;
            pl.smem = stages * buf + 128;
            return pl;
        }
    return pl;
}

template <typename T, int TAPS, bool RES>
__global__ void __launch_bounds__(288)
conv_apply_bulk_kernel(const T* __restrict__ x, int64_t n_items, int C, int B, int g, int G, int strips,
                       int stages, uint32_t buf_bytes, const float* __restrict__ base, const float* __restrict__ dyn,
                       int64_t dyn_ld, const T* __restrict__ res, T* __restrict__ y) {
    constexpr int N = Vec<T>::N;
    using Raw = typename Vec<T>::Raw;
    extern __shared__ __align__(16) uint8_t smem[];
    const int nt = blockDim.x - 32, tid = threadIdx.x;
    const int ngrp = nt * N / g;
    const uint32_t row = uint32_t(nt) * 16;
    const uint32_t xbytes = uint32_t(B) * row;
    const uint32_t rbytes = RES ? xbytes : 0u;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + size_t(stages) * buf_bytes);
    uint64_t* empty = full + kBulkMaxStages;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + kBulkMaxStages);
    if (tid == 0) {
        for (int s = 0; s < stages; ++s) {
            tc::mbar_init(&full[s], 1);
            tc::mbar_init(&empty[s], uint32_t(nt));
        }
        *abort_flag = 0;
        tc::fence_mbar_init();
    }
    __syncthreads();
    const int64_t stride = gridDim.x;
    const int64_t n_mine = blockIdx.x < n_items ? (n_items - blockIdx.x + stride - 1) / stride : 0;
    if (tid >= nt) {
        // ---------------------------------------------------------------- producer
        const int lane = tid - nt;
        const uint64_t pol = tc::l2_policy_evict_first();  // every byte is read once
        const int per_row = (RES ? 2 : 1) + TAPS;
        int64_t k = 0;
        for (; k < n_mine; ++k) {
            const int s = int(k % stages);
            if (k >= stages) {
                const bool got = tc::mbar_wait(&empty[s], uint32_t((k / stages - 1) & 1), abort_flag);
                if (!__all_sync(kFull, got)) break;
            }
            const int64_t item = blockIdx.x + k * stride;
            const int64_t nb = item / strips;
            const int c0 = int(item - nb * strips) * nt * N;
            const int grp0 = c0 / g;
            uint8_t* buf = smem + size_t(s) * buf_bytes;
            if (lane == 0) tc::mbar_arrive_expect_tx(&full[s], xbytes + rbytes + uint32_t(B) * TAPS * ngrp * 4);
            __syncwarp();
            for (int e = lane; e < B * per_row; e += 32) {
                const int t = e / per_row, kind = e - t * per_row;
                const int64_t p = nb * B + t;
                if (kind == 0) {
                    tc::bulk_load(buf + size_t(t) * row, x + p * C + c0, row, &full[s], pol);
                } else if (RES && kind == 1) {
                    tc::bulk_load(buf + xbytes + size_t(t) * row, res + p * C + c0, row, &full[s], pol);
                } else {
                    const int j = kind - (RES ? 2 : 1);
                    tc::bulk_load(buf + xbytes + rbytes + (size_t(t) * TAPS + j) * ngrp * 4,
                                  dyn + p * dyn_ld + j * G + grp0, uint32_t(ngrp) * 4, &full[s], pol);
                }
            }
        }
        if (lane == 0 && *abort_flag) {
            // wait (bounded) for the copies issued but not consumed: the last
            // `stages` items issued
            volatile int never = 0;
            for (int64_t kk = k - 1; kk >= 0 && kk >= k - stages; --kk)
                tc::mbar_wait(&full[kk % stages], uint32_t((kk / stages) & 1), &never);
        }
        return;
    }
    // -------------------------------------------------------------------- compute
    const int gl = (tid * N) / g;
    for (int64_t k = 0; k < n_mine; ++k) {
        const int s = int(k % stages);
        if (!tc::mbar_wait(&full[s], uint32_t((k / stages) & 1), abort_flag)) break;
        const int64_t item = blockIdx.x + k * stride;
        const int64_t nb = item / strips;
        const int c0 = int(item - nb * strips) * nt * N + tid * N;
        const uint8_t* buf = smem + size_t(s) * buf_bytes;
        const float* ds = reinterpret_cast<const float*>(buf + xbytes + rbytes);
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
            Vec<T>::widen(*reinterpret_cast<const Raw*>(buf + size_t(t) * row + size_t(tid) * 16), hist[0]);
            float acc[N];
#pragma unroll
            for (int e = 0; e < N; ++e) acc[e] = 0.f;
#pragma unroll
            for (int j = 0; j < TAPS; ++j) {
                if (j > t) break;
                const float d = ds[(size_t(t) * TAPS + j) * ngrp + gl];
#pragma unroll
                for (int e = 0; e < N; ++e) acc[e] = fmaf(kb[j][e] + d, hist[j][e], acc[e]);
            }
            if (RES)
                add_residual_raw<T>(acc, *reinterpret_cast<const Raw*>(buf + xbytes + size_t(t) * row +
                                                                      size_t(tid) * 16));
            Vec<T>::store(y + p * C + c0, acc);
        }
        tc::mbar_arrive(&empty[s]);  // this thread is done with the buffer
    }
}

// Few rows: one thread per (row, 16-byte channel chunk); the taps re-read the
// previous rows (from L1/L2) so every thread has at most `taps` independent loads.
template <typename T>
__global__ void __launch_bounds__(256)
conv_apply_rows_kernel(const T* __restrict__ x, int64_t P, int C, int B, int taps, int g, int G,
                       const float* __restrict__ base, const float* __restrict__ dyn, int64_t dyn_ld,
                       const T* __restrict__ res, T* __restrict__ y) {
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
    if (res) add_residual<T>(acc, res + p * C + c0);
    Vec<T>::store(y + p * C + c0, acc);
}

template <typename T>
cudaError_t launch_t(const T* x, int64_t P, int C, int B, int taps, int g, const float* base,
                     const float* dyn, int64_t dyn_ld, const T* res, T* y, cudaStream_t stream) {
    const int64_t nblocks = P / B;
    const int64_t total = nblocks * (C / Vec<T>::N);
    if (total == 0) return cudaSuccess;
    const int G = C / g;
    if (total < 32768) {
        // too few (block, chunk) pairs to fill the GPU: spread the rows instead
        const int64_t rows_total = P * (C / Vec<T>::N);
        conv_apply_rows_kernel<T><<<unsigned((rows_total + 255) / 256), 256, 0, stream>>>(
            x, P, C, B, taps, g, G, base, dyn, dyn_ld, res, y);
        note_launch();
        return cudaGetLastError();
    }
    {
        const BulkPlan bp = bulk_plan<T>(C, B, taps, g, G, dyn_ld, res != nullptr);
        if (bp.nt > 0) {
            const int64_t n_items = nblocks * bp.strips;
            cudaError_t e = cudaSuccess;
            int dev = 0, sms = 0, per_sm = 0;
#define DF2_BULK(TP, R)                                                                                     \
    do {                                                                                                    \
        auto kern = conv_apply_bulk_kernel<T, TP, R>;                                                       \
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(bp.smem));         \
        if (e != cudaSuccess) return e;                                                                    \
        e = cudaGetDevice(&dev);                                                                           \
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);        \
        if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, bp.nt + 32, bp.smem); \
        if (e != cudaSuccess) return e;                                                                    \
        const int64_t grid = n_items < int64_t(sms) * per_sm ? n_items : int64_t(sms) * per_sm;           \
        kern<<<unsigned(grid > 0 ? grid : 1), bp.nt + 32, bp.smem, stream>>>(x, n_items, C, B, g, G, bp.strips, \
                                                                          bp.stages, bp.buf, base, dyn, dyn_ld, \
                                                                          res, y);                              \
    } while (0)
#define DF2_BULK_T(TP)                 \
    do {                               \
        if (res) DF2_BULK(TP, true);   \
        else DF2_BULK(TP, false);      \
    } while (0)
            switch (taps) {
                case 1: DF2_BULK_T(1); break;
                case 2: DF2_BULK_T(2); break;
                case 3: DF2_BULK_T(3); break;
                default: DF2_BULK_T(4); break;
            }
#undef DF2_BULK_T
#undef DF2_BULK
            note_launch();
            return cudaGetLastError();
        }
    }
    // threads per CTA: a multiple of 32 that divides the row's chunks, so that no
    // strip of a block runs half empty (5120 channels: 640 chunks, 4 strips of 160)
    const int chunks = C / Vec<T>::N;
    int nt = kAsyncThreads;
    for (int cand = kAsyncThreads; cand >= 128; cand -= 32)
        if (chunks % cand == 0) { nt = cand; break; }
    const size_t slot = size_t(B) * ((res ? 32 : 16) + size_t(taps) * 4);  // bytes per thread
    while (nt > 64 && slot * nt > kAsyncSmemMax) nt /= 2;
    const size_t async_smem = slot * nt;
    if (taps <= 4 && async_smem <= kAsyncSmemMax) {
        const int strips = (C / Vec<T>::N + nt - 1) / nt;
        const unsigned agrid = unsigned(nblocks * strips);
        cudaError_t e = cudaSuccess;
#define DF2_CONVA_R(TP, R)                                                                                  \
    do {                                                                                                    \
        e = cudaFuncSetAttribute(conv_apply_async_kernel<T, TP, R>,                                         \
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, int(async_smem));            \
        if (e != cudaSuccess) return e;                                                                    \
        conv_apply_async_kernel<T, TP, R><<<agrid, nt, async_smem, stream>>>(                               \
            x, nblocks, C, B, g, G, strips, base, dyn, dyn_ld, res, y);                                    \
    } while (0)
#define DF2_CONVA(TP)                  \
    do {                               \
        if (res) DF2_CONVA_R(TP, true); \
        else DF2_CONVA_R(TP, false);    \
    } while (0)
        switch (taps) {
            case 1: DF2_CONVA(1); break;
            case 2: DF2_CONVA(2); break;
            case 3: DF2_CONVA(3); break;
            default: DF2_CONVA(4); break;
        }
#undef DF2_CONVA
#undef DF2_CONVA_R
        note_launch();
        return cudaGetLastError();
    }
    const unsigned grid = unsigned((total + 255) / 256);
#define DF2_CONV(TP)                                                                               \
    conv_apply_kernel<T, TP><<<grid, 256, 0, stream>>>(x, nblocks, C, B, taps, g, G, base, dyn,    \
                                                       dyn_ld, res, y)
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

// Few rows (P <= 64): the projection and the apply in one kernel.  CTA (gx, gy)
// owns channel groups [gx*gpc, gx*gpc + gpc) and rows [gy*PR, gy*PR + PR), PR a
// multiple of the block size so that no tap reaches outside the CTA's rows.  It
// stages its rows of x in shared memory and computes its groups' projection columns
// -- (io*taps + j)*G + gi for both sides io -- NC at a time: the CTA's 256 lanes
// split the C inputs into 8-element chunks, so each staged x element and each W
// element is read and widened once per column group, and every lane keeps NC x PG
// partial sums (64).  A reduce-scatter over the warp (recursive halving: 62
// shuffles leave each lane two of the 64 warp sums) and a sum over the 8 warps in
// shared memory finish the dot products.  The output-side columns go to dyn_out,
// the input-side ones stay in shared memory for the apply, which uses the
// arithmetic of conv_apply_rows_kernel.  One launch instead of two, and the
// input-side corrections never leave the chip.
__device__ __forceinline__ void cp_async16_p(void* smem_dst, const void* gmem_src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(
                     static_cast<uint32_t>(__cvta_generic_to_shared(smem_dst))),
                 "l"(gmem_src)
                 : "memory");
}
__device__ __forceinline__ void load8s(const uint16_t* p, float f[8]) {
    unpack8(*reinterpret_cast<const uint4*>(p), f);
}
__device__ __forceinline__ void load8s(const float* p, float f[8]) {
    const float4 a = *reinterpret_cast<const float4*>(p);
    const float4 b = *reinterpret_cast<const float4*>(p + 4);
    f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
    f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
}
__device__ __forceinline__ float to_f32(uint16_t v) { return bf16_to_f32(v); }
__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ void store1(uint16_t* p, float v) { *p = f32_to_bf16_rn(v); }
__device__ __forceinline__ void store1(float* p, float v) { *p = v; }

constexpr int kPrepThreads = 256;
constexpr int kPrepWarps = kPrepThreads / 32;
constexpr int kPrepSums = 64;  // partial sums per lane: columns x rows of one column group

// Sum v[0..64) over the warp; lane l returns the sums of entries 2l and 2l + 1.
// Each step halves the entries a lane holds: the lane keeps the half its bit of
// the step selects and adds the partner's copy of that half.
__device__ __forceinline__ float2 warp_reduce_scatter64(float (&v)[kPrepSums], int lane) {
#pragma unroll
    for (int step = 0; step < 5; ++step) {
        const int half = kPrepSums >> (step + 1);  // 32, 16, 8, 4, 2
        const int bit = 16 >> step;
        const bool upper = (lane & bit) != 0;
#pragma unroll
        for (int i = 0; i < half; ++i) {
            const float send = upper ? v[i] : v[i + half];
            const float keep = upper ? v[i + half] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, bit);
        }
    }
    return make_float2(v[0], v[1]);
}

template <int PG, typename T>
__global__ void __launch_bounds__(kPrepThreads, 1)
conv_prepare_rows_kernel(const T* __restrict__ x, int64_t P, int C, int B, int taps, int g, int G, int gpc,
                         int PR, const uint16_t* __restrict__ W, const float* __restrict__ base,
                         T* __restrict__ y, float* __restrict__ dyn_out) {
    constexpr int NC = kPrepSums / PG;  // columns per group
    extern __shared__ __align__(16) uint8_t smem[];
    T* xs = reinterpret_cast<T*>(smem);                                          // [PR][C]
    float* ds = reinterpret_cast<float*>(smem + size_t(PR) * C * sizeof(T));     // [PR][taps][gpc]
    float* red = ds + size_t(PR) * taps * gpc;                                   // [warps][64]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g0 = int(blockIdx.x) * gpc;
    const int ng = gpc < G - g0 ? gpc : G - g0;
    const int64_t m0 = int64_t(blockIdx.y) * PR;
    const int nm = int(P - m0 < PR ? P - m0 : PR);
    constexpr int kPer16 = 16 / int(sizeof(T));
    const int cpr = C / kPer16;
    for (int r = warp; r < nm; r += kPrepWarps)
        for (int c = lane; c < cpr; c += 32)
            cp_async16_p(xs + size_t(r) * C + c * kPer16, x + (m0 + r) * C + c * kPer16);
    asm volatile("cp.async.commit_group;" ::: "memory");

    const int k8 = C / 8;
    const int ncols = 2 * taps * ng;
    auto column = [&](int lc) {
        const int io = lc / (taps * ng), rem = lc % (taps * ng), j = rem / ng, gl = rem % ng;
        return int64_t(io * taps + j) * G + g0 + gl;
    };
    // this lane's chunks: c = c_first, c_first + 256, ...
    const int c_first = warp * 32 + lane;
    auto load_w = [&](uint4 (&w)[NC], int cg, int c) {
#pragma unroll
        for (int q = 0; q < NC; ++q) {
            const int lc = cg * NC + q;
            w[q] = (c < k8 && lc < ncols) ? __ldg(reinterpret_cast<const uint4*>(W + column(lc) * C) + c)
                                          : make_uint4(0, 0, 0, 0);
        }
    };
    uint4 wn[NC];
    load_w(wn, 0, c_first);  // the first chunk's W loads overlap the staging of x
    asm volatile("cp.async.wait_all;" ::: "memory");
    __syncthreads();

    for (int cg = 0; cg * NC < ncols; ++cg) {
        float acc[kPrepSums];  // [q][p]
#pragma unroll
        for (int i = 0; i < kPrepSums; ++i) acc[i] = 0.f;
        for (int c = c_first; c < k8; c += kPrepThreads) {
            float wf[NC][8];
#pragma unroll
            for (int q = 0; q < NC; ++q) unpack8(wn[q], wf[q]);
            // the next chunk's W (this group's, else the next group's first) is in
            // flight while this chunk is summed
            if (c + kPrepThreads < k8) load_w(wn, cg, c + kPrepThreads);
            else if ((cg + 1) * NC < ncols) load_w(wn, cg + 1, c_first);
#pragma unroll
            for (int p = 0; p < PG; ++p) {
                if (p < nm) {
                    float xf[8];
                    load8s(xs + size_t(p) * C + c * 8, xf);
#pragma unroll
                    for (int q = 0; q < NC; ++q)
#pragma unroll
                        for (int e = 0; e < 8; ++e) acc[q * PG + p] = fmaf(wf[q][e], xf[e], acc[q * PG + p]);
                }
            }
        }
        const float2 s2 = warp_reduce_scatter64(acc, lane);
        red[warp * kPrepSums + 2 * lane] = s2.x;
        red[warp * kPrepSums + 2 * lane + 1] = s2.y;
        __syncthreads();
        if (threadIdx.x < kPrepSums) {
            const int i = threadIdx.x, q = i / PG, p = i % PG, lc = cg * NC + q;
            float sum = 0.f;
#pragma unroll
            for (int w = 0; w < kPrepWarps; ++w) sum += red[w * kPrepSums + i];
            if (lc < ncols && p < nm) {
                const int io = lc / (taps * ng), rem = lc % (taps * ng), j = rem / ng, gl = rem % ng;
                if (io == 0) ds[(p * taps + j) * gpc + gl] = sum;
                else dyn_out[(m0 + p) * (int64_t(taps) * G) + int64_t(j) * G + g0 + gl] = sum;
            }
        }
        __syncthreads();  // red is reused by the next group
    }

    const int c_lo = g0 * g, nch = ng * g;
    for (int e = threadIdx.x; e < nm * nch; e += kPrepThreads) {
        const int r = e / nch, c = c_lo + e % nch;
        const int t = int((m0 + r) % B);
        float acc = 0.f;
        for (int j = 0; j < taps && j <= t; ++j) {
            const float k = __ldg(base + int64_t(j) * C + c) + ds[(r * taps + j) * gpc + (c / g - g0)];
            acc = fmaf(k, to_f32(xs[size_t(r - j) * C + c]), acc);
        }
        store1(y + (m0 + r) * C + c, acc);
    }
}

template <int PG, typename T>
cudaError_t launch_prepare_rows(const T* x, int64_t P, int C, int B, int taps, int g, int PR,
                                const uint16_t* W, const float* base, T* y, float* dyn_out,
                                cudaStream_t stream) {
    const int G = C / g;
    const int gpc = 2 * taps >= 8 ? 1 : 8 / (2 * taps);
    const size_t smem = size_t(PR) * C * sizeof(T) + size_t(PR) * taps * gpc * 4 +
                        size_t(kPrepWarps) * kPrepSums * 4;
    cudaError_t e = cudaFuncSetAttribute(conv_prepare_rows_kernel<PG, T>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (e != cudaSuccess) return e;
    const dim3 grid = dim3(static_cast<unsigned>((G + gpc - 1) / gpc), static_cast<unsigned>((P + PR - 1) / PR));
    conv_prepare_rows_kernel<PG, T><<<grid, kPrepThreads, smem, stream>>>(x, P, C, B, taps, g, G, gpc, PR, W,
                                                                          base, y, dyn_out);
    note_launch();
    return cudaGetLastError();
}

// Rows per CTA for the fused few-row path (a multiple of B, at most 16, its x
// rows within 160 KB of shared memory), or 0 when the path does not apply.
int prepare_rows_per_cta(int64_t P, int C, int B, int esz) {
    if (P > 64 || B > 16) return 0;
    const int pg = B <= 8 ? 8 : 16;
    const int pr = pg / B * B;
    if (size_t(pr) * C * esz + 4096 > 160 * 1024) return 0;
    return pr;
}

}  // namespace

cudaError_t conv_apply_launch(const void* x, bool f32, int64_t P, int C, int B, int taps, int g,
                              const float* base_io, const float* dyn, int64_t dyn_ld, void* y,
                              cudaStream_t stream, const void* res) {
    if (f32)
        return launch_t<float>(static_cast<const float*>(x), P, C, B, taps, g, base_io, dyn, dyn_ld,
                               static_cast<const float*>(res), static_cast<float*>(y), stream);
    return launch_t<uint16_t>(static_cast<const uint16_t*>(x), P, C, B, taps, g, base_io, dyn,
                              dyn_ld, static_cast<const uint16_t*>(res), static_cast<uint16_t*>(y), stream);
}

}  // namespace df2

namespace df2 {

bool conv_prepare_rows_supported(int64_t P, int C, int B, bool f32) {
    return prepare_rows_per_cta(P, C, B, f32 ? 4 : 2) > 0;
}

cudaError_t conv_prepare_rows_launch(const void* x, bool f32, int64_t P, int C, int B, int taps, int g,
                                     const uint16_t* W, const float* base, void* y, float* dyn_out,
                                     cudaStream_t stream) {
    const int pr = prepare_rows_per_cta(P, C, B, f32 ? 4 : 2);
    if (pr == 0) return cudaErrorInvalidValue;
    if (f32) {
        if (pr <= 8)
            return launch_prepare_rows<8, float>(static_cast<const float*>(x), P, C, B, taps, g, pr, W, base,
                                                 static_cast<float*>(y), dyn_out, stream);
        return launch_prepare_rows<16, float>(static_cast<const float*>(x), P, C, B, taps, g, pr, W, base,
                                              static_cast<float*>(y), dyn_out, stream);
    }
    if (pr <= 8)
        return launch_prepare_rows<8, uint16_t>(static_cast<const uint16_t*>(x), P, C, B, taps, g, pr, W, base,
                                                static_cast<uint16_t*>(y), dyn_out, stream);
    return launch_prepare_rows<16, uint16_t>(static_cast<const uint16_t*>(x), P, C, B, taps, g, pr, W, base,
                                             static_cast<uint16_t*>(y), dyn_out, stream);
}

}  // namespace df2
