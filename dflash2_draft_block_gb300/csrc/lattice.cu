// The lattice schedule of the candidate selector: every adjacent candidate pair
// scored in one parallel pass, then a sequential walk over the finished table
// ("DFlash 2 Explanation", "How It Works", Problem 1: the pair scores are computed
// together, and only the walk that reads them is serial, whether it takes the best
// successor or samples one from those scores).
//
// Table slot s = t-1 of request q (drafted position t = 1 .. B-1) holds
//   L[q][s][i][j] = vals[q,t,j] + sum_k A[a_i, k] * G[q,t,k] * Bc[ids[q,t,j], k]
// with a_i = ids[q, t-1, i] for t >= 2 and the anchor alone (row 0) for t = 1.
//
// lattice_kernel: one CTA per (request, slot, 16TM x 16TM output tile), 256
// threads as 16 x 16, each thread a TM x TM register tile.  The rank dimension
// streams through shared memory in chunks of 32: the gate rows x_i = A[a_i] (.) G_t
// are formed once per chunk in fp32, the successor rows y_j = Bc[b_j] are widened,
// both stored k-major so that a thread's TM x-values and TM y-values are
// contiguous.  The next chunk's gathers are issued into registers before the
// current chunk is consumed.
//
// lattice_walk_kernel: one warp per request; lane l owns a contiguous segment of
// each row so that a warp scan of the lanes' partial sums gives the CDF in
// candidate-list order.
#include "common.cuh"
#include "kernels.h"
#include "tc_ptx.cuh"

namespace df2 {

namespace {

constexpr int kLatThreads = 256;
constexpr int kLatChunk = 32;  // rank elements per shared-memory chunk

// 1 when the anchor and all candidate ids of rows 1 .. B-1 of request q are in [0, V).
__device__ bool lattice_request_valid(const int32_t* __restrict__ anchors, int64_t q, int B,
                                      const int32_t* __restrict__ ids, int K, int64_t V) {
    __shared__ int bad_s;
    if (threadIdx.x == 0) {
        const int32_t a = __ldg(anchors + q);
        bad_s = (a < 0 || a >= V) ? 1 : 0;
    }
    __syncthreads();
    const int64_t n = int64_t(B - 1) * K;
    const int32_t* base = ids + (q * B + 1) * K;
    int bad = 0;
    for (int64_t e = threadIdx.x; e < n; e += blockDim.x) {
        const int32_t b = __ldg(base + e);
        bad |= (b < 0 || b >= V);
    }
    if (__syncthreads_or(bad)) bad_s = 1;
    __syncthreads();
    return bad_s == 0;
}

// Gathers of one 8-element part of a chunk: A row pa, Bc row pb (bf16) and G_t at
// rank offset k; rows < 0 and offsets past r read as zero.
__device__ __forceinline__ void lattice_fetch(const uint16_t* __restrict__ A, const uint16_t* __restrict__ Bc,
                                              const float* __restrict__ Grow, int64_t pa, int64_t pb, int r,
                                              int k, uint4& ra, uint4& rb, float4& g0, float4& g1) {
    const bool in = k < r;
    const uint4 z4 = make_uint4(0, 0, 0, 0);
    const float4 zf = make_float4(0.f, 0.f, 0.f, 0.f);
    ra = (in && pa >= 0) ? __ldg(reinterpret_cast<const uint4*>(A + pa * r + k)) : z4;
    rb = (in && pb >= 0) ? __ldg(reinterpret_cast<const uint4*>(Bc + pb * r + k)) : z4;
    g0 = in ? __ldg(reinterpret_cast<const float4*>(Grow + k)) : zf;
    g1 = in ? __ldg(reinterpret_cast<const float4*>(Grow + k + 4)) : zf;
}

template <int TM>
__global__ void __launch_bounds__(kLatThreads)
lattice_kernel(const int32_t* __restrict__ anchors, int B, const int32_t* __restrict__ ids,
               const float* __restrict__ vals, const float* __restrict__ G,
               const uint16_t* __restrict__ A, const uint16_t* __restrict__ Bc, int64_t V, int K,
               int r, int tiles, float* __restrict__ lattice, int32_t* __restrict__ dev_status) {
    constexpr int TILE = 16 * TM;
    __shared__ __align__(16) float xs[kLatChunk][TILE + 4];
    __shared__ __align__(16) float ys[kLatChunk][TILE + 4];
    __shared__ int64_t pred_s[TILE];
    __shared__ int64_t cand_s[TILE];

    const int T = B - 1;
    int64_t blk = blockIdx.x;
    const int tj = int(blk % tiles);
    blk /= tiles;
    const int ti = int(blk % tiles);
    blk /= tiles;
    const int s = int(blk % T);
    const int64_t q = blk / T;
    const int t = s + 1;
    const int64_t row = q * B + t;  // the successor row (position t)
    const int i0 = ti * TILE, j0 = tj * TILE;
    const int tid = threadIdx.x;
    float* out = lattice + ((q * T + s) * int64_t(K)) * K;

    const bool valid = lattice_request_valid(anchors, q, B, ids, K, V);
    // rows that exist in this slot: all K, or the anchor's row 0 alone in slot 0
    const int rows_here = (s == 0) ? 1 : K;
    if (!valid || i0 >= rows_here) {
        for (int e = tid; e < TILE * TILE; e += kLatThreads) {
            const int i = i0 + e / TILE, j = j0 + e % TILE;
            if (i < K && j < K) out[int64_t(i) * K + j] = __int_as_float(0x7fc00000);
        }
        if (!valid && tid == 0 && s == 0 && ti == 0 && tj == 0 && dev_status)
            atomicOr(dev_status, DF2_STATUS_ID_OUT_OF_RANGE);
        return;
    }
    if (tid < TILE) {
        const int i = i0 + tid, j = j0 + tid;
        pred_s[tid] = (i < rows_here) ? (s == 0 ? int64_t(__ldg(anchors + q)) : int64_t(__ldg(ids + (row - 1) * K + i)))
                                      : int64_t(-1);
        cand_s[tid] = (j < K) ? int64_t(__ldg(ids + row * K + j)) : int64_t(-1);
    }
    __syncthreads();

    // loader mapping: thread -> (tile row lr, 8-element part lp) of a 32-wide chunk
    const int lr = tid >> 2, lp = tid & 3;
    const bool loader = lr < TILE;
    const int64_t pa = loader ? pred_s[lr] : -1;
    const int64_t pb = loader ? cand_s[lr] : -1;
    const float* Grow = G + row * r;

    uint4 ra = make_uint4(0, 0, 0, 0), rb = make_uint4(0, 0, 0, 0);
    float4 g0 = make_float4(0.f, 0.f, 0.f, 0.f), g1 = g0;

    const int ty = tid / 16, tx = tid % 16;
    float acc[TM][TM];
#pragma unroll
    for (int a = 0; a < TM; ++a)
#pragma unroll
        for (int b = 0; b < TM; ++b) acc[a][b] = 0.f;

    if (loader) lattice_fetch(A, Bc, Grow, pa, pb, r, lp * 8, ra, rb, g0, g1);
    for (int k0 = 0; k0 < r; k0 += kLatChunk) {
        __syncthreads();  // the previous chunk has been consumed
        if (loader) {
            float af[8], bf[8];
            unpack8(ra, af);
            unpack8(rb, bf);
            float* xc = &xs[lp * 8][lr];
            float* yc = &ys[lp * 8][lr];
            constexpr int ld = TILE + 4;
            xc[0 * ld] = af[0] * g0.x; xc[1 * ld] = af[1] * g0.y; xc[2 * ld] = af[2] * g0.z; xc[3 * ld] = af[3] * g0.w;
            xc[4 * ld] = af[4] * g1.x; xc[5 * ld] = af[5] * g1.y; xc[6 * ld] = af[6] * g1.z; xc[7 * ld] = af[7] * g1.w;
#pragma unroll
            for (int e = 0; e < 8; ++e) yc[e * ld] = bf[e];
        }
        __syncthreads();
        if (loader && k0 + kLatChunk < r)
            lattice_fetch(A, Bc, Grow, pa, pb, r, k0 + kLatChunk + lp * 8, ra, rb, g0, g1);
#pragma unroll 8
        for (int k = 0; k < kLatChunk; ++k) {
            float xv[TM], yv[TM];
#pragma unroll
            for (int a = 0; a < TM; ++a) xv[a] = xs[k][ty * TM + a];
#pragma unroll
            for (int b = 0; b < TM; ++b) yv[b] = ys[k][tx * TM + b];
#pragma unroll
            for (int a = 0; a < TM; ++a)
#pragma unroll
                for (int b = 0; b < TM; ++b) acc[a][b] = fmaf(xv[a], yv[b], acc[a][b]);
        }
    }

#pragma unroll
    for (int a = 0; a < TM; ++a) {
        const int i = i0 + ty * TM + a;
        if (i >= K) continue;
#pragma unroll
        for (int b = 0; b < TM; ++b) {
            const int j = j0 + tx * TM + b;
            if (j >= K) continue;
            out[int64_t(i) * K + j] = (i < rows_here) ? __ldg(vals + row * K + j) + acc[a][b]
                                                      : __int_as_float(0x7fc00000);
        }
    }
}

// ---------------------------------------------------------- tensor cores --
// lattice_tc_kernel (32 < K <= 64): one CTA of 256 threads per (request, slot).  The
// slot's table is a small GEMM, S = vals + X Y^T with X[i] = A[a_i] (.) G_t (fp32)
// and Y[j] = Bc[b_j] (bf16).  X is split into bf16 halves, x = hi + lo with
// lo = bf16(x - hi) (x - hi is exact in fp32; hi + lo is within 2^-17 of x), and
// the halves are stacked as the 128 rows of one tcgen05 MMA: rows 0..63 hi, rows
// 64..127 lo, N = K rounded up to 16 candidate rows, fp32 accumulation in TMEM.
// Row i + 64 of the result is added to row i in the epilogue, so one M = 128 MMA
// per 16-wide step covers both halves with no wasted rows.  The rank dimension
// goes through shared memory in 64-wide slices (one 128-byte swizzle row per
// operand row): the threads issue every gather of slice c + 1 before they wait for
// the tensor core to finish slice c (an mbarrier), then form the slice (the
// product with G, the split, the writes in the swizzled K-major layout).  What
// hides the gathers' latency is the CTAs sharing an SM: the launch bound holds a
// thread to 48 registers so that five fit (62 registers allowed four: 136.5 ->
// 133.0 us at 256 requests x 15 slots, K 64, r 512; six, at 40 registers, spill
// and took 141.7 us).  Waits are bounded.
constexpr int kLtcThreads = 256;
constexpr int kLtcCtasPerSm = 5;
constexpr int kLtcMaxK = 64;
constexpr uint32_t kLtcA = 128 * 128;            // A slice: 128 rows x 128 bytes
constexpr uint32_t kLtcB = kLtcMaxK * 128;       // B slice: up to 64 rows x 128 bytes
constexpr uint32_t kLtcBuf = kLtcA + kLtcB;      // 24 KB, a multiple of 1024

__device__ __forceinline__ uint32_t ltc_pack(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// 16-byte chunk cc of operand row `row` in a 128-byte-swizzled K-major slice.
__device__ __forceinline__ uint4* ltc_chunk(uint8_t* base, int row, int cc) {
    return reinterpret_cast<uint4*>(base + size_t(row) * 128 + size_t((cc ^ (row & 7)) * 16));
}

__global__ void __launch_bounds__(kLtcThreads, kLtcCtasPerSm)
lattice_tc_kernel(const int32_t* __restrict__ anchors, int B, const int32_t* __restrict__ ids,
                  const float* __restrict__ vals, const float* __restrict__ G,
                  const uint16_t* __restrict__ A, const uint16_t* __restrict__ Bc, int64_t V, int K, int r,
                  float* __restrict__ lattice, int32_t* __restrict__ dev_status) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kLtcBuf);  // [0] the slice's MMAs, [2] all MMAs
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + 3);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
    const int T = B - 1;
    const int s = int(blockIdx.x % T);
    const int64_t q = blockIdx.x / T;
    const int t = s + 1;
    const int64_t row = q * B + t;  // the successor row (position t)
    const int tid = threadIdx.x, warp = tid >> 5;
    float* out = lattice + ((q * T + s) * int64_t(K)) * K;
    const int NP = (K + 15) / 16 * 16;
    const int rows_here = (s == 0) ? 1 : K;

    const bool valid = lattice_request_valid(anchors, q, B, ids, K, V);
    if (!valid) {
        for (int e = tid; e < K * K; e += kLtcThreads) out[e] = __int_as_float(0x7fc00000);
        if (tid == 0 && s == 0 && dev_status) atomicOr(dev_status, DF2_STATUS_ID_OUT_OF_RANGE);
        return;
    }
    if (tid == 0) {
        tc::mbar_init(&bars[0], 1);
        tc::mbar_init(&bars[1], 1);
        tc::mbar_init(&bars[2], 1);
        *abort_flag = 0;
        tc::fence_mbar_init();
    }
    if (warp == 0) {
        tc::tmem_alloc(tmem_holder, 64);
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_holder;

    // every thread forms two 16-byte chunks of one predecessor row (hi row and lo
    // row) and two of one candidate row: row tid / 4, chunks 2 (tid % 4) and + 1
    const int my = tid >> 2;
    const int cc0 = (tid & 3) * 2;
    const int64_t src_a = my < rows_here ? (s == 0 ? int64_t(__ldg(anchors + q)) : int64_t(__ldg(ids + (row - 1) * K + my)))
                                         : int64_t(-1);
    const int64_t src_b = my < K ? int64_t(__ldg(ids + row * K + my)) : int64_t(-1);
    const float* Grow = G + row * r;
    // the whole gathered row into L2 at once (one contiguous stream per row), so the
    // slices' 128-byte pieces of it hit L2 instead of being separate DRAM accesses
    if ((tid & 3) == 0) {
        if (src_a >= 0) tc::bulk_prefetch_l2(A + src_a * r, uint32_t(r) * 2);
        if (src_b >= 0) tc::bulk_prefetch_l2(Bc + src_b * r, uint32_t(r) * 2);
    }
    const uint32_t idesc = tc::idesc_bf16_f32(128, NP);
    const int nsl = (r + 63) / 64;
    uint32_t ph[1] = {0u};
    bool ok = true;
    for (int c = 0; c < nsl; ++c) {
        const int k0 = c * 64;
        // every load of this thread's part of the slice first, into registers
        uint4 ra[2], rb[2];
        float4 gv[4];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int k = k0 + (cc0 + u) * 8;
            const bool in = k < r;
            ra[u] = (in && src_a >= 0) ? __ldg(reinterpret_cast<const uint4*>(A + src_a * r + k)) : make_uint4(0, 0, 0, 0);
            rb[u] = (in && src_b >= 0) ? __ldg(reinterpret_cast<const uint4*>(Bc + src_b * r + k)) : make_uint4(0, 0, 0, 0);
            gv[2 * u] = in ? __ldg(reinterpret_cast<const float4*>(Grow + k)) : make_float4(0.f, 0.f, 0.f, 0.f);
            gv[2 * u + 1] = in ? __ldg(reinterpret_cast<const float4*>(Grow + k + 4)) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        if (c >= 1) {
            // the MMAs that read the buffer for the previous slice are done (a slice's
            // MMAs take a small fraction of the time its gathers do)
            const bool got = tc::mbar_wait(&bars[0], ph[0], abort_flag);
            ph[0] ^= 1u;
            if (__syncthreads_or(!got)) { ok = false; break; }
        }
        uint8_t* bufA = smem;
        uint8_t* bufB = bufA + kLtcA;
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            float af[8];
            unpack8(ra[u], af);
            const float g8[8] = {gv[2 * u].x, gv[2 * u].y, gv[2 * u].z, gv[2 * u].w,
                                 gv[2 * u + 1].x, gv[2 * u + 1].y, gv[2 * u + 1].z, gv[2 * u + 1].w};
            uint32_t hi[4], lo[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float x0 = af[2 * e] * g8[2 * e], x1 = af[2 * e + 1] * g8[2 * e + 1];
                hi[e] = ltc_pack(x0, x1);  // nearest-even, as the split needs
                lo[e] = ltc_pack(x0 - bf16_lo(hi[e]), x1 - bf16_hi(hi[e]));
            }
            *ltc_chunk(bufA, my, cc0 + u) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
            *ltc_chunk(bufA, my + 64, cc0 + u) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
            if (my < NP) *ltc_chunk(bufB, my, cc0 + u) = rb[u];
        }
        // the generic-proxy writes above become visible to the tensor core's reads
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        tc::fence_before_sync();
        __syncthreads();
        if (tid == 0) {
            tc::fence_after_sync();
            const uint32_t a0 = tc::smem_u32(bufA), b0 = tc::smem_u32(bufB);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                tc::mma_bf16(tmem, tc::sw128_kmajor_desc(a0 + 32 * kk), tc::sw128_kmajor_desc(b0 + 32 * kk), idesc,
                             (c | kk) != 0 ? 1u : 0u);
            tc::mma_commit(&bars[0]);
        }
    }
    if (tid == 0) tc::mma_commit(&bars[2]);
    {
        volatile int never = 0;
        const bool done = tc::mbar_wait(&bars[2], 0, ok ? abort_flag : &never);
        if (!done) ok = false;
    }
    ok = !__syncthreads_or(!ok);
    tc::fence_after_sync();
    // the accumulator -> shared memory (the slice buffer is free): warps 2-3 (TMEM
    // lanes 64..127, the lo rows) store theirs, then warps 0-1 add their hi rows in
    // place, then every thread writes the table with consecutive threads on
    // consecutive columns
    float* red = reinterpret_cast<float*>(smem);  // [64][kLtcMaxK + 1]
    constexpr int ld = kLtcMaxK + 1;
    if (ok && (warp == 2 || warp == 3)) {
        for (int c0 = 0; c0 < NP; c0 += 16) {
            float v[16];
            tc::tmem_ld16(tmem + (uint32_t(warp * 32) << 16) + uint32_t(c0), v);
#pragma unroll
            for (int e = 0; e < 16; ++e) red[size_t(tid - 64) * ld + c0 + e] = v[e];
        }
    }
    __syncthreads();
    if (ok && warp < 2) {
        for (int c0 = 0; c0 < NP; c0 += 16) {
            float v[16];
            tc::tmem_ld16(tmem + (uint32_t(warp * 32) << 16) + uint32_t(c0), v);
#pragma unroll
            for (int e = 0; e < 16; ++e) red[size_t(tid) * ld + c0 + e] = v[e] + red[size_t(tid) * ld + c0 + e];
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    if (ok) {
        for (int e = tid; e < K * K; e += kLtcThreads) {
            const int i = e / K, j = e - i * K;
            out[e] = i < rows_here ? __ldg(vals + row * K + j) + red[size_t(i) * ld + j] : __int_as_float(0x7fc00000);
        }
    } else if (tid == 0 && dev_status) {
        atomicOr(dev_status, DF2_STATUS_WAIT_TIMEOUT);
    }
    if (warp == 0) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, 64);
    }
}

constexpr int kWalkWarps = 4;

// Warp-wide best by (value desc, token id asc); returns the winning column.
__device__ __forceinline__ int warp_best(float v, int id, int j) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, v, off);
        const int oid = __shfl_xor_sync(0xffffffffu, id, off);
        const int oj = __shfl_xor_sync(0xffffffffu, j, off);
        if (oj >= 0 && (j < 0 || ov > v || (ov == v && (oid < id || (oid == id && oj < j))))) {
            v = ov;
            id = oid;
            j = oj;
        }
    }
    return j;
}

__global__ void __launch_bounds__(kWalkWarps * 32)
lattice_walk_kernel(const float* __restrict__ lattice, const int32_t* __restrict__ ids, int R, int B,
                    int K, int64_t V, const float* __restrict__ uniforms, float temperature,
                    int32_t* __restrict__ path, float* __restrict__ path_scores,
                    int32_t* __restrict__ dev_status) {
    const int lane = threadIdx.x & 31;
    const int64_t q = int64_t(blockIdx.x) * kWalkWarps + (threadIdx.x >> 5);
    if (q >= R) return;
    const int T = B - 1;
    int bad = 0;
    for (int64_t e = lane; e < int64_t(T) * K; e += 32) {
        const int32_t b = __ldg(ids + (q * B + 1) * K + e);
        bad |= (b < 0 || b >= V);
    }
    if (__any_sync(0xffffffffu, bad)) {
        for (int t = lane; t < T; t += 32) {
            path[q * T + t] = -1;
            path_scores[q * T + t] = __int_as_float(0x7fc00000);
        }
        if (lane == 0 && dev_status) atomicOr(dev_status, DF2_STATUS_ID_OUT_OF_RANGE);
        return;
    }
    const int per = (K + 31) / 32;
    const int jb = dmin(K, lane * per), je = dmin(K, jb + per);
    int i = 0;
    for (int s = 0; s < T; ++s) {
        const int32_t* cand = ids + (q * B + s + 1) * K;
        const float* L = lattice + ((q * T + s) * int64_t(K) + i) * K;
        int pick;
        if (uniforms == nullptr) {
            float bv = 0.f;
            int bid = 0, bj = -1;
            for (int j = jb; j < je; ++j) {
                const float v = L[j];
                const int id = __ldg(cand + j);
                if (bj < 0 || v > bv || (v == bv && id < bid)) {
                    bv = v;
                    bid = id;
                    bj = j;
                }
            }
            pick = warp_best(bv, bid, bj);
        } else {
            float mx = -INFINITY;
            for (int j = jb; j < je; ++j) mx = fmaxf(mx, L[j]);
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
            float seg = 0.f;
            for (int j = jb; j < je; ++j) seg += expf((L[j] - mx) / temperature);
            // exclusive scan of the lanes' sums: the CDF before this lane's segment
            float incl = seg;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const float o = __shfl_up_sync(0xffffffffu, incl, off);
                if (lane >= off) incl += o;
            }
            const float excl = incl - seg;
            const float total = __shfl_sync(0xffffffffu, incl, 31);
            const float target = __ldg(uniforms + q * T + s) * total;
            // the running sums below restart from excl in the same order as seg,
            // so the lane's last running value is exactly excl + seg's sequence
            float run = excl;
            int mine = -1, last_pos = -1;
            for (int j = jb; j < je; ++j) {
                const float w = expf((L[j] - mx) / temperature);
                run += w;
                if (w > 0.f) last_pos = j;
                if (mine < 0 && run > target) mine = j;
            }
            const unsigned hit = __ballot_sync(0xffffffffu, mine >= 0);
            if (hit) {
                pick = __shfl_sync(0xffffffffu, mine, __ffs(hit) - 1);
            } else {
                // u * total rounded up to the full sum: the last candidate with weight
                const unsigned nz = __ballot_sync(0xffffffffu, last_pos >= 0);
                pick = nz ? __shfl_sync(0xffffffffu, last_pos, 31 - __clz(nz)) : 0;
            }
        }
        if (lane == 0) {
            path[q * T + s] = __ldg(cand + pick);
            path_scores[q * T + s] = L[pick];
        }
        i = pick;
    }
}

}  // namespace

cudaError_t lattice_launch(const int32_t* anchors, int R, int B, const int32_t* ids, const float* vals,
                           const float* G, const uint16_t* A, const uint16_t* Bc, int64_t V, int K,
                           int r, float* lattice, int32_t* dev_status, cudaStream_t stream) {
    const int T = B - 1;
    if (K > 32 && K <= kLtcMaxK) {  // shorter lists: latency-bound, the CUDA-core tiles below
        // one slice buffer (the accumulator is staged over it at the end), then the
        // barriers, the TMEM address and the abort flag: eight CTAs fit on an SM
        const size_t smem = size_t(kLtcBuf) + 64 + 1024;
        cudaError_t e = cudaFuncSetAttribute(lattice_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             int(smem));
        if (e != cudaSuccess) return e;
        lattice_tc_kernel<<<unsigned(int64_t(R) * T), kLtcThreads, smem, stream>>>(anchors, B, ids, vals, G, A, Bc,
                                                                                   V, K, r, lattice, dev_status);
        note_launch();
        return cudaGetLastError();
    }
#define DF2_LAT(TM)                                                                                   \
    do {                                                                                              \
        const int tiles = (K + 16 * (TM) - 1) / (16 * (TM));                                          \
        const int64_t grid = int64_t(R) * T * tiles * tiles;                                          \
        lattice_kernel<TM><<<unsigned(grid), kLatThreads, 0, stream>>>(anchors, B, ids, vals, G, A, Bc, \
                                                                       V, K, r, tiles, lattice,       \
                                                                       dev_status);                   \
    } while (0)
    if (K <= 16)
        DF2_LAT(1);
    else if (K <= 32)
        DF2_LAT(2);
    else
        DF2_LAT(4);
#undef DF2_LAT
    note_launch();
    return cudaGetLastError();
}

cudaError_t lattice_walk_launch(const float* lattice, const int32_t* ids, int R, int B, int K, int64_t V,
                                const float* uniforms, float temperature, int32_t* path,
                                float* path_scores, int32_t* dev_status, cudaStream_t stream) {
    const unsigned grid = unsigned((int64_t(R) + kWalkWarps - 1) / kWalkWarps);
    lattice_walk_kernel<<<grid, kWalkWarps * 32, 0, stream>>>(lattice, ids, R, B, K, V, uniforms,
                                                              temperature, path, path_scores,
                                                              dev_status);
    note_launch();
    return cudaGetLastError();
}

}  // namespace df2
