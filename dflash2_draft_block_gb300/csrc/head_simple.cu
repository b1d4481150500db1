// Unary logits + per-position top-K on the CUDA cores (the general-shape path).
//
// U[p, v] = h[p, :] . W_lm[v, :] for the full vocabulary ("DFlash2", vLLM
// Speculators guide, "Candidate Selector"), reduced on chip to the K best
// (value desc, id asc) per position; U is never written to global memory.
//
// Grid (S, ceil(P / PG)): CTA (s, b) owns vocabulary chunk s and positions
// [b*PG, b*PG + PG).  Its 8 warps compute 256 logits per tile (32 rows each, one
// lane per 16 bytes of a W_lm row, h staged in shared memory); warp p then folds
// position p's 256 new logits into that position's running list.  Each CTA writes
// its unsorted per-chunk lists to the workspace; topk_merge_kernel reduces the S
// lists of a position to the final sorted top-K.
#include "common.cuh"
#include "kernels.h"

namespace df2 {

namespace {

constexpr int kThreads = 256;
constexpr int kTile = 256;  // vocab rows per tile (8 warps x 32)

template <int PG>
__global__ void __launch_bounds__(kThreads)
head_simple_kernel(const uint16_t* __restrict__ h, int64_t P, int64_t D,
                   const uint16_t* __restrict__ W, int64_t V, int K, int64_t chunk_rows,
                   float* __restrict__ part_v, int* __restrict__ part_id) {
    extern __shared__ __align__(16) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t p0 = int64_t(blockIdx.y) * PG;
    const int np = int(dmin<int64_t>(PG, P - p0));
    const int64_t v_begin = int64_t(blockIdx.x) * chunk_rows;
    const int64_t v_end = dmin<int64_t>(V, v_begin + chunk_rows);

    uint16_t* hs = reinterpret_cast<uint16_t*>(smem);                         // [PG][D]
    float* stage = reinterpret_cast<float*>(smem + size_t(PG) * D * 2);       // [PG][kTile]
    float* lv = stage + PG * kTile;                                           // [PG][K]
    int* lid = reinterpret_cast<int*>(lv + size_t(PG) * K);                   // [PG][K]

    const int64_t d8 = D / 8;
    for (int64_t i = threadIdx.x; i < PG * d8; i += kThreads) {
        const int p = int(i / d8);
        uint4 val = make_uint4(0, 0, 0, 0);
        if (p < np) val = reinterpret_cast<const uint4*>(h + (p0 + p) * D)[i % d8];
        reinterpret_cast<uint4*>(hs)[i] = val;
    }
    __syncthreads();

    WarpTopK list;
    list.init(lv + warp * K, lid + warp * K, K);  // used only by warps < np

    for (int64_t tile = v_begin; tile < v_end; tile += kTile) {
        float mine[PG];
#pragma unroll
        for (int p = 0; p < PG; ++p) mine[p] = 0.f;
        for (int i = 0; i < 32; ++i) {
            const int64_t v = tile + warp * 32 + i;
            float acc[PG];
#pragma unroll
            for (int p = 0; p < PG; ++p) acc[p] = 0.f;
            if (v < v_end) {
                const uint4* wrow = reinterpret_cast<const uint4*>(W + v * D);
                for (int64_t c = lane; c < d8; c += 32) {
                    float wf[8];
                    unpack8(__ldg(wrow + c), wf);
#pragma unroll
                    for (int p = 0; p < PG; ++p) {
                        float hf[8];
                        unpack8(reinterpret_cast<const uint4*>(hs + size_t(p) * D)[c], hf);
#pragma unroll
                        for (int e = 0; e < 8; ++e) acc[p] = fmaf(wf[e], hf[e], acc[p]);
                    }
                }
            }
#pragma unroll
            for (int p = 0; p < PG; ++p) {
                const float s = warp_sum(acc[p]);
                if (lane == i) mine[p] = s;
            }
        }
#pragma unroll
        for (int p = 0; p < PG; ++p) stage[p * kTile + warp * 32 + lane] = mine[p];
        __syncthreads();
        if (warp < np) {
            for (int b = 0; b < kTile / 32; ++b) {
                const int64_t v = tile + b * 32 + lane;
                list.offer(v < v_end, stage[warp * kTile + b * 32 + lane], int(v), lane);
            }
        }
        __syncthreads();
    }

    if (warp < np) {
        const int64_t row = (int64_t(blockIdx.x) * P + p0 + warp) * K;
        for (int k = lane; k < K; k += 32) {
            const bool has = k < list.n;
            part_v[row + k] = has ? lv[warp * K + k] : -INFINITY;
            part_id[row + k] = has ? lid[warp * K + k] : -1;
        }
    }
}

// One CTA per position: fold the S partial lists into the final sorted top-K.
// Candidates are staged through shared memory in chunks with independent,
// coalesced loads (all 256 threads), so the selection never waits on a global
// load; each warp then keeps its own list over its share of a chunk, and warp 0
// folds the 8 lists together at the end.
constexpr int kMergeChunk = 4096;

__global__ void __launch_bounds__(kThreads)
topk_merge_kernel(const float* __restrict__ part_v, const int* __restrict__ part_id, int S,
                  int64_t P, int K, int32_t* __restrict__ out_ids, float* __restrict__ out_vals,
                  LogitMap lm) {
    extern __shared__ __align__(16) uint8_t smem[];
    float* cv_s = reinterpret_cast<float*>(smem);                       // [kMergeChunk]
    int* ci_s = reinterpret_cast<int*>(cv_s + kMergeChunk);             // [kMergeChunk]
    float* lv = reinterpret_cast<float*>(ci_s + kMergeChunk);           // [8][K]
    int* lid = reinterpret_cast<int*>(lv + 8 * K);                      // [8][K]
    int* counts = lid + 8 * K;                                          // [8]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t p = blockIdx.x;

    WarpTopK list;
    list.init(lv + warp * K, lid + warp * K, K);
    const int64_t total = int64_t(S) * K;
    for (int64_t c0 = 0; c0 < total; c0 += kMergeChunk) {
        const int n = int(dmin<int64_t>(kMergeChunk, total - c0));
        for (int i = threadIdx.x; i < n; i += kThreads) {
            const int64_t idx = c0 + i;
            const int64_t s = idx / K, k = idx - s * K;
            const int64_t at = (s * P + p) * K + k;
            cv_s[i] = part_v[at];
            ci_s[i] = part_id[at];
        }
        __syncthreads();
        for (int b = warp * 32; b < n; b += kThreads) {
            const int i = b + lane;
            const bool in = i < n;
            const int cid = in ? ci_s[i] : -1;
            list.offer(cid >= 0, in ? cv_s[i] : 0.f, cid, lane);
        }
        __syncthreads();
    }
    if (lane == 0) counts[warp] = list.n;
    __syncthreads();
    if (warp == 0) {
        for (int w = 1; w < kThreads / 32; ++w) {
            const int nw = counts[w];
            for (int k0 = 0; k0 < nw; k0 += 32) {
                const int k = k0 + lane;
                const bool valid = k < nw;
                list.offer(valid, valid ? lv[w * K + k] : 0.f, valid ? lid[w * K + k] : 0, lane);
            }
        }
        if (lane == 0) counts[0] = list.n;
    }
    __syncthreads();
    write_sorted(lv, lid, counts[0], K, out_ids + p * K, out_vals + p * K, threadIdx.x, kThreads, lm);
}

struct SimplePlan {
    int PG;
    int S;
    int64_t chunk_rows;
    size_t smem;
};

SimplePlan plan_simple(int64_t P, int64_t D, int64_t V, int K, int num_sms) {
    SimplePlan pl{};
    const size_t budget = 200 * 1024;
    pl.PG = 1;
    for (int pg : {8, 4, 2, 1}) {
        size_t need = size_t(pg) * (D * 2 + kTile * 4 + size_t(K) * 8);
        if (need <= budget) { pl.PG = pg; break; }
    }
    pl.smem = size_t(pl.PG) * (D * 2 + kTile * 4 + size_t(K) * 8);
    const int64_t groups = (P + pl.PG - 1) / pl.PG;
    const int64_t want_ctas = 2LL * num_sms;
    int64_t S = (want_ctas + groups - 1) / groups;
    const int64_t max_s = (V + kTile - 1) / kTile;
    S = S < 1 ? 1 : (S > max_s ? max_s : S);
    int64_t chunk = (V + S - 1) / S;
    chunk = (chunk + kTile - 1) / kTile * kTile;
    pl.chunk_rows = chunk;
    pl.S = int((V + chunk - 1) / chunk);
    return pl;
}

}  // namespace

bool head_simple_supported(int64_t D, int K) {
    const size_t need = D * 2 + kTile * 4 + size_t(K) * 8;
    return need <= 200 * 1024;
}

size_t head_simple_workspace(int64_t P, int64_t D, int64_t V, int K, int num_sms) {
    if (P <= 0) return 0;
    SimplePlan pl = plan_simple(P, D, V, K, num_sms);
    return size_t(pl.S) * size_t(P) * size_t(K) * 8;
}

cudaError_t head_simple_launch(const uint16_t* h, int64_t P, int64_t D, const uint16_t* W, int64_t V,
                               int K, int32_t* ids, float* vals, void* ws, int num_sms,
                               cudaStream_t stream, LogitMap lm) {
    SimplePlan pl = plan_simple(P, D, V, K, num_sms);
    float* part_v = reinterpret_cast<float*>(ws);
    int* part_id = reinterpret_cast<int*>(part_v + size_t(pl.S) * P * K);
    dim3 grid(pl.S, unsigned((P + pl.PG - 1) / pl.PG));
    cudaError_t e = cudaSuccess;
    switch (pl.PG) {
#define DF2_CASE(PGV)                                                                          \
    case PGV:                                                                                  \
        e = cudaFuncSetAttribute(head_simple_kernel<PGV>,                                      \
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, int(pl.smem));    \
        if (e != cudaSuccess) return e;                                                        \
        head_simple_kernel<PGV><<<grid, kThreads, pl.smem, stream>>>(h, P, D, W, V, K,         \
                                                                    pl.chunk_rows, part_v,    \
                                                                    part_id);                 \
        break;
        DF2_CASE(8)
        DF2_CASE(4)
        DF2_CASE(2)
        DF2_CASE(1)
#undef DF2_CASE
    }
    note_launch();
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    return topk_merge_launch(part_v, part_id, pl.S, P, K, ids, vals, stream, lm);
}

cudaError_t topk_merge_launch(const float* part_v, const int* part_id, int S, int64_t P, int K,
                              int32_t* ids, float* vals, cudaStream_t stream, LogitMap lm) {
    const size_t msmem = size_t(kMergeChunk) * 8 + size_t(8) * K * 8 + 64;
    cudaError_t e = cudaFuncSetAttribute(topk_merge_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, int(msmem));
    if (e != cudaSuccess) return e;
    topk_merge_kernel<<<unsigned(P), kThreads, msmem, stream>>>(part_v, part_id, S, P, K, ids, vals, lm);
    note_launch();
    return cudaGetLastError();
}

}  // namespace df2
