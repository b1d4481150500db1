// Cross-CTA merge of sorted per-CTA top-K lists (K <= 64) into the final top-K,
// shared by the merge kernel and the fused draft-head kernel.
//
// One CTA per position.  All lists of the position are first copied to shared
// memory in one round of independent loads.  Every list is sorted, so the K best
// list heads are K entries that rank at or above the K-th best head t: the final
// K entries all rank at or above t, and each list contributes only its prefix that
// does.  The threads rank the heads against each other to find t, compact the
// qualifying prefixes into a candidate buffer (a few dozen entries on typical
// data), and one warp folds the candidates into a register-resident list
// (topk_warp.cuh) and writes the K best in rank order.  Without a threshold
// (fewer than K non-empty lists) the 8 warps fold whole lists and warp 0 combines
// their lists.
#pragma once

#include "common.cuh"
#include "topk_warp.cuh"

namespace df2 {
namespace mrg {

constexpr int kWarps = 8;
constexpr int kMergeThreads = kWarps * 32;
constexpr int kOneWarpCands = 128;  // up to this many candidates one warp folds them alone

__host__ __device__ inline size_t merge_smem(int S, int K) { return size_t(S) * K * 16 + size_t(S) * 12; }

// The final top-K of position p from the S sorted lists part_[v|id][s][P][K], by
// one CTA of kMergeThreads threads with merge_smem(S, K) bytes at smem.  Warp 0
// writes out_ids/out_vals[p], each kept value passed through map; the other
// warps return without touching them.
template <int R, class Map>
__device__ __forceinline__ void merge_position(const float* __restrict__ part_v,
                                               const int* __restrict__ part_id, int S, int64_t P,
                                               int K, int64_t p, int32_t* __restrict__ out_ids,
                                               float* __restrict__ out_vals, uint8_t* smem, Map map) {
    float* cv = reinterpret_cast<float*>(smem);        // [S*K] this position's lists
    int* ci = reinterpret_cast<int*>(cv + S * K);
    float* bv = reinterpret_cast<float*>(ci + S * K);  // [S*K] candidates
    int* bi = reinterpret_cast<int*>(bv + S * K);
    __shared__ float xv[kWarps][R * 32];
    __shared__ int xi[kWarps][R * 32];
    __shared__ float t_v;
    __shared__ int t_id, have_t, n_cand;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0) {
        have_t = 0;
        n_cand = 0;
    }
    // one round of independent, coalesced loads of every list of this position
    for (int i = tid; i < S * K; i += kWarps * 32) {
        const int s = i / K, k = i - s * K;
        const size_t at = (size_t(s) * P + p) * K + k;
        cv[i] = __ldg(part_v + at);
        ci[i] = __ldg(part_id + at);
    }
    __syncthreads();
    // the K-th best head: the head that exactly K-1 other heads rank before.  The
    // heads are packed as rank keys (larger = ranks before; 0 = empty list) into
    // the still unused candidate buffer, and two threads count each head's rank.
    unsigned long long* hk = reinterpret_cast<unsigned long long*>(smem + size_t(S) * K * 16);
    int* rk = reinterpret_cast<int*>(hk + S);
    for (int s = tid; s < S; s += kWarps * 32) {
        const int id = ci[s * K];
        hk[s] = id < 0 ? 0ull : rank_key(cv[s * K], id);
        rk[s] = 0;
    }
    __syncthreads();
    const int half = (S + 1) / 2;
    for (int it = tid; it < 2 * S; it += kWarps * 32) {
        const int s = it >> 1, o0 = (it & 1) ? half : 0, o1 = (it & 1) ? S : half;
        const unsigned long long mine = hk[s];
        if (mine == 0ull) continue;
        int n = 0;
#pragma unroll 8
        for (int o = o0; o < o1; ++o) n += hk[o] > mine ? 1 : 0;
        atomicAdd(rk + s, n);
    }
    __syncthreads();
    for (int s = tid; s < S; s += kWarps * 32) {
        if (hk[s] != 0ull && rk[s] == K - 1) {
            t_v = cv[s * K];
            t_id = ci[s * K];
            have_t = 1;
        }
    }
    __syncthreads();
    wtk::List<R> m;
    m.clear();
    if (have_t) {
        const float tv = t_v;
        const int tk = t_id;
        for (int s = tid; s < S; s += kWarps * 32) {
            for (int k = 0; k < K; ++k) {
                const int id = ci[s * K + k];
                const float v = cv[s * K + k];
                if (id < 0 || !(ranks_before(v, id, tv, tk) || (v == tv && id == tk))) break;
                const int at = atomicAdd(&n_cand, 1);
                bv[at] = v;
                bi[at] = id;
            }
        }
        __syncthreads();
        const int M = n_cand;
        if (M <= kOneWarpCands) {
            if (warp == 0)
            for (int b = 0; b < M; b += 32) {
                const int i = b + lane;
                m.offer(i < M ? bv[i] : -INFINITY, i < M ? bi[i] : wtk::kEmptyId, K, lane);
            }
        } else {
            for (int b = warp * 32; b < M; b += kWarps * 32) {
                const int i = b + lane;
                m.offer(i < M ? bv[i] : -INFINITY, i < M ? bi[i] : wtk::kEmptyId, K, lane);
            }
        }
    } else {
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
    }
    if (!have_t || n_cand > kOneWarpCands) {
        // fold the 8 warps' lists into warp 0's
#pragma unroll
        for (int rr = 0; rr < R; ++rr) {
            xv[warp][rr * 32 + lane] = m.v[rr];
            xi[warp][rr * 32 + lane] = m.id[rr];
        }
        __syncthreads();
        if (warp == 0)
        for (int w = 1; w < kWarps; ++w)
#pragma unroll
            for (int rr = 0; rr < R; ++rr) m.offer_sorted(xv[w][rr * 32 + lane], xi[w][rr * 32 + lane], K, lane);
    }
    if (warp != 0) return;
#pragma unroll
    for (int rr = 0; rr < R; ++rr) {
        const int k = rr * 32 + lane;
        if (k < K) {
            const bool ok = m.id[rr] != wtk::kEmptyId;
            out_ids[p * K + k] = ok ? m.id[rr] : -1;
            out_vals[p * K + k] = ok ? map(m.v[rr]) : -INFINITY;
        }
    }
}

}  // namespace mrg
}  // namespace df2
