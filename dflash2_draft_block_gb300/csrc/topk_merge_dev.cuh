// Cross-CTA merge of sorted per-CTA top-K lists (K <= 64) into the final top-K,
// shared by the merge kernel and the fused draft-head kernel.
//
// One CTA per position.  All lists of the position are first copied to shared
// memory in one round of independent loads.  Every list is sorted, so the L best
// list heads are L entries that rank at or above the L-th best head t: the best L
// entries all rank at or above t, and each list contributes only its prefix that
// does.  The threads rank the heads against each other to find t, compact the
// qualifying prefixes into a candidate buffer (a few dozen entries on typical
// data), and one warp folds the candidates into a register-resident list
// (topk_warp.cuh).  Without a threshold (fewer than L non-empty lists) the 8 warps
// fold whole lists and warp 0 combines their lists.
//
// Exact decisions on near ties.  The head kernels sum the logits in fp32 on the
// tensor cores, in another order than a plain sum; two logits closer than that
// rounding (a few ulps of the accumulator over the reduction) may come out in the
// wrong order.  With a Refine argument the merge also finds the (K+1)-th entry, and
// wherever two neighbours of that list lie within 2^-14 of their magnitude (well
// above the fp32 accumulation error of the tensor-core sum), it recomputes those
// logits as correctly rounded fp32 values -- exact bf16 products, compensated
// summation, one final rounding: the precision the ranking is defined in -- and
// ranks the K + 1 entries again by (value, lower id).  The K-th/(K+1)-th boundary and the order inside the list are
// then decided on correctly rounded logits.  (A candidate a head CTA dropped
// because its own K entries were all better cannot be recovered: that needs the
// whole top K + 1 in one CTA's vocabulary range.)
#pragma once

#include "common.cuh"
#include "kernels.h"
#include "topk_warp.cuh"

namespace df2 {
namespace mrg {

constexpr int kWarps = 8;
constexpr int kMergeThreads = kWarps * 32;
constexpr int kOneWarpCands = 128;  // up to this many candidates one warp folds them alone

__host__ __device__ inline size_t merge_smem(int S, int K) { return size_t(S) * K * 16 + size_t(S) * 12; }

// Ask L2 for `bytes` (a multiple of 16) of global memory at p (16-byte aligned).
__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// Two neighbouring fp32 logits this close may be ordered wrongly by the
// tensor-core sum and are recomputed exactly.
__device__ __forceinline__ bool near_tie(float a, float b) {
    const float mag = fmaxf(fmaxf(fabsf(a), fabsf(b)), 1.f);
    return a - b <= mag * (1.f / 16384.f);
}

// s + e = a + b exactly (Knuth's TwoSum; round-to-nearest adds, never contracted).
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
    s = __fadd_rn(a, b);
    const float bb = __fsub_rn(s, a);
    e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
}

// Adds p to the unevaluated sum s + c: s takes the rounded sum, c collects every
// rounding error (compensated summation; the result carries about twice fp32's
// precision).
__device__ __forceinline__ void comp_add(float& s, float& c, float p) {
    float e;
    two_sum(s, p, s, e);
    c = __fadd_rn(c, e);
}

// Part of h . w over D elements: the 16-byte chunks k = k0, k0 + step, ... of the
// row (step a multiple of 32; lane l starts at k0 + l), every bf16 x bf16 product
// exact in fp32 and the products added with compensated summation in four
// independent accumulators per lane, then the lanes combined by a shuffle tree
// (fixed order).  All lanes of the warp call; every lane returns the warp's partial
// as the unevaluated sum S + Cc.  h may be in shared or global memory.  (fp32
// arithmetic: fp64 runs at a small fraction of the fp32 rate on this GPU.)
template <bool HG>
__device__ __forceinline__ void logit_partial(const uint16_t* h, const uint16_t* __restrict__ w, int64_t D,
                                              int64_t k0, int64_t step, int lane, float& S, float& Cc) {
    float s[4] = {0.f, 0.f, 0.f, 0.f}, c[4] = {0.f, 0.f, 0.f, 0.f};
    const int64_t nck = D / 8;  // 16-byte chunks of a row
    // four W chunks (and, HG: h in global memory, four h chunks) are loaded before
    // any is used: a row costs a few memory latencies, not one per chunk
    for (int64_t kb = k0 + lane; kb < nck; kb += 4 * step) {
        uint4 wv[4], hv[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int64_t k = kb + u * step;
            if (k < nck) {
                wv[u] = __ldg(reinterpret_cast<const uint4*>(w) + k);
                if (HG) hv[u] = __ldg(reinterpret_cast<const uint4*>(h) + k);
            }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int64_t k = kb + u * step;
            if (k >= nck) break;
            float hf[8], wf[8];
            unpack8(HG ? hv[u] : reinterpret_cast<const uint4*>(h)[k], hf);
            unpack8(wv[u], wf);
#pragma unroll
            for (int e = 0; e < 8; ++e) comp_add(s[e & 3], c[e & 3], __fmul_rn(hf[e], wf[e]));
        }
    }
    S = s[0];
    Cc = c[0];
#pragma unroll
    for (int a = 1; a < 4; ++a) {
        comp_add(S, Cc, s[a]);
        Cc = __fadd_rn(Cc, c[a]);
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) {
        const float S2 = __shfl_xor_sync(kFull, S, o), C2 = __shfl_xor_sync(kFull, Cc, o);
        // the same (S, C) in both lanes of a pair: the lower lane's operand first
        const bool lo = (lane & o) == 0;
        float a = lo ? S : S2, b = lo ? S2 : S, e;
        two_sum(a, b, S, e);
        Cc = __fadd_rn(__fadd_rn(lo ? Cc : C2, lo ? C2 : Cc), e);
    }
}

// The final top-K of position p from the S sorted lists part_[v|id][s][P][K], by
// one CTA of kMergeThreads threads with merge_smem(S, K) bytes at smem (32 R >=
// K).  Every thread of the CTA calls it.  Warp 0 writes
// out_ids/out_vals[p] in rank order, each kept value passed through map and the
// list ranked by (mapped value, lower id); the CTA's other warps write nothing.
template <int R, class Map>
__device__ __forceinline__ void merge_position(const float* __restrict__ part_v,
                                               const int* __restrict__ part_id, int S, int64_t P,
                                               int K, int64_t p, int32_t* __restrict__ out_ids,
                                               float* __restrict__ out_vals, uint8_t* smem, Map map,
                                               Refine rf = Refine{nullptr, nullptr, 0}) {
    float* cv = reinterpret_cast<float*>(smem);        // [S*K] this position's lists
    int* ci = reinterpret_cast<int*>(cv + S * K);
    float* bv = reinterpret_cast<float*>(ci + S * K);  // [S*K] candidates
    int* bi = reinterpret_cast<int*>(bv + S * K);
    __shared__ float xv[kWarps][R * 32 + 1];  // row 0 also holds the (K+1)-th entry
    __shared__ int xi[kWarps][R * 32 + 1];
    __shared__ int re_idx[R * 32 + 1];
    __shared__ int8_t link[R * 32 + 1];  // link[k]: entries k and k + 1 are near-tied
    __shared__ float red_s[kWarps], red_c[kWarps];
    __shared__ float t_v;
    __shared__ int t_id, have_t, n_cand, n_re;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const bool refine = rf.h != nullptr;
    // refining needs the (K+1)-th entry as well: the threshold is then the
    // (K+1)-th best head, so that the candidates hold the best K + 1
    const int L = refine ? K + 1 : K;
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
    // the L-th best head: the head that exactly L-1 other heads rank before.  The
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
        if (hk[s] != 0ull && rk[s] == L - 1) {
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
    if (!refine) {
        if (warp != 0) return;
        if (map.identity()) {
#pragma unroll
            for (int rr = 0; rr < R; ++rr) {
                const int k = rr * 32 + lane;
                if (k < K) {
                    const bool ok = m.id[rr] != wtk::kEmptyId;
                    out_ids[p * K + k] = ok ? m.id[rr] : -1;
                    out_vals[p * K + k] = ok ? m.v[rr] : -INFINITY;
                }
            }
            return;
        }
        // warp 0 alone from here: its entries to shared memory for the ranking
#pragma unroll
        for (int rr = 0; rr < R; ++rr) {
            xv[0][rr * 32 + lane] = m.v[rr];
            xi[0][rr * 32 + lane] = m.id[rr];
        }
        __syncwarp();
    } else {
        // Warp 0's K entries to shared memory, and after them the (K+1)-th: the best
        // entry that ranks after the K-th, found by a scan of the candidates (or,
        // without a threshold, of every list).  Then the entries in runs of near
        // ties get their exact logits, each recomputed by one warp of the CTA.
        __syncthreads();  // any fold through xv is over
        if (warp == 0) {
#pragma unroll
            for (int rr = 0; rr < R; ++rr) {
                xv[0][rr * 32 + lane] = m.v[rr];
                xi[0][rr * 32 + lane] = m.id[rr];
            }
            float kv;
            int kid;
            m.kth(K, kv, kid);
            float nv = -INFINITY;
            int nid = wtk::kEmptyId;
            const int n_scan = have_t ? n_cand : S * K;
            const float* sv = have_t ? bv : cv;
            const int* si = have_t ? bi : ci;
            for (int i = lane; i < n_scan; i += 32) {
                const int id = si[i];
                if (id < 0 || id == wtk::kEmptyId) continue;
                const float v = sv[i];
                if (kid != wtk::kEmptyId && !ranks_before(kv, kid, v, id)) continue;  // not after the K-th
                if (nid == wtk::kEmptyId || ranks_before(v, id, nv, nid)) { nv = v; nid = id; }
            }
#pragma unroll
            for (int o = 16; o; o >>= 1) {
                const float ov = __shfl_xor_sync(kFull, nv, o);
                const int oid = __shfl_xor_sync(kFull, nid, o);
                if (oid != wtk::kEmptyId && (nid == wtk::kEmptyId || ranks_before(ov, oid, nv, nid))) {
                    nv = ov;
                    nid = oid;
                }
            }
            if (lane == 0) {
                xv[0][K] = kid != wtk::kEmptyId ? nv : -INFINITY;
                xi[0][K] = kid != wtk::kEmptyId ? nid : wtk::kEmptyId;
                n_re = 0;
            }
            __syncwarp();
            for (int k = lane; k < L; k += 32) {
                const bool ok = xi[0][k] != wtk::kEmptyId;
                const bool up = k > 0 && ok && near_tie(xv[0][k - 1], xv[0][k]);
                const bool down =
                    k + 1 < L && ok && xi[0][k + 1] != wtk::kEmptyId && near_tie(xv[0][k], xv[0][k + 1]);
                link[k] = down ? 1 : 0;
                if (up || down) re_idx[atomicAdd(&n_re, 1)] = k;
            }
        }
        __syncthreads();
        const int nre = n_re;
        if (nre > 0) {
            // every recomputed entry's W row asked into L2 at once: the rounds after
            // the first then read it from there
            for (int f = tid; f < nre; f += kWarps * 32) {
                const int32_t id = xi[0][re_idx[f]];
                prefetch_l2(rf.W + int64_t(id) * rf.D, uint32_t(rf.D) * 2u);
            }
            // the row of h, read by every recompute: with more than two, into the
            // lists' shared memory (free again: the scan above was its last use) when
            // it fits; one or two read it from global memory beside their W rows
            const uint16_t* hrow = rf.h + p * rf.D;
            const bool staged = nre > 2 && size_t(rf.D) * 2 <= size_t(S) * K * 16;
            if (staged) {
                uint4* hs = reinterpret_cast<uint4*>(smem);
                for (int64_t i = tid; i < rf.D / 8; i += kWarps * 32)
                    hs[i] = __ldg(reinterpret_cast<const uint4*>(hrow) + i);
                __syncthreads();
                hrow = reinterpret_cast<const uint16_t*>(smem);
            }
            // gw warps per recompute (all eight for one): a recompute's loads are
            // spread over gw * 32 lanes, so one or two rows cost about one memory
            // latency; the warps' partials are added in warp order
            const int gw = nre >= 8 ? 1 : (nre >= 4 ? 2 : (nre >= 2 ? 4 : 8));
            const int per_round = kWarps / gw;
            for (int f0 = 0; f0 < nre; f0 += per_round) {
                const int f = f0 + warp / gw, sub = warp % gw;
                float S = 0.f, Cc = 0.f;
                if (f < nre) {
                    const uint16_t* wrow = rf.W + int64_t(xi[0][re_idx[f]]) * rf.D;
                    if (staged) logit_partial<false>(hrow, wrow, rf.D, int64_t(sub) * 32, int64_t(gw) * 32, lane, S, Cc);
                    else logit_partial<true>(hrow, wrow, rf.D, int64_t(sub) * 32, int64_t(gw) * 32, lane, S, Cc);
                }
                if (lane == 0) {
                    red_s[warp] = S;
                    red_c[warp] = Cc;
                }
                __syncthreads();
                if (sub == 0 && lane == 0 && f < nre) {
                    float T = red_s[warp], Tc = red_c[warp];
                    for (int q = 1; q < gw; ++q) {
                        float e;
                        two_sum(T, red_s[warp + q], T, e);
                        Tc = __fadd_rn(__fadd_rn(Tc, red_c[warp + q]), e);
                    }
                    xv[0][re_idx[f]] = __fadd_rn(T, Tc);
                }
                __syncthreads();
            }
        }
        if (warp != 0) return;
    }
    if (refine && map.identity()) {
        // The list is sorted by the fp32 values the kernels computed; only the
        // entries of a run of near ties (now holding exact values) may change places,
        // and only among themselves: each entry's rank is its run's first index plus
        // the run entries that rank before it.  Entries outside runs keep their
        // place, and the ranks of a run are a permutation of its indices whatever the
        // recomputed values are.
        for (int k = lane; k < L; k += 32) {
            const int id = xi[0][k];
            if (id == wtk::kEmptyId) {
                if (k < K) {
                    out_ids[p * K + k] = -1;
                    out_vals[p * K + k] = -INFINITY;
                }
                continue;
            }
            const float v = xv[0][k];
            int s0 = k, s1 = k;
            while (s0 > 0 && link[s0 - 1]) --s0;
            while (s1 + 1 < L && link[s1]) ++s1;
            int rank = s0;
            for (int j = s0; j <= s1; ++j)
                if (j != k && ranks_before(xv[0][j], xi[0][j], v, id)) ++rank;
            if (rank < K) {
                out_ids[p * K + rank] = id;
                out_vals[p * K + rank] = v;
            }
        }
        return;
    }
    // Rank the kept entries by (mapped value, id): the list is sorted by the fp32
    // values the kernels computed; this settles the recomputed near ties and the
    // neighbours a saturating map rounds to one value.  Empty slots stay at the end.
    int nvalid = 0;
    for (int k = 0; k < L; ++k) nvalid += xi[0][k] != wtk::kEmptyId ? 1 : 0;
    for (int k = lane; k < L; k += 32) {
        const int id = xi[0][k];
        if (id == wtk::kEmptyId) {
            if (k < K) {
                out_ids[p * K + k] = -1;
                out_vals[p * K + k] = -INFINITY;
            }
            continue;
        }
        const float mv = map(xv[0][k]);
        int rank = 0;
        for (int j = 0; j < L; ++j) {
            const int oj = xi[0][j];
            if (oj != wtk::kEmptyId && ranks_before(map(xv[0][j]), oj, mv, id)) ++rank;
        }
        if (rank < K && rank < nvalid) {
            out_ids[p * K + rank] = id;
            out_vals[p * K + rank] = mv;
        }
    }
}

}  // namespace mrg
}  // namespace df2
