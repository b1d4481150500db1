// Device-side building blocks of the candidate selector, shared by the selector
// kernels and the fused draft-head kernel.
//
// Pair score S_t(a, b) = U_t(b) + < A(a) (.) H(h_t), B(b) > (verl-SpeCo PR #62,
// "What DFlash2 adds"; "DFlash 2 Explanation", "Problem 1").  Every dot product
// here uses one lane slicing -- lane l owns rank elements [256c + 8l, 256c + 8l + 8)
// of the gate and of every B row, an fmaf chain over them -- and one shuffle tree
// over the lanes, so the walk, the teacher-forced scores and the fused head give
// bit-identical scores.
#pragma once

#include "common.cuh"

namespace df2 {
namespace sel {

// q[c][e] = A[a, 256c + 8l + e] * G[256c + 8l + e] for the lane's slice (NCH chunks).
template <int NCH>
__device__ __forceinline__ void load_gate(const uint16_t* __restrict__ A, int64_t a, int r,
                                          const float* __restrict__ Grow, int lane,
                                          float q[NCH][8]) {
#pragma unroll
    for (int c = 0; c < NCH; ++c) {
        const int i0 = c * 256 + lane * 8;
        if (i0 < r) {
            float af[8];
            unpack8(__ldg(reinterpret_cast<const uint4*>(A + a * r + i0)), af);
            const float4 g0 = __ldg(reinterpret_cast<const float4*>(Grow + i0));
            const float4 g1 = __ldg(reinterpret_cast<const float4*>(Grow + i0 + 4));
            q[c][0] = af[0] * g0.x; q[c][1] = af[1] * g0.y; q[c][2] = af[2] * g0.z; q[c][3] = af[3] * g0.w;
            q[c][4] = af[4] * g1.x; q[c][5] = af[5] * g1.y; q[c][6] = af[6] * g1.z; q[c][7] = af[7] * g1.w;
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) q[c][e] = 0.f;
        }
    }
}

template <int NCH>
__device__ __forceinline__ float dot_lane(const uint16_t* __restrict__ Bc, int64_t b, int r, int lane,
                                          const float q[NCH][8]) {
    float s = 0.f;
#pragma unroll
    for (int c = 0; c < NCH; ++c) {
        const int i0 = c * 256 + lane * 8;
        if (i0 < r) {
            float bf[8];
            unpack8(__ldg(reinterpret_cast<const uint4*>(Bc + b * r + i0)), bf);
#pragma unroll
            for (int e = 0; e < 8; ++e) s = fmaf(q[c][e], bf[e], s);
        }
    }
    return s;
}

__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gmem_src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(
                     static_cast<uint32_t>(__cvta_generic_to_shared(smem_dst))),
                 "l"(gmem_src)
                 : "memory");
}

// Walk with everything it can read gathered into shared memory: the B rows of
// every candidate of rows 1..B-1, the A rows of the anchor and of every candidate
// of rows 1..B-2 (the only possible predecessors), and the G rows.  The gathers
// are issued up front in one cp.async group per step, in the order the steps
// need them, so step t starts as soon as its own group has landed.  One CTA per
// request; all 8 warps score each step's candidates.
constexpr int kWalkThreads = 256;
constexpr int kWalkWarps = kWalkThreads / 32;

__host__ __device__ inline size_t walk_cta_smem(int B, int K, int r) {
    const size_t T = size_t(B) - 1;
    return T * K * r * 2 + ((T - 1) * K + 1) * r * 2 + T * r * 4 + T * K * 8 + 2 * size_t(K) * 4 + 64;
}

// A lane's slices [256c + 8l, 256c + 8l + 8) of a bf16 row and of an fp32 row in
// shared memory (zeros past r, or everywhere when !valid).
template <int NCH>
__device__ __forceinline__ void load_bslice(const uint16_t* row, int r, int lane, bool valid,
                                            float out[NCH][8]) {
#pragma unroll
    for (int c = 0; c < NCH; ++c) {
        const int i0 = c * 256 + lane * 8;
        if (valid && i0 < r) {
            unpack8(*reinterpret_cast<const uint4*>(row + i0), out[c]);
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) out[c][e] = 0.f;
        }
    }
}

template <int NCH>
__device__ __forceinline__ void load_gslice(const float* row, int r, int lane, float out[NCH][8]) {
#pragma unroll
    for (int c = 0; c < NCH; ++c) {
        const int i0 = c * 256 + lane * 8;
        if (i0 < r) {
            const float4 x = *reinterpret_cast<const float4*>(row + i0);
            const float4 y = *reinterpret_cast<const float4*>(row + i0 + 4);
            out[c][0] = x.x; out[c][1] = x.y; out[c][2] = x.z; out[c][3] = x.w;
            out[c][4] = y.x; out[c][5] = y.y; out[c][6] = y.z; out[c][7] = y.w;
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) out[c][e] = 0.f;
        }
    }
}

// Wait until at most n of this thread's cp.async groups are pending (n > 7: 7).
__device__ __forceinline__ void cp_async_wait_pending(int n) {
    switch (n) {
        case 0: asm volatile("cp.async.wait_group 0;" ::: "memory"); break;
        case 1: asm volatile("cp.async.wait_group 1;" ::: "memory"); break;
        case 2: asm volatile("cp.async.wait_group 2;" ::: "memory"); break;
        case 3: asm volatile("cp.async.wait_group 3;" ::: "memory"); break;
        case 4: asm volatile("cp.async.wait_group 4;" ::: "memory"); break;
        case 5: asm volatile("cp.async.wait_group 5;" ::: "memory"); break;
        case 6: asm volatile("cp.async.wait_group 6;" ::: "memory"); break;
        default: asm volatile("cp.async.wait_group 7;" ::: "memory"); break;
    }
}

// The greedy walk of one request by one CTA of kWalkThreads threads, with every
// gather staged in shared memory (walk_cta_smem bytes at smem).  kFresh: the
// candidate lists were written earlier in the same kernel, so they are read
// through L2 rather than the read-only path.
template <int NCH, bool kFresh>
__device__ __forceinline__ void walk_request_cta(int q, const int32_t* __restrict__ anchors, int B,
                                                 const int32_t* __restrict__ ids,
                                                 const float* __restrict__ vals,
                                                 const float* __restrict__ G,
                                                 const uint16_t* __restrict__ A,
                                                 const uint16_t* __restrict__ Bc, int64_t V, int K,
                                                 int r, int32_t* __restrict__ path,
                                                 float* __restrict__ path_scores,
                                                 int32_t* __restrict__ dev_status, uint8_t* smem) {
    const int T = B - 1;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    uint16_t* Bs = reinterpret_cast<uint16_t*>(smem);                     // [T*K][r]
    uint16_t* As = Bs + size_t(T) * K * r;                                // [(T-1)*K + 1][r]
    float* Gs = reinterpret_cast<float*>(As + (size_t(T - 1) * K + 1) * r);  // [T][r]
    float* vs = Gs + size_t(T) * r;                                       // [T*K]
    int* is = reinterpret_cast<int*>(vs + size_t(T) * K);                 // [T*K]
    float* sc = reinterpret_cast<float*>(is + size_t(T) * K);             // [2][K] step scores
    int* bad = reinterpret_cast<int*>(sc + 2 * size_t(K));

    const int64_t row1 = int64_t(q) * B + 1;  // first drafted row of the request
    const int32_t a0 = __ldg(anchors + q);
    if (tid == 0) *bad = (a0 < 0 || a0 >= V) ? 1 : 0;
    __syncthreads();
    for (int e = tid; e < T * K; e += kWalkThreads) {
        const int32_t b = kFresh ? __ldcg(ids + row1 * K + e) : __ldg(ids + row1 * K + e);
        is[e] = b;
        vs[e] = kFresh ? __ldcg(vals + row1 * K + e) : __ldg(vals + row1 * K + e);
        if (b < 0 || b >= V) *bad = 1;
    }
    __syncthreads();
    if (*bad) {
        for (int t = tid; t < T; t += kWalkThreads) {
            path[int64_t(q) * T + t] = -1;
            path_scores[int64_t(q) * T + t] = __int_as_float(0x7fc00000);
        }
        if (tid == 0 && dev_status) atomicOr(dev_status, DF2_STATUS_ID_OUT_OF_RANGE);
        return;
    }

    // group t: position t's B rows and G row, and the A rows of its possible
    // predecessors (the anchor for t = 1, else position t-1's candidates).  Warp w
    // copies rows w, w+8, ...; lane l copies 16-byte chunks l, l+32, ... of a row.
    const int cpr = r / 8;  // 16-byte chunks per bf16 row
    const int gpr = r / 4;  // 16-byte chunks per fp32 row
    for (int t = 1; t <= T; ++t) {
        for (int row = (t - 1) * K + warp; row < t * K; row += kWalkWarps) {
            const uint16_t* src = Bc + int64_t(is[row]) * r;
            for (int c = lane; c < cpr; c += 32) cp_async16(Bs + size_t(row) * r + c * 8, src + c * 8);
        }
        const int a_lo = (t == 1) ? 0 : 1 + (t - 2) * K;
        const int a_hi = (t == 1) ? 1 : 1 + (t - 1) * K;
        for (int arow = a_lo + warp; arow < a_hi; arow += kWalkWarps) {
            const uint16_t* src = A + (arow == 0 ? int64_t(a0) : int64_t(is[arow - 1])) * r;
            for (int c = lane; c < cpr; c += 32) cp_async16(As + size_t(arow) * r + c * 8, src + c * 8);
        }
        for (int i = tid; i < gpr; i += kWalkThreads)
            cp_async16(Gs + size_t(t - 1) * r + i * 4, G + (row1 + t - 1) * r + i * 4);
        asm volatile("cp.async.commit_group;" ::: "memory");
    }

    // Step t scores position t's candidates against the gate A[a_{t-1}] (.) G_t.
    // Warp w scores candidates w, w+8, ... in pairs; lane l owns rank elements
    // [256c + 8l, 256c + 8l + 8) of the gate and of every B row, and a shuffle tree
    // sums the lanes (the order of the other walk kernels, so the scores are
    // bit-identical).  One barrier per step: after it, the step's gathers and the
    // previous step's scores are visible to all warps, and every warp reduces those
    // scores to the same argmax on its own.  The critical path of a step is that
    // argmax, the predecessor's A row, one FMA chain and one shuffle tree: the B
    // and G slices of a warp's first pair do not depend on the argmax and are read
    // before it (for r <= 512).
    constexpr bool kEarly = NCH <= 2;
    int arow = 0;  // As row of the current predecessor
    for (int t = 1; t <= T + 1; ++t) {
        if (t <= T) cp_async_wait_pending(T - t);
        __syncthreads();
        const int ja = warp, jb = warp + kWalkWarps;
        constexpr int NE = kEarly ? NCH : 1;  // slices held across the argmax
        float gs[NE][8], b0[NE][8], b1[NE][8];
        if constexpr (kEarly) {
            if (t <= T) {
                load_gslice<NE>(Gs + size_t(t - 1) * r, r, lane, gs);
                load_bslice<NE>(Bs + (size_t(t - 1) * K + ja) * r, r, lane, ja < K, b0);
                load_bslice<NE>(Bs + (size_t(t - 1) * K + jb) * r, r, lane, jb < K, b1);
            }
        }
        if (t > 1) {
            const float* sp = sc + ((t - 1) & 1) * K;
            const int* ip = is + (t - 2) * K;
            float bv = -INFINITY;
            int bid = INT_MAX, bj = -1;
            for (int j = lane; j < K; j += 32) {
                const float v = sp[j];
                const int id = ip[j];
                if (bj < 0 || ranks_before(v, id, bv, bid)) {
                    bv = v;
                    bid = id;
                    bj = j;
                }
            }
#pragma unroll
            for (int o = 16; o; o >>= 1) {
                const float ov = __shfl_xor_sync(kFull, bv, o);
                const int oi = __shfl_xor_sync(kFull, bid, o);
                const int oj = __shfl_xor_sync(kFull, bj, o);
                if (oj >= 0 && (bj < 0 || ranks_before(ov, oi, bv, bid) ||
                                (ov == bv && oi == bid && oj < bj))) {
                    bv = ov;
                    bid = oi;
                    bj = oj;
                }
            }
            if (tid == 0) {
                path[int64_t(q) * T + (t - 2)] = bid;
                path_scores[int64_t(q) * T + (t - 2)] = bv;
            }
            arow = 1 + (t - 2) * K + bj;
        }
        if (t > T) break;
        float qv[NCH][8];
#pragma unroll
        for (int c = 0; c < NCH; ++c) {
            const int i0 = c * 256 + lane * 8;
            float af[8], gc[1][8];
            if constexpr (kEarly) {
#pragma unroll
                for (int e = 0; e < 8; ++e) gc[0][e] = gs[c][e];
            } else {
                load_gslice<1>(Gs + size_t(t - 1) * r + c * 256, r - c * 256, lane, gc);
            }
            if (i0 < r) {
                unpack8(*reinterpret_cast<const uint4*>(As + size_t(arow) * r + i0), af);
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e) af[e] = 0.f;
            }
#pragma unroll
            for (int e = 0; e < 8; ++e) qv[c][e] = af[e] * gc[0][e];
        }
        float* so = sc + (t & 1) * K;
        const float* vrow = vs + (t - 1) * K;
        for (int j = ja; j < K; j += 2 * kWalkWarps) {
            const int j2 = j + kWalkWarps;
            float pa = 0.f, pb = 0.f;
            if constexpr (kEarly) {
                if (j != ja) {
                    load_bslice<NE>(Bs + (size_t(t - 1) * K + j) * r, r, lane, true, b0);
                    load_bslice<NE>(Bs + (size_t(t - 1) * K + j2) * r, r, lane, j2 < K, b1);
                }
#pragma unroll
                for (int c = 0; c < NE; ++c)
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        pa = fmaf(qv[c][e], b0[c][e], pa);
                        pb = fmaf(qv[c][e], b1[c][e], pb);
                    }
            } else {
#pragma unroll
                for (int c = 0; c < NCH; ++c) {
                    float x[1][8], y[1][8];
                    load_bslice<1>(Bs + (size_t(t - 1) * K + j) * r + c * 256, r - c * 256, lane, true, x);
                    load_bslice<1>(Bs + (size_t(t - 1) * K + j2) * r + c * 256, r - c * 256, lane, j2 < K, y);
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        pa = fmaf(qv[c][e], x[0][e], pa);
                        pb = fmaf(qv[c][e], y[0][e], pb);
                    }
                }
            }
            if (j2 < K) {
#pragma unroll
                for (int o = 16; o; o >>= 1) {  // two shuffle trees, interleaved
                    pa += __shfl_xor_sync(kFull, pa, o);
                    pb += __shfl_xor_sync(kFull, pb, o);
                }
                if (lane == 0) {
                    so[j] = vrow[j] + pa;
                    so[j2] = vrow[j2] + pb;
                }
            } else {
                pa = warp_sum(pa);
                if (lane == 0) so[j] = vrow[j] + pa;
            }
        }
    }
}

// Sum 16 per-lane values over the warp at once: at each butterfly level a lane
// keeps half of its values and adds its partner's copy of them, so 16 shuffles in
// 5 levels replace 16 separate 5-level reductions.  Each partial pairs the same
// lanes as warp_sum at the same level, so the sums are bit-identical to
// warp_sum's.  Returns u = (lane >> 1) & 15: on return v[0] of this lane is the
// warp-wide sum of the lanes' v[u].
__device__ __forceinline__ int reduce16_transpose(float v[16], int lane) {
#pragma unroll
    for (int m = 16, h = 8; m >= 2; m >>= 1, h >>= 1) {
        const bool upper = (lane & m) != 0;
#pragma unroll
        for (int i = 0; i < h; ++i) {
            const float send = upper ? v[i] : v[i + h];
            const float keep = upper ? v[i + h] : v[i];
            v[i] = keep + __shfl_xor_sync(kFull, send, m);
        }
    }
    v[0] += __shfl_xor_sync(kFull, v[0], 1);
    return (lane >> 1) & 15;
}

__host__ __device__ inline size_t lattice_slot_smem(int K, int r) {
    return size_t(K) * 2 * r * 2 + size_t(r) * 4 + size_t(K) * K * 4 + size_t(K) * 12 + size_t(r) * 2 + 80;
}

// Offset of the teacher-forced predecessor's A row [r] bf16 in the slot layout.
__host__ __device__ inline size_t slot_pred_row_off(int K, int r) {
    return (size_t(K) * 2 * r * 2 + size_t(r) * 4 + size_t(K) * K * 4 + size_t(K) * 12 + 15) / 16 * 16;
}

// Lattice slot t-1 of request q, in two halves so that the part that needs only
// row t's own candidates can run before the CTA learns row t-1's: slot_stage_begin
// starts the copies of row t's B rows and G row; slot_finish stages the
// predecessors' A rows (the anchor alone for t = 1, else row t-1's K candidates),
// scores every pair with the walk's arithmetic (gate slices, fmaf chains,
// shuffle-tree sums: each entry bit-identical to the score the walk computes for
// that pair) into shared memory, and reduces each predecessor's row to its best
// candidate (value, then the lower token id, then the lower column).  Shared
// memory layout (lattice_slot_smem bytes at smem): B rows [K][r] bf16, A rows
// [K][r] bf16, G [r] fp32, slot [K][K] fp32, then row t's values and ids and the
// predecessor ids.  slot_stage_begin returns false when a candidate id of row t is
// out of range (nothing is copied).
__device__ __forceinline__ bool slot_stage_begin(int64_t row, const int32_t* __restrict__ ids,
                                                 const float* __restrict__ G,
                                                 const uint16_t* __restrict__ Bc,
                                                 const uint16_t* __restrict__ A, int32_t pred_id, int64_t V,
                                                 int K, int r, uint8_t* smem) {
    __shared__ int bad;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, nwarps = blockDim.x >> 5;
    uint16_t* Bs = reinterpret_cast<uint16_t*>(smem);
    float* Gs = reinterpret_cast<float*>(Bs + size_t(2) * K * r);
    if (tid == 0) bad = 0;
    __syncthreads();
    for (int j = tid; j < K; j += blockDim.x) {
        const int32_t b = __ldcg(ids + row * K + j);
        if (b < 0 || b >= V) bad = 1;
    }
    __syncthreads();
    if (bad) return false;
    const int cpr = r / 8;
    for (int j = warp; j < K; j += nwarps) {
        const int32_t b = __ldcg(ids + row * K + j);
        for (int c = lane; c < cpr; c += 32) cp_async16(Bs + size_t(j) * r + c * 8, Bc + int64_t(b) * r + c * 8);
    }
    for (int c = tid; c < r / 4; c += blockDim.x) cp_async16(Gs + c * 4, G + row * r + c * 4);
    if (pred_id >= 0 && pred_id < V) {
        uint16_t* Ap = reinterpret_cast<uint16_t*>(smem + slot_pred_row_off(K, r));
        for (int c = tid; c < cpr; c += blockDim.x) cp_async16(Ap + c * 8, A + int64_t(pred_id) * r + c * 8);
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
    return true;
}

// Teacher-forced scores of row `row` from the rows slot_stage_begin staged (its
// candidates' B rows, G and the predecessor's A row), every copy landed: warp w
// scores candidates w, w+8, ... with the lane slicing and shuffle tree of
// pair_scores_kernel (bit-identical).  The candidates' ids are in range.
template <int NCH>
__device__ __forceinline__ void pair_row_staged(int64_t row, bool pred_ok, const float* __restrict__ vals,
                                                int K, int r, const uint8_t* smem,
                                                float* __restrict__ scores) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nwarps = blockDim.x >> 5;
    if (!pred_ok) {
        for (int j = threadIdx.x; j < K; j += blockDim.x) scores[row * K + j] = __int_as_float(0x7fc00000);
        return;
    }
    const uint16_t* Bs = reinterpret_cast<const uint16_t*>(smem);
    const float* Gs = reinterpret_cast<const float*>(Bs + size_t(2) * K * r);
    const uint16_t* Ap = reinterpret_cast<const uint16_t*>(smem + slot_pred_row_off(K, r));
    float qv[NCH][8];
#pragma unroll
    for (int c = 0; c < NCH; ++c) {
        const int i0 = c * 256 + lane * 8;
        float af[8], gc[1][8];
        load_gslice<1>(Gs + c * 256, r - c * 256, lane, gc);
        if (i0 < r) {
            unpack8(*reinterpret_cast<const uint4*>(Ap + i0), af);
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) af[e] = 0.f;
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) qv[c][e] = af[e] * gc[0][e];
    }
    for (int j = warp; j < K; j += nwarps) {
        float part = 0.f;
#pragma unroll
        for (int c = 0; c < NCH; ++c) {
            float bf[1][8];
            load_bslice<1>(Bs + size_t(j) * r + c * 256, r - c * 256, lane, true, bf);
#pragma unroll
            for (int e = 0; e < 8; ++e) part = fmaf(qv[c][e], bf[0][e], part);
        }
        const float d = warp_sum(part);
        if (lane == 0) scores[row * K + j] = __ldcg(vals + row * K + j) + d;
    }
}

// Row t's unary values and candidate ids into the slot layout (vs, cs).
__device__ __forceinline__ void slot_load_row(int64_t row, const int32_t* __restrict__ ids,
                                              const float* __restrict__ vals, int K, int r, uint8_t* smem) {
    float* vs = reinterpret_cast<float*>(smem + size_t(K) * 2 * r * 2 + size_t(r) * 4 + size_t(K) * K * 4);
    int* cs = reinterpret_cast<int*>(vs + K);
    for (int i = threadIdx.x; i < K; i += blockDim.x) {
        vs[i] = __ldcg(vals + row * K + i);
        cs[i] = __ldcg(ids + row * K + i);
    }
}

// Scores slot t-1 from staged rows: the candidates' B rows and G (slot_stage_begin,
// landed), row t's values and ids (slot_load_row, or slot_finish's own loads), and
// the predecessors' A rows [rows][r] at As; best_j/best_v/best_id[i] for each
// predecessor i < rows.  Starts with a CTA barrier (the staged rows are visible).
// PAIRS: a warp may score two predecessor rows at once (more registers).
template <int NCH, bool PAIRS = true>
__device__ __forceinline__ void slot_score(int rows, int K, int r, uint8_t* smem, const uint16_t* As,
                                           int* best_j, float* best_v, int* best_id) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, nwarps = blockDim.x >> 5;
    const uint16_t* Bs = reinterpret_cast<const uint16_t*>(smem);
    const float* Gs = reinterpret_cast<const float*>(Bs + size_t(2) * K * r);
    float* Ls = const_cast<float*>(Gs) + r;    // [K][K]
    const float* vs = Ls + size_t(K) * K;      // [K] unary values of row t
    const int* cs = reinterpret_cast<const int*>(vs + K);  // [K] candidate ids of row t
    __syncthreads();
    const int jblocks = (K + 15) / 16;
    const int n_items = rows * jblocks;
    // the predecessor's gate slices, A[i] (.) G, in the walk's lane slicing
    auto gate = [&](int i, float (&qv)[NCH][8]) {
#pragma unroll
        for (int c = 0; c < NCH; ++c) {
            const int i0 = c * 256 + lane * 8;
            float af[8], gc[1][8];
            load_gslice<1>(Gs + c * 256, r - c * 256, lane, gc);
            if (i0 < r) {
                unpack8(*reinterpret_cast<const uint4*>(As + size_t(i) * r + i0), af);
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e) af[e] = 0.f;
            }
#pragma unroll
            for (int e = 0; e < 8; ++e) qv[c][e] = af[e] * gc[0][e];
        }
    };
    bool paired = false;
    if constexpr (NCH <= 2 && PAIRS) {
        // a warp scores items `item` and `item + nwarps` together (the same 16
        // candidates when nwarps is a multiple of jblocks): each candidate slice is
        // loaded once for both, and the two sets of fmaf chains hide each other's
        // latency.  Every sum is formed as in the one-item loop below.
        paired = nwarps % jblocks == 0;
        for (int item = warp; paired && item < n_items; item += 2 * nwarps) {
            const int itemb = item + nwarps;
            const bool hasb = itemb < n_items;
            const int i = item / jblocks, j0 = (item % jblocks) * 16;
            const int ib = hasb ? itemb / jblocks : i;
            float qa[NCH][8], qb[NCH][8];
            gate(i, qa);
            gate(ib, qb);
            float pa[16], pb[16];
#pragma unroll
            for (int u = 0; u < 16; ++u) {
                pa[u] = 0.f;
                pb[u] = 0.f;
            }
#pragma unroll
            for (int c = 0; c < NCH; ++c) {
                const int i0 = c * 256 + lane * 8;
                uint4 raw[16];
#pragma unroll
                for (int u = 0; u < 16; ++u) {
                    const int j = j0 + u < K ? j0 + u : j0;  // rows past K: loaded, not used
                    raw[u] = i0 < r ? *reinterpret_cast<const uint4*>(Bs + size_t(j) * r + i0)
                                    : make_uint4(0, 0, 0, 0);
                }
#pragma unroll
                for (int u = 0; u < 16; ++u) {
                    if (j0 + u < K) {
                        float bf[8];
                        unpack8(raw[u], bf);
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            pa[u] = fmaf(qa[c][e], bf[e], pa[u]);
                            pb[u] = fmaf(qb[c][e], bf[e], pb[u]);
                        }
                    }
                }
            }
            const int u = reduce16_transpose(pa, lane);
            if ((lane & 1) == 0 && j0 + u < K) Ls[size_t(i) * K + j0 + u] = vs[j0 + u] + pa[0];
            if (hasb) {
                const int ub = reduce16_transpose(pb, lane);
                if ((lane & 1) == 0 && j0 + ub < K) Ls[size_t(ib) * K + j0 + ub] = vs[j0 + ub] + pb[0];
            }
        }
    }
    if (!paired) {
        for (int item = warp; item < n_items; item += nwarps) {
            const int i = item / jblocks, j0 = (item % jblocks) * 16;
            float qv[NCH][8];
            gate(i, qv);
            float part[16];
#pragma unroll
            for (int u = 0; u < 16; ++u) {
                part[u] = 0.f;
                if (j0 + u < K) {
#pragma unroll
                    for (int c = 0; c < NCH; ++c) {
                        float bf[1][8];
                        load_bslice<1>(Bs + size_t(j0 + u) * r + c * 256, r - c * 256, lane, true, bf);
#pragma unroll
                        for (int e = 0; e < 8; ++e) part[u] = fmaf(qv[c][e], bf[0][e], part[u]);
                    }
                }
            }
            const int u = reduce16_transpose(part, lane);
            if ((lane & 1) == 0 && j0 + u < K) Ls[size_t(i) * K + j0 + u] = vs[j0 + u] + part[0];
        }
    }
    __syncthreads();
    for (int i = tid; i < rows; i += blockDim.x) {
        float bv = -INFINITY;
        int bid = INT_MAX, bj = -1;
        if (K % 4 == 0) {
            // the row in 16-byte pieces (fewer shared-memory wavefronts), same scan order
            for (int j4 = 0; j4 < K; j4 += 4) {
                const float4 v4 = *reinterpret_cast<const float4*>(Ls + size_t(i) * K + j4);
                const int4 c4 = *reinterpret_cast<const int4*>(cs + j4);
                const float vv[4] = {v4.x, v4.y, v4.z, v4.w};
                const int cc[4] = {c4.x, c4.y, c4.z, c4.w};
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    if (bj < 0 || ranks_before(vv[e], cc[e], bv, bid)) {
                        bv = vv[e];
                        bid = cc[e];
                        bj = j4 + e;
                    }
            }
        } else {
            for (int j = 0; j < K; ++j) {
                const float v = Ls[size_t(i) * K + j];
                if (bj < 0 || ranks_before(v, cs[j], bv, bid)) {
                    bv = v;
                    bid = cs[j];
                    bj = j;
                }
            }
        }
        best_j[i] = bj;
        best_v[i] = bv;
        best_id[i] = bid;
    }
}

// Finishes the slot started by slot_stage_begin: fetches the predecessors' A rows
// itself, then slot_score.  best_j/best_v/best_id[i] for each predecessor i < rows
// (rows = 1 and the anchor when pred_row < 0).  Returns false when a predecessor id
// is out of range (the outputs are untouched).
template <int NCH, bool PAIRS = true>
__device__ __forceinline__ bool slot_finish(int64_t row, int64_t pred_row, int32_t anchor,
                                            const int32_t* __restrict__ ids,
                                            const float* __restrict__ vals,
                                            const uint16_t* __restrict__ A, int64_t V, int K, int r,
                                            uint8_t* smem, int* best_j, float* best_v, int* best_id) {
    __shared__ int bad;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, nwarps = blockDim.x >> 5;
    const int rows = pred_row < 0 ? 1 : K;
    uint16_t* Bs = reinterpret_cast<uint16_t*>(smem);
    uint16_t* As = Bs + size_t(K) * r;
    float* Gs = reinterpret_cast<float*>(As + size_t(K) * r);
    float* Ls = Gs + r;                        // [K][K]
    float* vs = Ls + size_t(K) * K;            // [K] unary values of row t
    int* cs = reinterpret_cast<int*>(vs + K);  // [K] candidate ids of row t
    int* ps = cs + K;                          // [K] predecessor ids
    if (tid == 0) bad = 0;
    __syncthreads();
    for (int i = tid; i < K; i += blockDim.x) {
        vs[i] = __ldcg(vals + row * K + i);
        cs[i] = __ldcg(ids + row * K + i);
        if (i < rows) {
            const int32_t a = pred_row < 0 ? anchor : __ldcg(ids + pred_row * K + i);
            ps[i] = a;
            if (a < 0 || a >= V) bad = 1;
        }
    }
    __syncthreads();
    if (bad) {
        asm volatile("cp.async.wait_all;" ::: "memory");
        return false;
    }
    const int cpr = r / 8;
    for (int i = warp; i < rows; i += nwarps)
        for (int c = lane; c < cpr; c += 32) cp_async16(As + size_t(i) * r + c * 8, A + int64_t(ps[i]) * r + c * 8);
    asm volatile("cp.async.commit_group;\n\tcp.async.wait_all;" ::: "memory");
    slot_score<NCH, PAIRS>(rows, K, r, smem, As, best_j, best_v, best_id);
    return true;
}

// Teacher-forced scores of row p by one warp: every candidate with the lane
// slicing and shuffle tree of pair_scores_kernel (bit-identical), four candidates
// in flight.  kFresh: the row's list was written earlier in the same kernel.
// Returns false when pred[p] or a candidate id is out of range (NaN written there).
template <int NCH, bool kFresh>
__device__ __forceinline__ bool pair_row_warp(int64_t p, const int32_t* __restrict__ pred,
                                              const int32_t* __restrict__ ids,
                                              const float* __restrict__ vals,
                                              const float* __restrict__ G,
                                              const uint16_t* __restrict__ A,
                                              const uint16_t* __restrict__ Bc, int64_t V, int K, int r,
                                              float* __restrict__ scores) {
    const int lane = threadIdx.x & 31;
    const float nan = __int_as_float(0x7fc00000);
    const int32_t a = __ldg(pred + p);
    if (a < 0 || a >= V) {
        for (int j = lane; j < K; j += 32) scores[p * K + j] = nan;
        return false;
    }
    float qv[NCH][8];
    load_gate<NCH>(A, a, r, G + p * r, lane, qv);
    bool ok = true;
    for (int j0 = 0; j0 < K; j0 += 4) {
        float part[4];
        int32_t b[4];
        bool inr[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const bool has = j0 + u < K;
            b[u] = has ? (kFresh ? __ldcg(ids + p * K + j0 + u) : __ldg(ids + p * K + j0 + u)) : 0;
            inr[u] = b[u] >= 0 && b[u] < V;
            part[u] = (has && inr[u]) ? dot_lane<NCH>(Bc, b[u], r, lane, qv) : 0.f;
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const float d = warp_sum(part[u]);
            if (j0 + u < K) {
                if (lane == 0) {
                    const float uv = kFresh ? __ldcg(vals + p * K + j0 + u) : __ldg(vals + p * K + j0 + u);
                    scores[p * K + j0 + u] = inr[u] ? uv + d : nan;
                }
                ok = ok && inr[u];
            }
        }
    }
    return ok;
}

}  // namespace sel
}  // namespace df2
