// Shared device helpers for libdflash2 (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <climits>
#include <cmath>

#include "dflash2.h"

#define DF2_API extern "C" __attribute__((visibility("default")))

namespace df2 {

// Host side: count one kernel launch by this library (read back through
// dflash2_kernels_launched).
void note_launch();

constexpr unsigned kFull = 0xFFFFFFFFu;

template <class T>
__host__ __device__ __forceinline__ T dmin(T a, T b) { return a < b ? a : b; }
template <class T>
__host__ __device__ __forceinline__ T dmax(T a, T b) { return a < b ? b : a; }

// bf16 -> fp32 is exact: the bf16 bits are the top half of the fp32 word.
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ float bf16_to_f32(uint16_t b) { return __uint_as_float(uint32_t(b) << 16); }

// Round-to-nearest-even fp32 -> bf16 bits (finite inputs).
__device__ __forceinline__ uint16_t f32_to_bf16_rn(float f) {
    uint32_t u = __float_as_uint(f);
    if ((u & 0x7F800000u) == 0x7F800000u) return uint16_t((u >> 16) | ((u & 0xFFFFu) ? 0x40u : 0u));
    u += 0x7FFFu + ((u >> 16) & 1u);
    return uint16_t(u >> 16);
}

__device__ __forceinline__ void unpack8(const uint4& w, float f[8]) {
    f[0] = bf16_lo(w.x); f[1] = bf16_hi(w.x);
    f[2] = bf16_lo(w.y); f[3] = bf16_hi(w.y);
    f[4] = bf16_lo(w.z); f[5] = bf16_hi(w.z);
    f[6] = bf16_lo(w.w); f[7] = bf16_hi(w.w);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
    return v;
}

// A 64-bit key whose unsigned order is the rank order below (for id >= 0, finite
// values; -0 and +0 compare equal, as floats do).
__device__ __forceinline__ unsigned long long rank_key(float v, int id) {
    const unsigned u = __float_as_uint(v + 0.0f);  // -0 -> +0
    const unsigned k = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    return (static_cast<unsigned long long>(k) << 32) | static_cast<unsigned>(0x7FFFFFFF - id);
}

// Rank order of (value, token id) pairs: larger value first, then lower id.
__device__ __forceinline__ bool ranks_before(float va, int ia, float vb, int ib) {
    return va > vb || (va == vb && ia < ib);
}

// A top-K list kept by one warp in shared memory (K entries, unsorted).  The
// bookkeeping (fill count, current worst entry) lives in registers and is the
// same in every lane.  Candidates arrive 32 at a time, one per lane; a ballot
// against the worst entry rejects almost all of them once the list is full.
struct WarpTopK {
    float* v;
    int* id;
    int K;
    int n;      // entries filled
    float wv;   // worst entry (valid once n == K)
    int wid;
    int wpos;

    __device__ __forceinline__ void init(float* v_, int* id_, int K_) {
        v = v_; id = id_; K = K_; n = 0; wv = -INFINITY; wid = INT_MAX; wpos = 0;
    }

    __device__ __forceinline__ void find_worst(int lane) {
        float bv = 0.f; int bi = 0, bp = -1;
        for (int i = lane; i < K; i += 32) {
            float vv = v[i]; int ii = id[i];
            if (bp < 0 || ranks_before(bv, bi, vv, ii)) { bv = vv; bi = ii; bp = i; }
        }
#pragma unroll
        for (int o = 16; o; o >>= 1) {
            float ov = __shfl_xor_sync(kFull, bv, o);
            int oi = __shfl_xor_sync(kFull, bi, o);
            int op = __shfl_xor_sync(kFull, bp, o);
            bool take = op >= 0 && (bp < 0 || ranks_before(bv, bi, ov, oi));
            if (take) { bv = ov; bi = oi; bp = op; }
        }
        wv = bv; wid = bi; wpos = bp;
    }

    // Every lane of the warp calls this with its own candidate.
    __device__ __forceinline__ void offer(bool valid, float cv, int cid, int lane) {
        unsigned m = __ballot_sync(kFull, valid && (n < K || ranks_before(cv, cid, wv, wid)));
        while (m) {
            const int src = __ffs(m) - 1;
            m &= m - 1;
            const float sv = __shfl_sync(kFull, cv, src);
            const int si = __shfl_sync(kFull, cid, src);
            if (n < K) {
                if (lane == 0) { v[n] = sv; id[n] = si; }
                ++n;
                __syncwarp();
                if (n == K) find_worst(lane);
            } else if (ranks_before(sv, si, wv, wid)) {
                if (lane == 0) { v[wpos] = sv; id[wpos] = si; }
                __syncwarp();
                find_worst(lane);
            }
        }
    }
};

// Writes the n entries of a list in rank order to out_ids/out_vals[0..K), each
// value passed through map and ranked by (mapped value, lower id): a map that
// rounds neighbours to one value (a saturating cap) leaves them in id order.
// Slots past n get id -1 / -inf.  Called by `nthreads` cooperating threads
// (index tid).
template <class Map>
__device__ __forceinline__ void write_sorted(const float* v, const int* id, int n, int K,
                                             int32_t* out_ids, float* out_vals, int tid,
                                             int nthreads, Map map) {
    const bool plain = map.identity();
    for (int i = tid; i < n; i += nthreads) {
        const int ii = id[i];
        const float vi = plain ? v[i] : map(v[i]);
        int rank = 0;
        if (plain)
            for (int j = 0; j < n; ++j) rank += ranks_before(v[j], id[j], vi, ii);
        else
            for (int j = 0; j < n; ++j) rank += ranks_before(map(v[j]), id[j], vi, ii);
        out_ids[rank] = ii;
        out_vals[rank] = vi;
    }
    for (int i = n + tid; i < K; i += nthreads) {
        out_ids[i] = -1;
        out_vals[i] = -INFINITY;
    }
}

}  // namespace df2
