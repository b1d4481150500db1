// Register-resident top-K for one warp, K <= 32 R (R = 1, 2 or 3 rows of 32).
//
// A list is R = ceil(K/32) "rows" of 32 entries, one entry per lane per row,
// sorted in rank order (value descending, then token id ascending) across
// (row, lane): row 0 lane 0 is the best.  A batch of 32 candidates (one per lane)
// is folded in with shuffle-based bitonic networks only -- no shared memory and
// no per-candidate serial work:
//   1. sort the batch (bitonic sort across lanes, 15 compare-exchange steps);
//   2. pair list row 0 lane i with batch lane 31-i: the better of each pair is the
//      best 32 of the union (a bitonic sequence, sorted by a 5-step merge), the
//      worse ones are the rest;
//   3. for each further row, the rest is folded into it the same way.
// Entries with id == INT_MAX are empty slots (value -inf) and rank last.
#pragma once

#include "common.cuh"

namespace df2 {
namespace wtk {

constexpr int kEmptyId = INT_MAX;

// One compare-exchange of a bitonic network: this lane keeps the better entry of
// (mine, lane ^ j) iff keep_better.
__device__ __forceinline__ void cx(float& v, int& id, int j, bool keep_better) {
    const float ov = __shfl_xor_sync(kFull, v, j);
    const int oid = __shfl_xor_sync(kFull, id, j);
    const bool mine_better = ranks_before(v, id, ov, oid);
    if (keep_better ? !mine_better : mine_better) {
        v = ov;
        id = oid;
    }
}

// Sort 32 entries across the warp into rank order (lane 0 best).
__device__ __forceinline__ void sort32(float& v, int& id, int lane) {
#pragma unroll
    for (int k = 2; k <= 32; k <<= 1) {
#pragma unroll
        for (int j = k >> 1; j > 0; j >>= 1) {
            const bool lower = (lane & j) == 0;
            const bool descending = (lane & k) == 0;  // k == 32: the whole warp, descending
            cx(v, id, j, lower == descending);
        }
    }
}

// A bitonic sequence across the warp -> rank order.
__device__ __forceinline__ void merge32(float& v, int& id, int lane) {
#pragma unroll
    for (int j = 16; j > 0; j >>= 1) cx(v, id, j, (lane & j) == 0);
}

// Fold the sorted batch (bv, bid) into the sorted row (v, id): the row becomes the
// best 32 of both; (bv, bid) is left holding the other 32, sorted.
__device__ __forceinline__ void fold_row(float& v, int& id, float& bv, int& bid, int lane) {
    const float rv = __shfl_sync(kFull, bv, 31 - lane);
    const int rid = __shfl_sync(kFull, bid, 31 - lane);
    const bool mine_better = ranks_before(v, id, rv, rid);
    const float lo_v = mine_better ? rv : v;
    const int lo_id = mine_better ? rid : id;
    if (!mine_better) {
        v = rv;
        id = rid;
    }
    merge32(v, id, lane);
    bv = lo_v;
    bid = lo_id;
    merge32(bv, bid, lane);
}

template <int R>
struct List {
    float v[R];
    int id[R];

    __device__ __forceinline__ void clear() {
#pragma unroll
        for (int r = 0; r < R; ++r) {
            v[r] = -INFINITY;
            id[r] = kEmptyId;
        }
    }

    // The K-th entry (the admission threshold), in every lane.
    __device__ __forceinline__ void kth(int K, float& tv, int& tid) const {
        const int r = (K - 1) >> 5, l = (K - 1) & 31;
        float sv = v[0];
        int sid = id[0];
#pragma unroll
        for (int rr = 1; rr < R; ++rr)
            if (rr == r) { sv = v[rr]; sid = id[rr]; }
        tv = __shfl_sync(kFull, sv, l);
        tid = __shfl_sync(kFull, sid, l);
    }

    // Offer one candidate per lane (cid = kEmptyId for none).  All lanes call.
    __device__ __forceinline__ void offer(float cv, int cid, int K, int lane) {
        float tv;
        int tid;
        kth(K, tv, tid);
        const bool pass = cid != kEmptyId && ranks_before(cv, cid, tv, tid);
        if (__ballot_sync(kFull, pass) == 0) return;
        float bv = pass ? cv : -INFINITY;
        int bid = pass ? cid : kEmptyId;
        sort32(bv, bid, lane);
        add_sorted(bv, bid, lane);
    }

    // Offer a batch already in rank order across the warp (entries that do not
    // beat the K-th are dropped; the survivors are a prefix, so order is kept).
    __device__ __forceinline__ void offer_sorted(float cv, int cid, int K, int lane) {
        float tv;
        int tid;
        kth(K, tv, tid);
        const bool pass = cid != kEmptyId && ranks_before(cv, cid, tv, tid);
        if (__ballot_sync(kFull, pass) == 0) return;
        add_sorted(pass ? cv : -INFINITY, pass ? cid : kEmptyId, lane);
    }

    // Fold a batch already in rank order across the warp.
    __device__ __forceinline__ void add_sorted(float bv, int bid, int lane) {
#pragma unroll
        for (int r = 0; r < R; ++r) fold_row(v[r], id[r], bv, bid, lane);
    }
};

}  // namespace wtk
}  // namespace df2
