// The fused tail of the draft head: after the head kernel has left its sorted
// per-CTA (or per-range) top-K lists in the workspace, one launch finishes the
// selector's part of the cycle with the lattice schedule ("DFlash 2
// Explanation", "How It Works", Problem 1: all adjacent pairs are scored in one
// parallel pass, and only the final walk over the finished scores is sequential).
//
// Each request's B rows form one thread-block cluster; CTA t of the cluster owns
// row t:
//   1. every CTA folds its row's lists into the row's top-K (merge_position),
//      then starts copying its candidates' B rows, its G row and its
//      teacher-forced predecessor's A row, and sends CTA t+1 the A rows of its
//      candidates (CTA 0: of the anchor), the predecessors of slot t: 1-D bulk
//      copies from global memory into CTA t+1's shared memory, completing on
//      CTA t+1's barrier, so that CTA t+1 neither waits for a cluster barrier nor
//      reads row t's ids before it can fetch them.  (Where those rows do not fit
//      in shared memory, every CTA prefetches its candidates' A rows into L2
//      instead, and a cluster barrier marks every row folded.)
//   2. CTA t >= 1 scores lattice slot t-1 (every candidate of row t after every
//      candidate of row t-1, after the anchor for t = 1) with the walk's own
//      arithmetic, reduces each predecessor's row to its best candidate, and
//      writes those argmaxes into CTA 0's shared memory; every CTA then scores
//      its row after its teacher-forced predecessor from the rows it staged
//      (pair_row_staged; verl-SpeCo PR #62, "Selector training objective");
//   -- cluster barrier --
//   3. CTA 0 walks: from the anchor, each step follows the stored argmax of the
//      current predecessor's row (vLLM Speculators "DFlash2" guide, "Candidate
//      Selector": start at the anchor, feed the best successor in as the next
//      predecessor).
// Every score uses the lane slicing, fmaf chains and shuffle-tree sums of the
// separate walk and teacher-forced kernels, and every argmax the same order
// (value, then the lower token id, then the lower column), so the outputs are
// bit-identical to the separate calls'.  The cluster barriers are the hardware's;
// the wait for the sent rows is an mbarrier wait with the library's bound.
#include <cooperative_groups.h>

#include <mutex>
#include <unordered_map>

#include "common.cuh"
#include "kernels.h"
#include "selector_dev.cuh"
#include "tc_pair.cuh"
#include "topk_merge_dev.cuh"

namespace df2 {

namespace {

namespace cg = cooperative_groups;

constexpr int kTailThreads = 256;
static_assert(kTailThreads == mrg::kMergeThreads, "the phases share one CTA shape");
constexpr int kMaxCluster = 16;
constexpr int kMaxLatticeK = 32;

// Dynamic shared memory: the merge's and the slot's layouts overlap at offset 0;
// CTA 0's argmax table follows both.
size_t tail_tab_off(int K, int r, int S) {
    const size_t a = mrg::merge_smem(S, K), b = sel::lattice_slot_smem(K, r);
    return ((a > b ? a : b) + 15) / 16 * 16;
}
size_t tail_smem(int B, int K, int r, int S) { return tail_tab_off(K, r, S) + size_t(B - 1) * K * 12 + 16; }

// The rows a CTA receives from its predecessor CTA ([K][r] bf16), the sender's
// verdict on their ids and the barrier they complete on, after the table.
constexpr size_t kTailSmemLimit = 200 * 1024;
size_t tail_push_off(int B, int K, int r, int S) { return (tail_smem(B, K, r, S) + 15) / 16 * 16; }
size_t tail_push_smem(int B, int K, int r, int S) {
    return tail_push_off(B, K, r, S) + (size_t(K) * r * 2 + 15) / 16 * 16 + 16;
}
bool tail_push_fits(int B, int K, int r, int S) { return tail_push_smem(B, K, r, S) <= kTailSmemLimit; }

// 1-D bulk copy global -> the shared memory of a CTA of the cluster (dst and bar:
// shared::cluster addresses), completing the bytes on that CTA's barrier.
__device__ __forceinline__ void bulk_load_remote(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     dst),
                 "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}
__device__ __forceinline__ void arrive_expect_tx_remote(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.release.cluster.shared::cluster.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void st_remote_u32(uint32_t addr, uint32_t v) {
    asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ void cluster_arrive() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }

// MINB: CTAs per SM the registers must allow.  1: the fast instance (a warp scores
// two predecessor rows at once); 4: for launches with more clusters than the fast
// instance holds at once, which then run in one wave instead of two.
template <int R, int NCH, int MINB>
__global__ void __launch_bounds__(kTailThreads, MINB)
draft_tail_kernel(const float* __restrict__ part_v, const int* __restrict__ part_id, int S, int64_t P,
                  int K, int32_t* __restrict__ ids, float* __restrict__ vals,
                  const int32_t* __restrict__ anchors, int B, const float* __restrict__ G,
                  const uint16_t* __restrict__ A, const uint16_t* __restrict__ Bc, int64_t V, int r,
                  int32_t* __restrict__ path, float* __restrict__ path_scores,
                  const int32_t* __restrict__ pred, float* __restrict__ pair_scores,
                  int32_t* __restrict__ dev_status, unsigned tab_off, unsigned push_off, LogitMap lm,
                  Refine rf) {
    extern __shared__ __align__(16) uint8_t smem[];
    cg::cluster_group cluster = cg::this_cluster();
    const int t = int(cluster.block_rank());
    const int64_t p = blockIdx.x;
    const int q = int(p / B), T = B - 1;
    const int warp = threadIdx.x >> 5;
    // CTA 0's table: for slot s and predecessor i, the best candidate's column,
    // token id and score
    int* tab_j = reinterpret_cast<int*>(smem + tab_off);
    int* tab_id = tab_j + T * K;
    float* tab_v = reinterpret_cast<float*>(tab_id + T * K);
    int* tab_bad = reinterpret_cast<int*>(tab_v + T * K);
    // push_off != 0: the rows this CTA receives from CTA t-1 (see the layout above)
    const bool push = push_off != 0;
    uint16_t* in_rows = reinterpret_cast<uint16_t*>(smem + push_off);
    int* in_bad = reinterpret_cast<int*>(smem + push_off + (size_t(K) * r * 2 + 15) / 16 * 16);
    uint64_t* in_bar = reinterpret_cast<uint64_t*>(in_bad + 2);
    if (threadIdx.x == 0) {
        if (t == 0) *tab_bad = 0;
        if (push) {
            *in_bad = 0;
            tc::mbar_init(in_bar, 1);
            tc::fence_mbar_init();
        }
    }
    __syncthreads();
    // push: every CTA's barrier and flags are initialised before the first remote
    // access; the wait comes after the fold, so the barrier's latency hides under it
    if (push) cluster_arrive();

    mrg::merge_position<R>(part_v, part_id, S, P, K, p, ids, vals, smem, lm, rf);
    __syncthreads();  // row p's list is written (by warp 0) and smem is free again
    // push: send CTA t+1 its predecessors' rows as soon as this row is folded
    if (push) {
        cluster_wait();
        if (t < T && warp == 0) {
            // the predecessors of slot t: the anchor (t = 0) or this row's candidates
            const int lane = threadIdx.x & 31;
            const int n = t == 0 ? 1 : K;
            int32_t a[kMaxLatticeK / 32 > 0 ? kMaxLatticeK / 32 : 1];
            bool bad = false;
#pragma unroll
            for (int k = 0; k < kMaxLatticeK / 32; ++k) {
                const int i = k * 32 + lane;
                a[k] = i < n ? (t == 0 ? __ldg(anchors + q) : __ldcg(ids + p * K + i)) : 0;
                bad |= i < n && (a[k] < 0 || a[k] >= V);
            }
            bad = __any_sync(kFull, bad);
            const uint32_t nx = uint32_t(t + 1);
            const uint32_t bar = tc::mapa_shared(tc::smem_u32(in_bar), nx);
            if (bad) {
                if (lane == 0) {
                    st_remote_u32(tc::mapa_shared(tc::smem_u32(in_bad), nx), 1u);
                    tc::mbar_arrive_cluster(bar);  // releases the flag
                }
            } else {
                if (lane == 0) arrive_expect_tx_remote(bar, uint32_t(n) * uint32_t(r) * 2u);
                __syncwarp();
                const uint32_t dst = tc::mapa_shared(tc::smem_u32(in_rows), nx);
#pragma unroll
                for (int k = 0; k < kMaxLatticeK / 32; ++k) {
                    const int i = k * 32 + lane;
                    if (i < n)
                        bulk_load_remote(dst + uint32_t(i) * uint32_t(r) * 2u, A + int64_t(a[k]) * r,
                                         uint32_t(r) * 2u, bar);
                }
            }
        }
    }
    const int32_t pid = pred ? __ldg(pred + p) : -1;
    const bool pred_ok = pid >= 0 && pid < V;
    // row p's candidates' B rows, its G row and its teacher-forced predecessor's A row
    const bool staged = sel::slot_stage_begin(p, ids, G, Bc, A, pid, V, K, r, smem);
    if (!push) {
        if (t < T) {
            // the next row's predecessors are this row's candidates: warm L2 with their A rows
            const int lines = (r * 2 + 127) / 128;
            for (int e = threadIdx.x; e < K * lines; e += blockDim.x) {
                const int32_t a = __ldcg(ids + p * K + e / lines);
                if (a >= 0 && a < V)
                    asm volatile("prefetch.global.L2 [%0];" ::"l"(A + int64_t(a) * r + (e % lines) * 64));
            }
        }
        __threadfence();
        cluster.sync();
    }

    bool slot_ok = true;
    if (t >= 1) {
        int* rj = cluster.map_shared_rank(tab_j, 0) + size_t(t - 1) * K;
        int* rid = cluster.map_shared_rank(tab_id, 0) + size_t(t - 1) * K;
        float* rv = cluster.map_shared_rank(tab_v, 0) + size_t(t - 1) * K;
        if (push) {
            sel::slot_load_row(p, ids, vals, K, r, smem);
            // this CTA's own copies (B rows, G, the teacher-forced row), then the rows
            // CTA t-1 sent (bounded wait; a timeout fails the slot)
            asm volatile("cp.async.wait_all;" ::: "memory");
            volatile int never = 0;
            const bool got = tc::mbar_wait_cluster(in_bar, 0, &never);
            const bool ok_in = __syncthreads_and(got && *in_bad == 0) != 0;
            if (!got && threadIdx.x == 0 && dev_status) atomicOr(dev_status, DF2_STATUS_WAIT_TIMEOUT);
            slot_ok = staged && ok_in;
            if (slot_ok) sel::slot_score<NCH, (MINB < 4)>(t == 1 ? 1 : K, K, r, smem, in_rows, rj, rv, rid);
        } else {
            slot_ok = staged && sel::slot_finish<NCH, (MINB < 4)>(p, t == 1 ? -1 : p - 1, __ldg(anchors + q), ids, vals, A,
                                                      V, K, r, smem, rj, rv, rid);
        }
        if (!slot_ok && threadIdx.x == 0) *cluster.map_shared_rank(tab_bad, 0) = 1;
    } else if (staged) {
        asm volatile("cp.async.wait_all;" ::: "memory");
        __syncthreads();
    }
    if (pred) {
        // row p's teacher-forced scores: from the staged rows when they are all there
        if (staged && (t == 0 || slot_ok)) {
            sel::pair_row_staged<NCH>(p, pred_ok, vals, K, r, smem, pair_scores);
            if (!pred_ok && threadIdx.x == 0 && dev_status) atomicOr(dev_status, DF2_STATUS_ID_OUT_OF_RANGE);
        } else if (warp == 0) {
            if (!sel::pair_row_warp<NCH, true>(p, pred, ids, vals, G, A, Bc, V, K, r, pair_scores) && dev_status &&
                (threadIdx.x & 31) == 0)
                atomicOr(dev_status, DF2_STATUS_ID_OUT_OF_RANGE);
        }
    }
    cluster.sync();

    if (t == 0 && threadIdx.x == 0) {
        const int32_t a0 = __ldg(anchors + q);
        if (*tab_bad || a0 < 0 || a0 >= V) {
            for (int s = 0; s < T; ++s) {
                path[int64_t(q) * T + s] = -1;
                path_scores[int64_t(q) * T + s] = __int_as_float(0x7fc00000);
            }
            if (dev_status) atomicOr(dev_status, DF2_STATUS_ID_OUT_OF_RANGE);
        } else {
            int i = 0;
            for (int s = 0; s < T; ++s) {
                const int at = s * K + i;
                path[int64_t(q) * T + s] = tab_id[at];
                path_scores[int64_t(q) * T + s] = tab_v[at];
                i = tab_j[at];
            }
        }
    }
}

template <int R, int N, int MINB>
cudaError_t launch_tail(int64_t P, int B, size_t smem, cudaStream_t stream, const TopkParts& parts, int K,
                        int32_t* ids, float* vals, const int32_t* anchors, const float* G,
                        const uint16_t* A, const uint16_t* Bc, int64_t V, int r, int32_t* path,
                        float* path_scores, const int32_t* pred, float* pair_scores, int32_t* dev_status,
                        LogitMap lm, Refine rf, bool probe_only, bool* fits, int* max_clusters) {
    auto kernel = draft_tail_kernel<R, N, MINB>;
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (e != cudaSuccess) return e;
    if (B > 8) {
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return e;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(P));
    cfg.blockDim = dim3(kTailThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = unsigned(B);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (probe_only) {
        int clusters = 0;
        e = cudaOccupancyMaxActiveClusters(&clusters, kernel, &cfg);
        *fits = e == cudaSuccess && clusters > 0;
        if (max_clusters) *max_clusters = e == cudaSuccess ? clusters : 0;
        return e;
    }
    const unsigned push_off = tail_push_fits(B, K, r, parts.S) ? unsigned(tail_push_off(B, K, r, parts.S)) : 0u;
    return cudaLaunchKernelEx(&cfg, kernel, parts.v, parts.id, parts.S, P, K, ids, vals, anchors, B, G, A,
                              Bc, V, r, path, path_scores, pred, pair_scores, dev_status,
                              unsigned(tail_tab_off(K, r, parts.S)), push_off, lm, rf);
}

// Runs (or, probe_only, checks that the cluster shape can run) the right instance.
// many: the launch has more clusters than the fast instance holds at once.
cudaError_t dispatch_tail(bool probe_only, bool* fits, const TopkParts& parts, int64_t P, int K, int32_t* ids,
                          float* vals, const int32_t* anchors, int B, const float* G, const uint16_t* A,
                          const uint16_t* Bc, int64_t V, int r, int32_t* path, float* path_scores,
                          const int32_t* pred, float* pair_scores, int32_t* dev_status, LogitMap lm,
                          Refine rf, cudaStream_t stream, bool many = false, int* max_clusters = nullptr) {
    const size_t smem = tail_push_fits(B, K, r, parts.S) ? tail_push_smem(B, K, r, parts.S)
                                                          : tail_smem(B, K, r, parts.S);
    const int nch = (r + 255) / 256;
    cudaError_t e = cudaSuccess;
#define DF2_TAIL(RV, N, MB)                                                                            \
    e = launch_tail<RV, N, MB>(P, B, smem, stream, parts, K, ids, vals, anchors, G, A, Bc, V, r, path, \
                               path_scores, pred, pair_scores, dev_status, lm, rf, probe_only, fits,    \
                               max_clusters)
#define DF2_TAIL_N(RV)                                         \
    do {                                                       \
        if (nch <= 1) {                                        \
            if (many) DF2_TAIL(RV, 1, 4);                      \
            else DF2_TAIL(RV, 1, 1);                           \
        } else if (nch <= 2) {                                 \
            if (many) DF2_TAIL(RV, 2, 4);                      \
            else DF2_TAIL(RV, 2, 1);                           \
        } else if (nch <= 4) DF2_TAIL(RV, 4, 1);               \
        else if (nch <= 8) DF2_TAIL(RV, 8, 1);                 \
        else DF2_TAIL(RV, 16, 1);                              \
    } while (0)
    if (K <= 32) DF2_TAIL_N(1);
    else DF2_TAIL_N(2);
#undef DF2_TAIL_N
#undef DF2_TAIL
    return e;
}

std::mutex g_fit_mu;
std::unordered_map<uint64_t, bool> g_fit;  // cluster-shape probe results
std::unordered_map<uint64_t, int> g_clusters;  // clusters at once per instance (key | many)

}  // namespace

bool draft_tail_supported(int64_t P, int B, int K, int r, int S, int num_sms) {
    (void)num_sms;
    // the lattice costs K times the greedy walk's products: worth its latency only
    // for short candidate lists
    if (P < 1 || B < 2 || B > kMaxCluster || K > kMaxLatticeK || r > 4096 || P % B != 0) return false;
    if (tail_smem(B, K, r, S) > kTailSmemLimit) return false;
    // whether one cluster of this shape fits on an SM group depends on the cluster
    // size, the instance and its shared memory, not on P: probe once per device
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    const size_t smem = tail_push_fits(B, K, r, S) ? tail_push_smem(B, K, r, S) : tail_smem(B, K, r, S);
    const uint64_t key = (uint64_t(unsigned(dev)) << 48) ^ (uint64_t(B) << 40) ^
                         (uint64_t(K <= 32) << 37) ^ (uint64_t((r + 255) / 256) << 32) ^
                         uint64_t(smem);
    {
        std::lock_guard<std::mutex> lock(g_fit_mu);
        auto it = g_fit.find(key);
        if (it != g_fit.end()) return it->second;
    }
    bool fits = false;
    const TopkParts probe{nullptr, nullptr, S};
    static const uint16_t probe_row = 0;  // any non-null operand: the tail always refines
    if (dispatch_tail(true, &fits, probe, P, K, nullptr, nullptr, nullptr, B, nullptr, nullptr, nullptr, 1, r,
                      nullptr, nullptr, nullptr, nullptr, nullptr, LogitMap{}, Refine{&probe_row, nullptr, 0},
                      nullptr) != cudaSuccess)
        fits = false;
    std::lock_guard<std::mutex> lock(g_fit_mu);
    g_fit[key] = fits;
    return fits;
}

// Clusters of the fast (many = false) or the four-CTAs-per-SM instance that fit at
// once for this shape, from the occupancy query, cached per device and shape.
int tail_max_clusters(int S, int K, int B, int r, bool many) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    const size_t smem = tail_push_fits(B, K, r, S) ? tail_push_smem(B, K, r, S) : tail_smem(B, K, r, S);
    const uint64_t key = (uint64_t(unsigned(dev)) << 48) ^ (uint64_t(B) << 40) ^ (uint64_t(many) << 38) ^
                         (uint64_t(K <= 32) << 37) ^ (uint64_t((r + 255) / 256) << 32) ^ uint64_t(smem);
    {
        std::lock_guard<std::mutex> lock(g_fit_mu);
        auto it = g_clusters.find(key);
        if (it != g_clusters.end()) return it->second;
    }
    bool fits = false;
    int clusters = 0;
    const TopkParts probe{nullptr, nullptr, S};
    static const uint16_t probe_row = 0;
    if (dispatch_tail(true, &fits, probe, B, K, nullptr, nullptr, nullptr, B, nullptr, nullptr, nullptr, 1, r,
                      nullptr, nullptr, nullptr, nullptr, nullptr, LogitMap{}, Refine{&probe_row, nullptr, 0},
                      nullptr, many, &clusters) != cudaSuccess)
        clusters = 0;
    std::lock_guard<std::mutex> lock(g_fit_mu);
    g_clusters[key] = clusters;
    return clusters;
}

cudaError_t draft_tail_launch(const TopkParts& parts, int64_t P, int K, int32_t* ids, float* vals,
                              const int32_t* anchors, int B, const float* G, const uint16_t* A,
                              const uint16_t* Bc, int64_t V, int r, int32_t* path, float* path_scores,
                              const int32_t* pred, float* pair_scores, int32_t* dev_status,
                              cudaStream_t stream, LogitMap lm, Refine rf) {
    // more clusters than the fast instance holds at once: the instance that fits
    // four CTAs per SM, if that holds more (one-row scoring, lower register count)
    bool many = false;
    if ((r + 255) / 256 <= 2) {
        const int fast = tail_max_clusters(parts.S, K, B, r, false);
        if (P / B > fast) many = tail_max_clusters(parts.S, K, B, r, true) > fast;
    }
    bool unused = false;
    const cudaError_t e = dispatch_tail(false, &unused, parts, P, K, ids, vals, anchors, B, G, A, Bc, V, r, path,
                                        path_scores, pred, pair_scores, dev_status, lm, rf, stream, many);
    note_launch();
    return e;
}

}  // namespace df2
