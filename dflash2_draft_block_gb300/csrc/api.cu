// The C-ABI of libdflash2: argument validation, workspace sizing and dispatch.
// Every rule checked here is stated beside the call in include/dflash2.h.
#include <atomic>
#include <cfloat>
#include <cstring>

#include "common.cuh"
#include "kernels.h"
#include "head_tc.h"

namespace {

constexpr int kAbiVersion = 2;

int num_sms_current() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return n;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int from_cuda(cudaError_t e) { return e == cudaSuccess ? DF2_OK : DF2_ERR_CUDA; }

size_t round_up(size_t n, size_t a) { return (n + a - 1) / a * a; }

// The unary logits' output multiplier (finite, > 0) and final softcap (finite,
// >= 0; 0 = none) as the map the top-K kernels apply to the values they keep.
bool make_logit_map(float mul, float cap, df2::LogitMap* lm) {
    if (!(mul > 0.f) || !(mul <= FLT_MAX) || !(cap >= 0.f) || !(cap <= FLT_MAX)) return false;
    lm->mul = mul;
    lm->cap = cap;
    return true;
}

}  // namespace

DF2_API const char* dflash2_status_string(int status) {
    switch (status) {
        case DF2_OK: return "DF2_OK";
        case DF2_ERR_INVALID_ARGUMENT: return "DF2_ERR_INVALID_ARGUMENT";
        case DF2_ERR_UNSUPPORTED: return "DF2_ERR_UNSUPPORTED";
        case DF2_ERR_CUDA: return "DF2_ERR_CUDA";
        case DF2_ERR_WORKSPACE_TOO_SMALL: return "DF2_ERR_WORKSPACE_TOO_SMALL";
        case DF2_ERR_TIMEOUT: return "DF2_ERR_TIMEOUT";
        default: return "DF2_ERR_UNKNOWN";
    }
}

DF2_API int dflash2_abi_version(void) { return kAbiVersion; }

namespace {
std::atomic<long long> g_launches{0};
}  // namespace

void df2::note_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

DF2_API long long dflash2_kernels_launched(void) { return g_launches.load(std::memory_order_relaxed); }

// ------------------------------------------------------------ unary_topk --

namespace {

int check_head(int64_t P, int64_t D, int64_t V, int K, int r, bool has_wh) {
    if (P < 0 || D < 1 || V < 1 || K < 1 || K > V) return DF2_ERR_INVALID_ARGUMENT;
    if (has_wh && r < 1) return DF2_ERR_INVALID_ARGUMENT;
    if (D % 8 != 0 || K > DF2_MAX_TOPK || V > DF2_MAX_VOCAB) return DF2_ERR_UNSUPPORTED;
    if (has_wh && (r > DF2_MAX_RANK || r % 8 != 0)) return DF2_ERR_UNSUPPORTED;
    if (!df2::head_simple_supported(D, K)) return DF2_ERR_UNSUPPORTED;
    return DF2_OK;
}


enum class HeadPath { Skinny, Wide, Simple };

// Few positions: the HBM-streaming swap-AB kernel; many: the tensor-core GEMM with
// a per-position top-K epilogue; anything else (K > 64): the CUDA-core path.
HeadPath pick_head(int64_t P, int64_t D, int64_t V, int K) {
    if (df2::head_tc_supported(P, D, V, K)) return HeadPath::Skinny;
    if (df2::wide_supported(P, V, D, K)) return HeadPath::Wide;
    return HeadPath::Simple;
}

size_t head_workspace(HeadPath path, int64_t P, int64_t D, int64_t V, int K, int sms) {
    switch (path) {
        case HeadPath::Skinny: return df2::head_tc_workspace(P, D, V, K, sms);
        case HeadPath::Wide: return df2::wide_topk_workspace(P, V, K, sms);
        default: return df2::head_simple_workspace(P, D, V, K, sms);
    }
}

}  // namespace

DF2_API int dflash2_unary_topk_path(int64_t P, int64_t D, int64_t V, int K) {
    if (check_head(P, D, V, K, 0, false) != DF2_OK) return -1;
    switch (pick_head(P, D, V, K)) {
        case HeadPath::Skinny: return DF2_HEAD_PATH_STREAM;
        case HeadPath::Wide: return DF2_HEAD_PATH_GEMM;
        default: return DF2_HEAD_PATH_CUDA_CORE;
    }
}

DF2_API size_t dflash2_unary_topk_workspace_size(int64_t P, int64_t D, int64_t V, int K, int r) {
    (void)r;
    if (check_head(P, D, V, K, 0, false) != DF2_OK || P == 0) return 0;
    const int sms = num_sms_current();
    if (sms <= 0) return 0;
    return round_up(head_workspace(pick_head(P, D, V, K), P, D, V, K, sms), 256);
}

DF2_API int dflash2_unary_topk(const uint16_t* h, int64_t P, int64_t D, const uint16_t* W_lm,
                               int64_t V, int K, float output_multiplier,
                               float final_logit_softcapping, const uint16_t* W_H, int r, float* G,
                               int32_t* topk_ids, float* topk_vals, void* workspace,
                               size_t workspace_bytes, int32_t* dev_status, void* stream) {
    const bool has_wh = W_H != nullptr;
    int rc = check_head(P, D, V, K, r, has_wh);
    if (rc != DF2_OK) return rc;
    df2::LogitMap lm;
    if (!make_logit_map(output_multiplier, final_logit_softcapping, &lm)) return DF2_ERR_INVALID_ARGUMENT;
    if (P == 0) return DF2_OK;
    if (!h || !W_lm || !topk_ids || !topk_vals || (has_wh && !G)) return DF2_ERR_INVALID_ARGUMENT;
    if (!aligned16(h) || !aligned16(W_lm) || !aligned16(topk_ids) || !aligned16(topk_vals) ||
        (has_wh && (!aligned16(W_H) || !aligned16(G))) || !aligned16(workspace))
        return DF2_ERR_UNSUPPORTED;
    const int sms = num_sms_current();
    if (sms <= 0) return DF2_ERR_CUDA;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const HeadPath path = pick_head(P, D, V, K);
    const size_t need = round_up(head_workspace(path, P, D, V, K, sms), 256);
    if (workspace_bytes < need || (need > 0 && !workspace)) return DF2_ERR_WORKSPACE_TOO_SMALL;
    if (path == HeadPath::Skinny || path == HeadPath::Wide) {
        // the head leaves its sorted per-CTA lists; the merge folds them and maps the kept values
        df2::TopkParts parts{};
        if (path == HeadPath::Skinny) {
            rc = df2::head_tc_launch(h, P, D, W_lm, V, K, W_H, r, G, topk_ids, topk_vals, workspace,
                                     dev_status, sms, st, -1, &parts);
            if (rc != DF2_OK) return rc;
        } else {
            cudaError_t e = df2::wide_topk_launch(h, P, W_lm, V, D, K, topk_ids, topk_vals, workspace,
                                                  dev_status, sms, st, &parts, nullptr, 0,
                                                  has_wh ? W_H : nullptr, r, G);
            if (e != cudaSuccess) return DF2_ERR_CUDA;
        }
        return from_cuda(df2::topk_merge_sorted_launch(parts.v, parts.id, parts.S, P, K, topk_ids, topk_vals,
                                                       st, lm, df2::Refine{h, W_lm, D}));
    }
    cudaError_t e = df2::head_simple_launch(h, P, D, W_lm, V, K, topk_ids, topk_vals, workspace,
                                            sms, st, lm);
    if (e != cudaSuccess) return DF2_ERR_CUDA;
    if (has_wh) {
        e = df2::gemm_simple_launch(h, false, W_H, P, r, D, G, r, r, G, r, st);
        if (e != cudaSuccess) return DF2_ERR_CUDA;
    }
    return DF2_OK;
}

// ------------------------------------------------------------ draft head --

namespace {

// The fused path: the head kernel leaves its sorted lists in the workspace and one
// tail launch (a thread-block cluster per request) folds them, scores the
// teacher-forced pairs and the lattice, and walks each request.
bool draft_fused(HeadPath path, int64_t P, int B, int64_t D, int64_t V, int K, int r, int sms) {
    if (path == HeadPath::Simple) return false;
    int S = 0;
    if (path == HeadPath::Skinny) S = int(df2::head_tc_workspace(P, D, V, K, sms) / (size_t(P) * K * 8));
    else S = int((df2::wide_topk_workspace(P, V, K, sms) - size_t(P) * 4) / (size_t(P) * K * 8));
    return df2::draft_tail_supported(P, B, K, r, S, sms);
}

size_t draft_workspace(int64_t P, int R, int B, int64_t D, int64_t V, int K, int r, int sms) {
    const HeadPath path = pick_head(P, D, V, K);
    (void)R;
    return round_up(head_workspace(path, P, D, V, K, sms), 256);
}

}  // namespace

DF2_API size_t dflash2_draft_head_workspace_size(int R, int B, int64_t D, int64_t V, int K, int r) {
    if (R < 1 || B < 2) return 0;
    const int64_t P = int64_t(R) * B;
    if (check_head(P, D, V, K, r, true) != DF2_OK) return 0;
    const int sms = num_sms_current();
    if (sms <= 0) return 0;
    return draft_workspace(P, R, B, D, V, K, r, sms);
}

DF2_API int dflash2_draft_head(const uint16_t* h, int R, int B, int64_t D, const uint16_t* W_lm,
                               int64_t V, int K, float output_multiplier,
                               float final_logit_softcapping, const uint16_t* W_H, int r, const uint16_t* A,
                               const uint16_t* Bc, const int32_t* anchors, const int32_t* pred,
                               int32_t* topk_ids, float* topk_vals, float* G, int32_t* path,
                               float* path_scores, float* pair_scores, void* workspace,
                               size_t workspace_bytes, int32_t* dev_status, void* stream) {
    if (R < 0 || B < 2) return DF2_ERR_INVALID_ARGUMENT;
    const int64_t P = int64_t(R) * B;
    int rc = check_head(P, D, V, K, r, true);
    if (rc != DF2_OK) return rc;
    df2::LogitMap lm;
    if (!make_logit_map(output_multiplier, final_logit_softcapping, &lm)) return DF2_ERR_INVALID_ARGUMENT;
    if (r > DF2_MAX_RANK || r % 8 != 0) return DF2_ERR_UNSUPPORTED;
    if (R == 0) return DF2_OK;
    if (!h || !W_lm || !W_H || !A || !Bc || !anchors || !topk_ids || !topk_vals || !G || !path ||
        !path_scores || (pred && !pair_scores))
        return DF2_ERR_INVALID_ARGUMENT;
    if (!aligned16(h) || !aligned16(W_lm) || !aligned16(W_H) || !aligned16(A) || !aligned16(Bc) ||
        !aligned16(topk_ids) || !aligned16(topk_vals) || !aligned16(G) || !aligned16(workspace))
        return DF2_ERR_UNSUPPORTED;
    const int sms = num_sms_current();
    if (sms <= 0) return DF2_ERR_CUDA;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const HeadPath hp = pick_head(P, D, V, K);
    const size_t need = draft_workspace(P, R, B, D, V, K, r, sms);
    if (workspace_bytes < need || !workspace) return DF2_ERR_WORKSPACE_TOO_SMALL;
    if (!draft_fused(hp, P, B, D, V, K, r, sms)) {
        // the separate calls, in order
        rc = dflash2_unary_topk(h, P, D, W_lm, V, K, output_multiplier, final_logit_softcapping, W_H, r, G,
                                topk_ids, topk_vals, workspace, workspace_bytes, dev_status, stream);
        if (rc != DF2_OK) return rc;
        rc = dflash2_selector_walk(anchors, R, B, topk_ids, topk_vals, G, A, Bc, V, K, r, path,
                                   path_scores, dev_status, stream);
        if (rc != DF2_OK || !pred) return rc;
        return dflash2_selector_pair_scores(pred, P, topk_ids, topk_vals, G, A, Bc, V, K, r,
                                            pair_scores, dev_status, stream);
    }
    df2::TopkParts parts{};
    if (hp == HeadPath::Skinny) {
        rc = df2::head_tc_launch(h, P, D, W_lm, V, K, W_H, r, G, topk_ids, topk_vals, workspace,
                                 dev_status, sms, st, -1, &parts);
        if (rc != DF2_OK) return rc;
    } else {
        cudaError_t e = df2::wide_topk_launch(h, P, W_lm, V, D, K, topk_ids, topk_vals, workspace,
                                              dev_status, sms, st, &parts, nullptr, 0, W_H, r, G);
        if (e != cudaSuccess) return DF2_ERR_CUDA;
    }
    return from_cuda(df2::draft_tail_launch(parts, P, K, topk_ids, topk_vals, anchors, B, G, A, Bc, V,
                                            r, path, path_scores, pred, pair_scores, dev_status, st, lm,
                                            df2::Refine{h, W_lm, D}));
}

// -------------------------------------------------------------- selector --

namespace {

int check_selector(int64_t V, int K, int r) {
    if (V < 1 || K < 1 || r < 1) return DF2_ERR_INVALID_ARGUMENT;
    if (K > DF2_MAX_TOPK || r > DF2_MAX_RANK || r % 8 != 0 || V > DF2_MAX_VOCAB) return DF2_ERR_UNSUPPORTED;
    return DF2_OK;
}

}  // namespace

DF2_API int dflash2_selector_walk(const int32_t* anchors, int R, int B, const int32_t* topk_ids,
                                  const float* topk_vals, const float* G, const uint16_t* A,
                                  const uint16_t* Bc, int64_t V, int K, int r, int32_t* path,
                                  float* path_scores, int32_t* dev_status, void* stream) {
    if (R < 0 || B < 2 || K > V) return DF2_ERR_INVALID_ARGUMENT;
    int rc = check_selector(V, K, r);
    if (rc != DF2_OK) return rc;
    if (R == 0) return DF2_OK;
    if (!anchors || !topk_ids || !topk_vals || !G || !A || !Bc || !path || !path_scores)
        return DF2_ERR_INVALID_ARGUMENT;
    if (!aligned16(G) || !aligned16(A) || !aligned16(Bc)) return DF2_ERR_UNSUPPORTED;
    return from_cuda(df2::walk_launch(anchors, R, B, topk_ids, topk_vals, G, A, Bc, V, K, r, path,
                                      path_scores, dev_status, static_cast<cudaStream_t>(stream)));
}

DF2_API int dflash2_selector_pair_scores(const int32_t* pred, int64_t P, const int32_t* topk_ids,
                                         const float* topk_vals, const float* G, const uint16_t* A,
                                         const uint16_t* Bc, int64_t V, int K, int r, float* scores,
                                         int32_t* dev_status, void* stream) {
    if (P < 0) return DF2_ERR_INVALID_ARGUMENT;
    int rc = check_selector(V, K, r);
    if (rc != DF2_OK) return rc;
    if (P == 0) return DF2_OK;
    if (!pred || !topk_ids || !topk_vals || !G || !A || !Bc || !scores)
        return DF2_ERR_INVALID_ARGUMENT;
    if (!aligned16(G) || !aligned16(A) || !aligned16(Bc)) return DF2_ERR_UNSUPPORTED;
    if (P * ((K + 7) / 8) / 8 + 1 > INT32_MAX) return DF2_ERR_UNSUPPORTED;
    return from_cuda(df2::pair_scores_launch(pred, P, topk_ids, topk_vals, G, A, Bc, V, K, r,
                                             scores, dev_status,
                                             static_cast<cudaStream_t>(stream)));
}

DF2_API int dflash2_selector_ce(const float* scores, const int32_t* topk_ids, const int32_t* targets,
                                int64_t P, int K, int64_t V, float* loss, int32_t* label_idx,
                                int32_t* dev_status, void* stream) {
    if (P < 0 || K < 1 || V < 1) return DF2_ERR_INVALID_ARGUMENT;
    if (K > DF2_MAX_TOPK || V > DF2_MAX_VOCAB) return DF2_ERR_UNSUPPORTED;
    if (P == 0) return DF2_OK;
    if (!scores || !topk_ids || !targets || !loss) return DF2_ERR_INVALID_ARGUMENT;
    if ((P + 7) / 8 > INT32_MAX) return DF2_ERR_UNSUPPORTED;
    return from_cuda(df2::selector_ce_launch(scores, topk_ids, targets, P, K, V, loss, label_idx, dev_status,
                                             static_cast<cudaStream_t>(stream)));
}

// --------------------------------------------------------------- lattice --

DF2_API int dflash2_selector_lattice(const int32_t* anchors, int R, int B, const int32_t* topk_ids,
                                     const float* topk_vals, const float* G, const uint16_t* A,
                                     const uint16_t* Bc, int64_t V, int K, int r, float* lattice,
                                     int32_t* dev_status, void* stream) {
    if (R < 0 || B < 2 || K > V) return DF2_ERR_INVALID_ARGUMENT;
    int rc = check_selector(V, K, r);
    if (rc != DF2_OK) return rc;
    if (R == 0) return DF2_OK;
    if (!anchors || !topk_ids || !topk_vals || !G || !A || !Bc || !lattice)
        return DF2_ERR_INVALID_ARGUMENT;
    if (!aligned16(G) || !aligned16(A) || !aligned16(Bc)) return DF2_ERR_UNSUPPORTED;
    const int64_t tile = K <= 16 ? 16 : (K <= 32 ? 32 : 64);
    const int64_t tiles = (K + tile - 1) / tile;
    if (int64_t(R) * (B - 1) * tiles * tiles > INT32_MAX) return DF2_ERR_UNSUPPORTED;
    return from_cuda(df2::lattice_launch(anchors, R, B, topk_ids, topk_vals, G, A, Bc, V, K, r, lattice,
                                         dev_status, static_cast<cudaStream_t>(stream)));
}

DF2_API int dflash2_lattice_walk(const float* lattice, const int32_t* topk_ids, int R, int B, int K,
                                 int64_t V, const float* uniforms, float temperature, int32_t* path,
                                 float* path_scores, int32_t* dev_status, void* stream) {
    if (R < 0 || B < 2 || K < 1 || V < 1 || K > V) return DF2_ERR_INVALID_ARGUMENT;
    if (K > DF2_MAX_TOPK || V > DF2_MAX_VOCAB) return DF2_ERR_UNSUPPORTED;
    if (uniforms && !(temperature > 0.f && temperature <= FLT_MAX)) return DF2_ERR_INVALID_ARGUMENT;
    if (R == 0) return DF2_OK;
    if (!lattice || !topk_ids || !path || !path_scores) return DF2_ERR_INVALID_ARGUMENT;
    return from_cuda(df2::lattice_walk_launch(lattice, topk_ids, R, B, K, V, uniforms, temperature, path,
                                              path_scores, dev_status,
                                              static_cast<cudaStream_t>(stream)));
}

// ------------------------------------------------------------------ conv --

namespace {

int check_conv(int dtype, int64_t P, int C, int B, int taps, int g) {
    if (dtype != DF2_DTYPE_BF16 && dtype != DF2_DTYPE_F32) return DF2_ERR_INVALID_ARGUMENT;
    if (P < 0 || C < 1 || B < 1 || g < 1 || taps < 1 || taps > B) return DF2_ERR_INVALID_ARGUMENT;
    if (C % g != 0 || P % B != 0) return DF2_ERR_INVALID_ARGUMENT;
    if (C % 8 != 0) return DF2_ERR_UNSUPPORTED;
    if ((P + 63) / 64 > 65535) return DF2_ERR_UNSUPPORTED;
    return DF2_OK;
}

}  // namespace

DF2_API size_t dflash2_conv_prepare_workspace_size(int64_t P, int C, int taps, int g, int dtype) {
    if (P <= 0 || C < 1 || g < 1 || taps < 1 || C % g != 0) return 0;
    (void)dtype;
    return round_up(size_t(P) * taps * (C / g) * sizeof(float), 256);
}

DF2_API int dflash2_conv_prepare(const void* x, int dtype, int64_t P, int C, int B, int taps, int g,
                                 const uint16_t* W_proj, const float* base, void* y, float* dyn_out,
                                 void* workspace, size_t workspace_bytes, void* stream) {
    int rc = check_conv(dtype, P, C, B, taps, g);
    if (rc != DF2_OK) return rc;
    if (P == 0) return DF2_OK;
    if (!x || !W_proj || !base || !y || !dyn_out || x == y) return DF2_ERR_INVALID_ARGUMENT;
    if (!aligned16(x) || !aligned16(y) || !aligned16(base) || !aligned16(W_proj) ||
        !aligned16(dyn_out) || !aligned16(workspace))
        return DF2_ERR_UNSUPPORTED;
    const size_t need = dflash2_conv_prepare_workspace_size(P, C, taps, g, dtype);
    if (workspace_bytes < need || !workspace) return DF2_ERR_WORKSPACE_TOO_SMALL;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int G = C / g;
    const int64_t half = int64_t(taps) * G;
    float* d_in = static_cast<float*>(workspace);
    cudaError_t e;
    if (df2::conv_prepare_rows_supported(P, C, B, dtype == DF2_DTYPE_F32))
        return from_cuda(df2::conv_prepare_rows_launch(x, dtype == DF2_DTYPE_F32, P, C, B, taps, g, W_proj,
                                                       base, y, dyn_out, st));
    if (dtype == DF2_DTYPE_BF16 && P > 64 && df2::conv_prepare_tc_supported(P, C, B, taps, g))
        return from_cuda(df2::conv_prepare_tc_launch(static_cast<const uint16_t*>(x), P, C, B, taps, g, W_proj,
                                                     base, static_cast<uint16_t*>(y), dyn_out, nullptr, st));
    if (P <= 64) {
        const int sms = num_sms_current();
        if (sms <= 0) return DF2_ERR_CUDA;
        e = df2::gemm_rows_launch(x, dtype == DF2_DTYPE_F32, W_proj, P, 2 * half, C, d_in, half, half,
                                  dyn_out, half, sms, st);
    } else if (dtype == DF2_DTYPE_BF16 && df2::wide_supported(P, 2 * half, C, 1)) {
        e = df2::wide_store_launch(static_cast<const uint16_t*>(x), P, W_proj, 2 * half, C, d_in, half,
                                   half, dyn_out, half, nullptr, st);
    } else {
        e = df2::gemm_simple_launch(x, dtype == DF2_DTYPE_F32, W_proj, P, 2 * half, C, d_in, half,
                                    half, dyn_out, half, st);
    }
    if (e != cudaSuccess) return DF2_ERR_CUDA;
    e = df2::conv_apply_launch(x, dtype == DF2_DTYPE_F32, P, C, B, taps, g, base, d_in, half, y, st);
    return from_cuda(e);
}

DF2_API int dflash2_conv_finish(const void* z, int dtype, int64_t P, int C, int B, int taps, int g,
                                const float* dyn_out, const float* base, void* y, void* stream) {
    int rc = check_conv(dtype, P, C, B, taps, g);
    if (rc != DF2_OK) return rc;
    if (P == 0) return DF2_OK;
    if (!z || !dyn_out || !base || !y || z == y) return DF2_ERR_INVALID_ARGUMENT;
    if (!aligned16(z) || !aligned16(y) || !aligned16(base) || !aligned16(dyn_out))
        return DF2_ERR_UNSUPPORTED;
    const int G = C / g;
    return from_cuda(df2::conv_apply_launch(z, dtype == DF2_DTYPE_F32, P, C, B, taps, g,
                                            base + int64_t(taps) * C, dyn_out, int64_t(taps) * G, y,
                                            static_cast<cudaStream_t>(stream)));
}

DF2_API size_t dflash2_conv_finish_prepare_workspace_size(int64_t P, int C, int taps, int g, int dtype) {
    return dflash2_conv_prepare_workspace_size(P, C, taps, g, dtype);
}

DF2_API int dflash2_conv_finish_prepare(const void* z, int dtype, int64_t P, int C, int B, int taps, int g,
                                        const float* dyn_out, const float* base, const void* residual, void* h,
                                        const uint16_t* W_proj, const float* base_next, void* y_next,
                                        float* dyn_out_next, void* workspace, size_t workspace_bytes,
                                        void* stream) {
    int rc = check_conv(dtype, P, C, B, taps, g);
    if (rc != DF2_OK) return rc;
    if (P == 0) return DF2_OK;
    if (!z || !dyn_out || !base || !h || !W_proj || !base_next || !y_next || !dyn_out_next)
        return DF2_ERR_INVALID_ARGUMENT;
    // an output aliasing an input would be read and written by different threads
    if (h == z || h == residual || y_next == z || y_next == residual || y_next == h ||
        dyn_out_next == dyn_out)
        return DF2_ERR_INVALID_ARGUMENT;
    if (!aligned16(z) || !aligned16(dyn_out) || !aligned16(base) || !aligned16(residual) || !aligned16(h) ||
        !aligned16(W_proj) || !aligned16(base_next) || !aligned16(y_next) || !aligned16(dyn_out_next) ||
        !aligned16(workspace))
        return DF2_ERR_UNSUPPORTED;
    const size_t need = dflash2_conv_finish_prepare_workspace_size(P, C, taps, g, dtype);
    if (workspace_bytes < need || !workspace) return DF2_ERR_WORKSPACE_TOO_SMALL;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const bool f32 = dtype == DF2_DTYPE_F32;
    const int64_t half = int64_t(taps) * (C / g);
    // the finish with the residual add in its store writes h, then the next prepare
    // reads it (a kernel that recomputed h per CTA instead ran 2.7x longer at P = 8)
    cudaError_t e = df2::conv_apply_launch(z, f32, P, C, B, taps, g, base + int64_t(taps) * C, dyn_out, half, h,
                                           st, residual);
    if (e != cudaSuccess) return DF2_ERR_CUDA;
    return dflash2_conv_prepare(h, dtype, P, C, B, taps, g, W_proj, base_next, y_next, dyn_out_next, workspace,
                                workspace_bytes, stream);
}

// ---------------------------------------------------------------- self-test --

DF2_API int dflash2_selftest_wait_timeout(const uint16_t* h, int64_t P, int64_t D, const uint16_t* W_lm,
                                          int64_t V, int K, int32_t* topk_ids, float* topk_vals,
                                          void* workspace, size_t workspace_bytes, int32_t* dev_status,
                                          void* stream) {
    int rc = check_head(P, D, V, K, 0, false);
    if (rc != DF2_OK) return rc;
    if (P == 0 || !df2::head_tc_supported(P, D, V, K) || !dev_status) return DF2_ERR_UNSUPPORTED;
    if (!h || !W_lm || !topk_ids || !topk_vals) return DF2_ERR_INVALID_ARGUMENT;
    const int sms = num_sms_current();
    if (sms <= 0) return DF2_ERR_CUDA;
    const size_t need = round_up(df2::head_tc_workspace(P, D, V, K, sms), 256);
    if (workspace_bytes < need || !workspace) return DF2_ERR_WORKSPACE_TOO_SMALL;
    return df2::head_tc_launch(h, P, D, W_lm, V, K, nullptr, 0, nullptr, topk_ids, topk_vals, workspace,
                               dev_status, sms, static_cast<cudaStream_t>(stream), /*stall_stage=*/0);
}
