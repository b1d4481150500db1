/*
 * libdflash2 — the DFlash2 draft-block head on one GB300 (sm_103a).
 *
 * Five calls cover the data-parallel part of one DFlash2 draft cycle:
 *
 *   dflash2_unary_topk            unary logits over the full verifier vocabulary,
 *                                 the per-position top-K, and the hidden projection H
 *   dflash2_selector_walk         the candidate selector's greedy walk
 *   dflash2_selector_pair_scores  the selector scores with teacher-forced predecessors
 *   dflash2_selector_ce           the selector's K-way cross-entropy on those scores
 *   dflash2_draft_head            the four steps above for one draft block, fused
 *   dflash2_selector_lattice      every adjacent candidate pair scored at once
 *   dflash2_lattice_walk          the greedy or sampling walk over that table
 *   dflash2_conv_prepare          the grouped dynamic causal conv before a sublayer
 *   dflash2_conv_finish           the same conv after the sublayer
 *   dflash2_conv_finish_prepare   a finish and the next sublayer's prepare in one call
 *
 * Sources (web pages, cited by title and section):
 *   [vLLM]  "DFlash2", vLLM Speculators user guide: "Local Convolution",
 *           "Candidate Selector", "Key Parameters".
 *   [SF]    "DFlash2", SpecForge concept doc: "Architecture" and the dflash_config
 *           validity rules under it.
 *   [PR62]  verl-SpeCo PR #62 "feat: add DFlash2 drafter training backend":
 *           "What DFlash2 adds" (conv and selector equations), "Two deltas over the
 *           upstream inference implementation", "Selector training objective".
 *   [KB]    "DFlash 2 Explanation": "Component Breakdown", "Draft-Verify Cycle",
 *           "Problem 1" (pair score; all pairs scored in one pass, then a greedy or
 *           sampling walk over the scores), "Problem 2" (two-tap conv).
 *
 * Conventions shared by every call
 * ---------------------------------
 * - Every pointer argument except the documented host ones is a DEVICE pointer
 *   on the current CUDA device.  Tensors are dense and row-major with the shapes
 *   given; the caller owns every buffer, the library allocates nothing per call.
 * - bf16 tensors are passed as uint16_t: raw IEEE bfloat16 bit patterns.
 * - Every call is asynchronous on `stream` (a cudaStream_t; NULL = the legacy
 *   default stream) and does not synchronise the host.  Host-side validation
 *   happens before any launch; on any non-zero return nothing was launched
 *   (DF2_ERR_CUDA: a launch was attempted and failed).
 * - Workspace: calls that need scratch take (workspace, workspace_bytes), a device
 *   buffer the caller allocates; the matching *_workspace_size() query returns the
 *   bytes needed for those shapes on the current device (0 = none).  The
 *   workspace must be 256-byte aligned and must not be used concurrently by
 *   another call.  Its contents on entry do not matter.
 * - dev_status (nullable): a device int32 that kernels OR DF2_STATUS_* bits into.
 *   The library never clears it; the caller zeroes it when it wants a fresh read.
 * - Inputs must be finite; NaN/Inf inputs give unspecified ids.
 * - Alignment: every tensor pointer must be 16-byte aligned.
 */
#ifndef DFLASH2_H
#define DFLASH2_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Return codes. */
#define DF2_OK 0
#define DF2_ERR_INVALID_ARGUMENT 1   /* a shape or value rule below is broken */
#define DF2_ERR_UNSUPPORTED 2        /* valid for the method but outside this build's limits */
#define DF2_ERR_CUDA 3               /* a CUDA runtime call failed (launch, attribute, ...) */
#define DF2_ERR_WORKSPACE_TOO_SMALL 4
#define DF2_ERR_TIMEOUT 5            /* reserved: a bounded device wait gave up */

/* Activation dtypes for the conv calls. */
#define DF2_DTYPE_BF16 0
#define DF2_DTYPE_F32 1

/* Bits OR-ed into *dev_status by the kernels. */
#define DF2_STATUS_ID_OUT_OF_RANGE 0x1  /* a token id outside [0, V) was read */
#define DF2_STATUS_WAIT_TIMEOUT 0x2     /* a bounded in-kernel wait gave up; outputs invalid */

/* Limits of this build (DF2_ERR_UNSUPPORTED beyond them).  DF2_MAX_VOCAB bounds V
 * (token ids, rows of W_lm, A and Bc) so that a row index plus a tile's rows stays
 * inside int32 in every kernel. */
#define DF2_MAX_TOPK 1024
#define DF2_MAX_RANK 4096
#define DF2_MAX_VOCAB (1 << 30)

/* Name of a return code ("DF2_OK", ...); never NULL. */
const char* dflash2_status_string(int status);

/* ABI version of this library (bumped on any signature change). */
int dflash2_abi_version(void);

/* Diagnostics: how many CUDA kernels this library has launched in this process
 * so far (every device and call; a launch that failed is counted too).  Read it
 * before and after a region to count the region's kernels. */
long long dflash2_kernels_launched(void);

/* Diagnostics: which kernel path dflash2_unary_topk (and the head of
 * dflash2_draft_head) takes for these shapes on the current device.  No
 * counterpart in the pages.  Returns DF2_HEAD_PATH_* (>= 0), or -1 when the shapes
 * break a rule of dflash2_unary_topk. */
#define DF2_HEAD_PATH_STREAM 0     /* few positions: the HBM-streaming tensor-core head */
#define DF2_HEAD_PATH_GEMM 1       /* many positions: the tensor-core GEMM with a top-K epilogue */
#define DF2_HEAD_PATH_CUDA_CORE 2  /* K > 64 or shapes the tensor-core kernels do not take */
int dflash2_unary_topk_path(int64_t P, int64_t D, int64_t V, int K);

/* ------------------------------------------------------------------------
 * dflash2_unary_topk — unary logits, per-position top-K, hidden projection.
 *
 * For every row p of the draft hidden state (P = requests x block_size rows;
 * row 0 of each block is the anchor position):
 *   U[p, v] = sum_d h[p, d] * W_lm[v, d]        for all v in [0, V)   ([vLLM]
 *             "Candidate Selector": the drafter's per-token logits; [KB] "Draft-Verify
 *             Cycle": the shared lm_head gives logits and top-K per position;
 *             the full verifier vocabulary, [vLLM] "Candidate Selector")
 *   U'[p, v] = c * tanh(m * U[p, v] / c)          (m * U[p, v] when c = 0)
 *             the optional output multiplier m and final logit softcap c of the
 *             unary logits ([SF] "Export and serve": both act on the unary
 *             logits; no formula is given there, this is the common form with
 *             the cap applied last).  m = 1, c = 0 leaves U as it is, bit for bit.
 *   topk_ids[p, :], topk_vals[p, :] = the K largest U'[p, .], ordered by value
 *             descending, equal values by token id ascending.  U' is increasing
 *             in U, so the selection runs on U and only the K kept values are
 *             mapped (fp32, tanhf); where fp32 rounding merges two mapped values
 *             their order is U's, which can differ from the id rule
 *   G[p, i]  = sum_d h[p, d] * W_H[i, d]         the hidden projection H(h_t) of
 *             the pair score ([PR62] "What DFlash2 adds"; [KB] "Problem 1"), read
 *             as linear with no bias
 * U never leaves the chip; products are of the bf16 inputs, sums in fp32.
 *
 *   h         [P, D]  bf16        draft hidden state
 *   W_lm      [V, D]  bf16        LM head (the verifier's, shared)
 *   K                              selector_top_k, 1 <= K <= min(V, DF2_MAX_TOPK)
 *   output_multiplier              m: finite and > 0 (1 = none)
 *   final_logit_softcapping        c: finite and >= 0 (0 = none)
 *   W_H       [r, D]  bf16        hidden projection, or NULL (then G is not written
 *                                  and r is ignored)
 *   G         [P, r]  fp32        out (when W_H != NULL); 1 <= r <= DF2_MAX_RANK
 *   topk_ids  [P, K]  int32       out
 *   topk_vals [P, K]  fp32        out
 *   workspace                      >= dflash2_unary_topk_workspace_size(P, D, V, K, r)
 * Rules: P >= 0 (P = 0 launches nothing), D >= 1, D % 8 == 0, 1 <= V <= DF2_MAX_VOCAB.
 * ---------------------------------------------------------------------- */
size_t dflash2_unary_topk_workspace_size(int64_t P, int64_t D, int64_t V, int K, int r);
int dflash2_unary_topk(const uint16_t* h, int64_t P, int64_t D, const uint16_t* W_lm, int64_t V,
                       int K, float output_multiplier, float final_logit_softcapping,
                       const uint16_t* W_H, int r, float* G, int32_t* topk_ids,
                       float* topk_vals, void* workspace, size_t workspace_bytes,
                       int32_t* dev_status, void* stream);

/* ------------------------------------------------------------------------
 * dflash2_unary_topk_noalloc — dflash2_unary_topk without a caller workspace.
 *
 * No counterpart in the pages: this is a convenience of the library.  It is for
 * callers that cannot allocate device memory at call time, such as code running
 * inside a host framework that owns all device allocations and forbids new ones
 * during a step, or a latency-critical path where a cudaMalloc (which may
 * synchronise the device) is not acceptable.  Same arguments, results and rules
 * as dflash2_unary_topk, minus (workspace, workspace_bytes).
 *
 * Scratch: a DF2_NOALLOC_SCRATCH_BYTES array inside the library, one per GPU,
 * held by every GPU that loads the library until the process exits.  Shapes
 * whose dflash2_unary_topk_workspace_size() exceeds it return
 * DF2_ERR_UNSUPPORTED (use dflash2_unary_topk with your own workspace then).
 * Allocates nothing: no cudaMalloc / cudaFree or allocating library call.
 * The first call on a device looks up that device's copy of the array
 * (cudaGetSymbolAddress, with the device current); make that first call before
 * any stream capture.  The address is kept for the life of the process: after a
 * cudaDeviceReset of that device it is stale, so do not use this entry point on
 * a device that has been reset.  `stream` must belong to the current device
 * (DF2_ERR_INVALID_ARGUMENT otherwise).  All calls share the one array: calls
 * that may overlap on the GPU (different streams, no ordering between them) race
 * and give wrong results.  The array keeps the last call's contents; none of it
 * needs to start at zero.
 * ---------------------------------------------------------------------- */
#define DF2_NOALLOC_SCRATCH_BYTES ((size_t)8 << 20)
int dflash2_unary_topk_noalloc(const uint16_t* h, int64_t P, int64_t D, const uint16_t* W_lm,
                               int64_t V, int K, float output_multiplier,
                               float final_logit_softcapping, const uint16_t* W_H, int r, float* G,
                               int32_t* topk_ids, float* topk_vals, int32_t* dev_status,
                               void* stream);

/* ------------------------------------------------------------------------
 * dflash2_selector_walk — the candidate selector's greedy walk.
 *
 * Per request q (R requests, blocks of B rows, T = B - 1 drafted positions):
 *   a_0 = anchors[q]                            (the last verified token)
 *   for t = 1 .. B-1, row = q*B + t:
 *     s_j = topk_vals[row, j] + sum_i A[a_{t-1}, i] * G[row, i] * Bc[topk_ids[row, j], i]
 *     j*  = argmax_j s_j   (equal scores: the lower token id)
 *     a_t = topk_ids[row, j*];  path[q, t-1] = a_t;  path_scores[q, t-1] = s_{j*}
 * ([vLLM] "Candidate Selector": the walk begins at the anchor and each choice
 * becomes the next position's predecessor; [PR62] "What DFlash2 adds": S_t(a, b) =
 * U_t(b) + <A(a) * H(h_t), B(b)>; [KB] "Problem 1": the greedy walk takes the
 * highest-scoring successor.)  Rows t = 0 (the anchor rows) are not read.  Scores are fp32.
 *
 *   anchors     [R]        int32   device
 *   topk_ids    [R*B, K]   int32   candidates (as written by dflash2_unary_topk)
 *   topk_vals   [R*B, K]   fp32    their unary logits
 *   G           [R*B, r]   fp32    H(h_t)
 *   A, Bc       [V, r]     bf16    predecessor / successor codebooks
 *   path        [R, B-1]   int32   out
 *   path_scores [R, B-1]   fp32    out
 * Rules: R >= 0, B >= 2, 1 <= K <= min(V, DF2_MAX_TOPK), 1 <= r <= DF2_MAX_RANK,
 * V <= DF2_MAX_VOCAB.
 * An anchor or candidate id outside [0, V) sets DF2_STATUS_ID_OUT_OF_RANGE and
 * writes -1 / NaN over that request's whole path.
 * ---------------------------------------------------------------------- */
int dflash2_selector_walk(const int32_t* anchors, int R, int B, const int32_t* topk_ids,
                          const float* topk_vals, const float* G, const uint16_t* A,
                          const uint16_t* Bc, int64_t V, int K, int r, int32_t* path,
                          float* path_scores, int32_t* dev_status, void* stream);

/* ------------------------------------------------------------------------
 * dflash2_selector_pair_scores — teacher-forced selector scores.
 *
 *   scores[p, j] = topk_vals[p, j] + sum_i A[pred[p], i] * G[p, i] * Bc[topk_ids[p, j], i]
 * for all P rows at once: the predecessor is given (the previous ground-truth
 * token) instead of walked ([PR62] "Selector training objective").  Replaying a
 * walk's own predecessors through this call reproduces the walk.
 *
 *   pred [P] int32; topk_ids/topk_vals [P, K]; G [P, r]; A, Bc [V, r] bf16;
 *   scores [P, K] fp32 out.
 * Rules: P >= 0, 1 <= K <= DF2_MAX_TOPK, 1 <= r <= DF2_MAX_RANK, 1 <= V <= DF2_MAX_VOCAB.
 * A pred or candidate id outside [0, V) sets DF2_STATUS_ID_OUT_OF_RANGE and
 * writes NaN for the affected scores.
 * ---------------------------------------------------------------------- */
int dflash2_selector_pair_scores(const int32_t* pred, int64_t P, const int32_t* topk_ids,
                                 const float* topk_vals, const float* G, const uint16_t* A,
                                 const uint16_t* Bc, int64_t V, int K, int r, float* scores,
                                 int32_t* dev_status, void* stream);

/* ------------------------------------------------------------------------
 * dflash2_selector_ce — the selector's training loss, forward.
 *
 * The K-way cross-entropy of the teacher-forced scores against the ground truth
 * ([PR62] "Selector training objective"; [vLLM] "Training Objective"): a
 * categorical loss over the K candidates the head kept, to which a row contributes
 * only when its ground-truth token is one of them.  For row p:
 *
 *   label_idx[p] = the column j with topk_ids[p, j] == targets[p], else -1
 *   loss[p]      = log(sum_j exp(scores[p, j])) - scores[p, label_idx[p]]
 *                  (NaN where label_idx[p] == -1: the row contributes nothing)
 *
 * The variant that swaps the target into the weakest candidate's slot when it is
 * missing ([vLLM] "Training Objective") is the same call on the edited candidate
 * list and scores.  Forward only; fp32 with the row maximum subtracted before exp.
 *
 *   scores [P, K] fp32 (dflash2_selector_pair_scores' output); topk_ids [P, K]
 *   int32; targets [P] int32 (the ground-truth token of each row, < 0: none);
 *   loss [P] fp32 out; label_idx [P] int32 out (nullable).
 * Rules: P >= 0, 1 <= K <= DF2_MAX_TOPK, 1 <= V <= DF2_MAX_VOCAB.  A target >= V sets
 * DF2_STATUS_ID_OUT_OF_RANGE (label -1, loss NaN).
 * ---------------------------------------------------------------------- */
int dflash2_selector_ce(const float* scores, const int32_t* topk_ids, const int32_t* targets, int64_t P,
                        int K, int64_t V, float* loss, int32_t* label_idx, int32_t* dev_status,
                        void* stream);

/* ------------------------------------------------------------------------
 * dflash2_draft_head — unary top-K, H, greedy walk and teacher-forced scores of one
 * draft block in one call.
 *
 * The same results as dflash2_unary_topk (with W_H), then dflash2_selector_walk,
 * then (pred != NULL) dflash2_selector_pair_scores, on P = R*B rows: the same
 * kernels' arithmetic in the same order, so every output is bit-identical to the
 * three calls'.  Where the shapes allow (K <= 32 on a tensor-core head, B <= 16,
 * a lattice slot's rows within shared memory) the fold of the head's partial
 * lists, the walk and the teacher-forced scores run in one launch after the head
 * kernel, one thread-block cluster per request, with the walk taken over the
 * lattice of adjacent pair scores ([KB] "How It Works", Problem 1); otherwise the
 * three calls run in sequence.  The pages describe the steps, not this fusion;
 * the call exists to cut the launches and the serial latency of a draft step.
 *
 *   h [R*B, D] bf16; W_lm [V, D] bf16; output_multiplier, final_logit_softcapping as
 *   for dflash2_unary_topk; W_H [r, D] bf16 (required); A, Bc [V, r] bf16;
 *   anchors [R] int32; pred [R*B] int32 (nullable);
 *   topk_ids, topk_vals [R*B, K] out; G [R*B, r] fp32 out; path, path_scores [R, B-1]
 *   out; pair_scores [R*B, K] fp32 out (required iff pred != NULL).
 *   workspace: dflash2_draft_head_workspace_size(R, B, D, V, K, r) bytes, 256-byte
 *   aligned (it holds the head's partial lists).
 * Rules: the union of the three calls' rules; B >= 2.  Status bits as those calls;
 * in the fused launch each CTA of a cluster waits (bounded, about one second) for
 * the predecessor rows the previous CTA sends it, and a wait that gives up ORs
 * DF2_STATUS_WAIT_TIMEOUT and fails that request's path like a bad id (-1 / NaN).
 * ---------------------------------------------------------------------- */
size_t dflash2_draft_head_workspace_size(int R, int B, int64_t D, int64_t V, int K, int r);
int dflash2_draft_head(const uint16_t* h, int R, int B, int64_t D, const uint16_t* W_lm, int64_t V,
                       int K, float output_multiplier, float final_logit_softcapping,
                       const uint16_t* W_H, int r, const uint16_t* A, const uint16_t* Bc,
                       const int32_t* anchors, const int32_t* pred, int32_t* topk_ids,
                       float* topk_vals, float* G, int32_t* path, float* path_scores,
                       float* pair_scores, void* workspace, size_t workspace_bytes,
                       int32_t* dev_status, void* stream);

/* ------------------------------------------------------------------------
 * dflash2_selector_lattice — every adjacent candidate pair scored at once.
 *
 * [KB] "How It Works", Problem 1: all pairs of adjacent candidates are scored in
 * one parallel pass, and only the final walk over those scores is sequential.
 * For request q and drafted position t = 1 .. B-1 (table slot t-1), row = q*B + t:
 *   lattice[q, t-1, i, j] = topk_vals[row, j]
 *                         + sum_k A[a_i, k] * G[row, k] * Bc[topk_ids[row, j], k]
 * where a_i = topk_ids[row - 1, i] (the i-th candidate of position t-1) for t >= 2,
 * and for t = 1 the predecessor is the anchor alone: row i = 0 of slot 0 holds
 * S_1(anchors[q], .) and rows 1 .. K-1 of slot 0 are NaN.
 *
 *   anchors     [R]               int32   device
 *   topk_ids    [R*B, K]          int32   candidates (as written by dflash2_unary_topk)
 *   topk_vals   [R*B, K]          fp32    their unary logits
 *   G           [R*B, r]          fp32    H(h_t)
 *   A, Bc       [V, r]            bf16    predecessor / successor codebooks
 *   lattice     [R, B-1, K, K]    fp32    out (caller-allocated, fully written)
 * Rules: as dflash2_selector_walk; G, A, Bc 16-byte aligned; r % 8 == 0;
 * R * (B-1) * ceil(K/64)^2 (K > 32), ceil(K/32)^2 (16 < K <= 32) or 1 (K <= 16)
 * below 2^31 (else DF2_ERR_UNSUPPORTED).  An anchor or candidate id outside
 * [0, V) sets DF2_STATUS_ID_OUT_OF_RANGE and writes NaN over that request's table.
 * Scores are fp32 sums of exact bf16 x fp32 products, summed in a different order
 * than dflash2_selector_walk's, so the two agree to fp32 rounding.
 * ---------------------------------------------------------------------- */
int dflash2_selector_lattice(const int32_t* anchors, int R, int B, const int32_t* topk_ids,
                             const float* topk_vals, const float* G, const uint16_t* A,
                             const uint16_t* Bc, int64_t V, int K, int r, float* lattice,
                             int32_t* dev_status, void* stream);

/* ------------------------------------------------------------------------
 * dflash2_lattice_walk — the walk over a finished lattice.
 *
 * [KB] "How It Works", Problem 1: the greedy walk takes the highest-scoring
 * successor, and the sampled walk draws one from the same pair scores.  Per request q the state is the row i of the
 * current predecessor (i = 0, the anchor, at t = 1); step t reads row i of slot
 * t-1 and picks a column j, which becomes the next row:
 *   uniforms == NULL (greedy): the largest score, equal scores to the lower token id
 *     (the same path as dflash2_selector_walk up to fp32 rounding of the scores);
 *   uniforms != NULL (sampling): a draw from softmax(lattice[q, t-1, i, :] / temperature)
 *     by the inverse CDF in candidate-list order with u = uniforms[q, t-1]: the
 *     smallest j whose running sum w_0 + .. + w_j exceeds u * sum(w), with
 *     w_j = exp((S_j - max S) / temperature); if rounding leaves no such j, the
 *     last j with w_j > 0.  The pages name neither the scheme nor the
 *     temperature: the caller supplies both, and the uniforms, so the draw is
 *     reproducible.
 *   path[q, t-1] = topk_ids[q*B + t, j];  path_scores[q, t-1] = lattice[q, t-1, i, j].
 *
 *   lattice     [R, B-1, K, K]  fp32   (as written by dflash2_selector_lattice)
 *   topk_ids    [R*B, K]        int32  rows t = 0 are not read
 *   uniforms    [R, B-1]        fp32   in [0, 1), nullable
 *   temperature                 host float, > 0 and finite when uniforms is given
 *   path        [R, B-1]        int32  out
 *   path_scores [R, B-1]        fp32   out
 * Rules: R >= 0, B >= 2, 1 <= K <= min(V, DF2_MAX_TOPK), V <= DF2_MAX_VOCAB.  A
 * candidate id outside [0, V) sets DF2_STATUS_ID_OUT_OF_RANGE and writes -1 / NaN
 * over that request's path.  The sampling draw computes its weights and running sums in fp32, so a u
 * that lies within rounding of an interval end may pick the neighbouring column.
 * ---------------------------------------------------------------------- */
int dflash2_lattice_walk(const float* lattice, const int32_t* topk_ids, int R, int B, int K,
                         int64_t V, const float* uniforms, float temperature, int32_t* path,
                         float* path_scores, int32_t* dev_status, void* stream);

/* ------------------------------------------------------------------------
 * dflash2_conv_prepare — grouped dynamic causal conv before a sublayer.
 *
 * Rows are packed anchor blocks: row p has in-block position t = p mod B, and no
 * tap reads across a block boundary ([PR62] "Two deltas", item 1; [vLLM] "Local
 * Convolution").  With G = C / g groups of g contiguous channels:
 *   d[p, io, j, gi] = sum_c W_proj[(io*taps + j)*G + gi, c] * x[p, c]
 *   y[p, c]         = sum_{j < taps, t-j >= 0} (base[0, j, c] + d[p, 0, j, c/g]) * x[p-j, c]
 *   dyn_out[p, j, gi] = d[p, 1, j, gi]
 * ([PR62] "What DFlash2 adds": Conv_k(x)_t = k_{t,0} * x_t + k_{t,1} * x_{t-1}, where
 * each k is a fixed kernel per channel with a correction common to a group of
 * conv_group_size channels added, and prepare hands finish the kernel it will use;
 * [vLLM] "Local Convolution": both kernels come from one projection of the hidden
 * state at that position.)  io = 0 is the
 * kernel applied here, io = 1 the one dflash2_conv_finish applies.
 *
 *   x       [P, C]            dtype (DF2_DTYPE_BF16 or DF2_DTYPE_F32)
 *   W_proj  [2*taps*G, C]     bf16
 *   base    [2, taps, C]      fp32
 *   y       [P, C]            dtype, out (must not alias x)
 *   dyn_out [P, taps, G]      fp32, out
 *   workspace                  >= dflash2_conv_prepare_workspace_size(P, C, taps, g, dtype)
 * Rules ([SF] dflash_config rules and [PR62] item 1): P >= 0, P % B == 0,
 * 1 <= taps <= B, g >= 1, C % g == 0, C % 8 == 0.
 * ---------------------------------------------------------------------- */
size_t dflash2_conv_prepare_workspace_size(int64_t P, int C, int taps, int g, int dtype);
int dflash2_conv_prepare(const void* x, int dtype, int64_t P, int C, int B, int taps, int g,
                         const uint16_t* W_proj, const float* base, void* y, float* dyn_out,
                         void* workspace, size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------
 * dflash2_conv_finish — the same conv after the sublayer, with the dynamic
 * kernel correction dflash2_conv_prepare emitted:
 *   y[p, c] = sum_{j < taps, t-j >= 0} (base[1, j, c] + dyn_out[p, j, c/g]) * z[p-j, c]
 *
 *   z [P, C] dtype; dyn_out [P, taps, G] fp32; base [2, taps, C] fp32 (uses base[1]);
 *   y [P, C] dtype out (must not alias z).  Rules as for dflash2_conv_prepare.
 * ---------------------------------------------------------------------- */
int dflash2_conv_finish(const void* z, int dtype, int64_t P, int C, int B, int taps, int g,
                        const float* dyn_out, const float* base, void* y, void* stream);

/* ------------------------------------------------------------------------
 * dflash2_conv_finish_prepare — the two convs between consecutive sublayers.
 *
 * ([vLLM] "Local Convolution": each attention and MLP sublayer has a conv on its
 * input side and one on its output side.)  The finish of one sublayer, then the prepare of the
 * next, with the sum in between written out:
 *   h        = dflash2_conv_finish(z; dyn_out, base)  (+ residual)
 *   y_next, dyn_out_next = dflash2_conv_prepare(h; W_proj, base_next)
 * The pages do not state the residual wiring between the two convs.  Here the
 * caller passes the residual stream (or NULL for none), and the sum is rounded to
 * dtype as a separate elementwise add in dtype would round it.  The results are
 * bit-identical to dflash2_conv_finish, that add, and dflash2_conv_prepare.  The
 * add happens in the finish kernel's store, so h is written once and never re-read
 * for the add; the prepare then reads it.
 *
 *   z, residual (nullable), h        [P, C] dtype; h out
 *   dyn_out [P, taps, G] fp32, base [2, taps, C] fp32   the finishing conv's (uses base[1])
 *   W_proj [2*taps*G, C] bf16, base_next [2, taps, C]    the next conv's
 *   y_next [P, C] dtype out; dyn_out_next [P, taps, G] fp32 out
 *   workspace >= dflash2_conv_finish_prepare_workspace_size(P, C, taps, g, dtype)
 * Rules as for dflash2_conv_prepare; no output may alias an input, and y_next
 * must not alias h (DF2_ERR_INVALID_ARGUMENT).
 * ---------------------------------------------------------------------- */
size_t dflash2_conv_finish_prepare_workspace_size(int64_t P, int C, int taps, int g, int dtype);
int dflash2_conv_finish_prepare(const void* z, int dtype, int64_t P, int C, int B, int taps, int g,
                                const float* dyn_out, const float* base, const void* residual, void* h,
                                const uint16_t* W_proj, const float* base_next, void* y_next,
                                float* dyn_out_next, void* workspace, size_t workspace_bytes,
                                void* stream);

/* ------------------------------------------------------------------------
 * dflash2_selftest_wait_timeout — exercises the in-kernel timeout path.
 *
 * No counterpart in the pages: a diagnostic.  Runs the tensor-core head of
 * dflash2_unary_topk (same arguments, no W_H; shapes must take that path:
 * P <= 32, K <= 64) with the copies of its first pipeline stage never issued.
 * The kernel's bounded waits give up after about one second, every role drains
 * its own work, frees its tensor memory and exits, and DF2_STATUS_WAIT_TIMEOUT is
 * OR-ed into *dev_status (required, not NULL).  The outputs are meaningless; the
 * device and context stay usable.  Returns DF2_ERR_UNSUPPORTED for shapes that
 * do not take the tensor-core head.
 * ---------------------------------------------------------------------- */
int dflash2_selftest_wait_timeout(const uint16_t* h, int64_t P, int64_t D, const uint16_t* W_lm,
                                  int64_t V, int K, int32_t* topk_ids, float* topk_vals,
                                  void* workspace, size_t workspace_bytes, int32_t* dev_status,
                                  void* stream);

#ifdef __cplusplus
}
#endif

#endif /* DFLASH2_H */
