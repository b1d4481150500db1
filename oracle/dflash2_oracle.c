/*
 * DFlash2 draft-block head: the CPU oracle.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or call
 * this file; only the tests, __graft_entry__.smoke() and bench.py's cpu_baseline
 * and reference legs use it.  It shares no code, header, table or helper with the
 * CUDA library.
 *
 * What it computes, and where the pages define it:
 *
 *   unary logits    U_t(v) = h_t . W_lm[v] over the full verifier vocabulary
 *                   (vLLM Speculators "DFlash2" guide, "Candidate Selector";
 *                   "DFlash 2 Explanation", "Draft-Verify Cycle", node HEAD)
 *   top-K           the selector_top_k largest unary logits per position
 *                   (vLLM guide, "Candidate Selector" and "Key Parameters")
 *   pair score      S_t(a,b) = U_t(b) + < A(a) (.) H(h_t), B(b) >
 *                   (verl-SpeCo PR #62, "What DFlash2 adds", selector equation;
 *                   "DFlash 2 Explanation", "Problem 1")
 *   greedy walk     start at the anchor, take the best successor, feed it in as
 *                   the next predecessor (vLLM guide, "Candidate Selector";
 *                   PR #62, "Selector training objective")
 *   teacher-forced  the same score with the predecessor given, all positions at
 *                   once (PR #62, "Selector training objective")
 *   selector loss   the K-way cross-entropy of the teacher-forced scores against
 *                   the ground truth, on rows whose ground truth is a candidate
 *                   (PR #62, "Selector training objective"; vLLM guide,
 *                   "Training Objective")
 *   lattice         every adjacent candidate pair scored at once, then a greedy or
 *                   sampling walk over the finished table ("DFlash 2 Explanation",
 *                   "How It Works", Problem 1)
 *   conv            Conv_k(x)_t = k_{t,0} (.) x_t + k_{t,1} (.) x_{t-1}, k = base +
 *                   a per-group correction projected from the hidden state; the
 *                   projection made before the sublayer also yields the kernel
 *                   applied after it; no tap crosses an anchor-block boundary
 *                   (vLLM guide, "Local Convolution"; PR #62, "What DFlash2 adds"
 *                   and "Two deltas", item 1; "DFlash 2 Explanation", "Problem 2")
 *
 * Readings taken where the pages are silent (each is listed in the design notes):
 *   - H is linear with no bias and no activation; G = H(h) is kept in fp32.
 *   - the codebooks A and B are materialised [V, r] tables gathered by token id.
 *   - top-K ranks by (value descending, token id ascending); the walk's argmax
 *     breaks equal scores toward the lower token id.  Both decisions are taken
 *     on fp32 values, the precision the kernels produce.
 *   - sampling draws from softmax(S / temperature) over the K candidates by the
 *     inverse CDF in candidate-list order, with one uniform per step passed in.
 *   - taps generalise the two-tap form: y_t = sum_{j < taps, t-j >= 0} k_{t,j} x_{t-j},
 *     with t the position inside its anchor block (zero padding inside a block).
 *   - projection row index (io*taps + j)*G + gi, io = 0 for the kernel applied
 *     before the sublayer ("prepare"), io = 1 for the one applied after ("finish");
 *     channel c belongs to group c / g (contiguous groups of g channels).
 *   - base kernel layout [2][taps][C]: one base per side of the sublayer.
 *
 * Arithmetic: every product and sum is taken in double from the exact values of
 * the bf16 / fp32 inputs, then rounded once to the output type (fp32 by C's
 * round-to-nearest-even conversion; bf16 by a direct round-to-nearest-even from
 * double).  Loops are the plain definitions; OpenMP only spreads independent rows
 * or requests over threads and does not change any result.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define DF2O_OK 0
#define DF2O_INVALID 1
#define DF2O_NOMEM 2

/* Exact value of an IEEE bfloat16 bit pattern. */
static double bf16_value(uint16_t bits)
{
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Round a double to the nearest bfloat16, ties to even, in one step.
 * Going through float first is exact except when the float lands on a bf16
 * midpoint; that case is decided from the double itself. */
static uint16_t bf16_round(double d)
{
    float f = (float)d;
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7F800000u) == 0x7F800000u) {
        if (u & 0x007FFFFFu) return (uint16_t)0x7FC0u; /* NaN */
        return (uint16_t)(u >> 16);                     /* +-inf */
    }
    uint32_t hi = u >> 16, lo = u & 0xFFFFu;
    if (lo == 0x8000u) {
        double ad = fabs(d), am = fabs((double)f);
        if (ad > am) return (uint16_t)(hi + 1u);
        if (ad < am) return (uint16_t)hi;
        return (uint16_t)(hi + (hi & 1u));
    }
    return (uint16_t)(lo > 0x8000u ? hi + 1u : hi);
}

static double act_value(const void* x, int x_is_f32, int64_t idx)
{
    if (x_is_f32) return (double)((const float*)x)[idx];
    return bf16_value(((const uint16_t*)x)[idx]);
}

static void act_store(void* y, int y_is_f32, int64_t idx, double v)
{
    if (y_is_f32) ((float*)y)[idx] = (float)v;
    else ((uint16_t*)y)[idx] = bf16_round(v);
}

int df2o_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Host threads the following calls use (timing only; results do not depend on it). */
void df2o_set_num_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* ---------------------------------------------------------------- logits -- */

/* U[p,v] = sum_d h[p,d] * W[v,d], rounded to fp32. */
int df2o_logits(const uint16_t* h, int64_t P, int64_t D, const uint16_t* W, int64_t V, float* U)
{
    if (P < 0 || D < 1 || V < 1) return DF2O_INVALID;
    int64_t p;
#pragma omp parallel for schedule(dynamic, 1)
    for (p = 0; p < P; ++p) {
        for (int64_t v = 0; v < V; ++v) {
            double acc = 0.0;
            for (int64_t d = 0; d < D; ++d)
                acc += bf16_value(h[p * D + d]) * bf16_value(W[v * D + d]);
            U[p * V + v] = (float)acc;
        }
    }
    return DF2O_OK;
}

/* --------------------------------------------------------------- top-K -- */

typedef struct {
    float val;
    int32_t id;
} cand_t;

/* Rank order: larger value first; equal values, lower token id first. */
static int cand_order(const void* pa, const void* pb)
{
    const cand_t* a = (const cand_t*)pa;
    const cand_t* b = (const cand_t*)pb;
    if (a->val > b->val) return -1;
    if (a->val < b->val) return 1;
    return (a->id > b->id) - (a->id < b->id);
}

/*
 * The optional output multiplier and final logit softcap of the unary logits
 * (SpecForge "DFlash2" concept doc, "Export and serve": both act on the unary
 * logits; the page gives no formula).  Read as the common forms, the multiplier
 * first and the cap last ("final"): u -> mul * u, then cap * tanh(u / cap);
 * cap = 0 means no cap, and mul = 1, cap = 0 leaves the logits as they are.
 */
static double logit_map(double u, double mul, double cap)
{
    const double x = mul * u;
    return cap > 0.0 ? cap * tanh(x / cap) : x;
}

/*
 * Per position p: U[p,.] over all V tokens, each mapped by logit_map, a full
 * sort of the V (value, id) pairs, the first K kept.  margin[p] = U_(K) -
 * U_(K+1) of the mapped values (+inf when K == V).  When W_H is given,
 * G[p,i] = sum_d h[p,d] * W_H[i,d] (the hidden projection H).  mul must be
 * finite and > 0, cap finite and >= 0.
 */
int df2o_unary_topk(const uint16_t* h, int64_t P, int64_t D, const uint16_t* W_lm, int64_t V,
                    int32_t K, double mul, double cap, const uint16_t* W_H, int32_t r, float* G,
                    int32_t* ids, float* vals, double* margin)
{
    if (P < 0 || D < 1 || V < 1 || K < 1 || K > V) return DF2O_INVALID;
    if (!(mul > 0.0) || !isfinite(mul) || !(cap >= 0.0) || !isfinite(cap)) return DF2O_INVALID;
    if (W_H && (r < 1 || !G)) return DF2O_INVALID;
    int failed = 0;
    int64_t p;
#pragma omp parallel for schedule(dynamic, 1)
    for (p = 0; p < P; ++p) {
        cand_t* c = (cand_t*)malloc((size_t)V * sizeof(cand_t));
        if (!c) {
#pragma omp atomic write
            failed = 1;
            continue;
        }
        for (int64_t v = 0; v < V; ++v) {
            double acc = 0.0;
            for (int64_t d = 0; d < D; ++d)
                acc += bf16_value(h[p * D + d]) * bf16_value(W_lm[v * D + d]);
            c[v].val = (float)logit_map(acc, mul, cap);
            c[v].id = (int32_t)v;
        }
        qsort(c, (size_t)V, sizeof(cand_t), cand_order);
        for (int32_t j = 0; j < K; ++j) {
            ids[p * K + j] = c[j].id;
            vals[p * K + j] = c[j].val;
        }
        if (margin) margin[p] = (K < V) ? (double)c[K - 1].val - (double)c[K].val : INFINITY;
        free(c);
        if (W_H) {
            for (int32_t i = 0; i < r; ++i) {
                double acc = 0.0;
                for (int64_t d = 0; d < D; ++d)
                    acc += bf16_value(h[p * D + d]) * bf16_value(W_H[(int64_t)i * D + d]);
                G[p * r + i] = (float)acc;
            }
        }
    }
    return failed ? DF2O_NOMEM : DF2O_OK;
}

/* ------------------------------------------------------------ selector -- */

/* S(a,b) = u + sum_i A[a,i] * G[i] * B[b,i], rounded to fp32. */
static float pair_score(float u, int32_t a, int32_t b, const float* Grow, const uint16_t* A,
                        const uint16_t* Bc, int32_t r)
{
    double s = (double)u;
    for (int32_t i = 0; i < r; ++i)
        s += bf16_value(A[(int64_t)a * r + i]) * (double)Grow[i] * bf16_value(Bc[(int64_t)b * r + i]);
    return (float)s;
}

/*
 * Greedy walk, request q: a_0 = anchors[q]; for t = 1 .. Bsz-1 score the K
 * candidates of row (q, t) against a_{t-1}, pick the best (equal scores: lower
 * token id), record it and its score, and make it a_t.  margin = best - second
 * best (+inf when K == 1).  Row t = 0 (the anchor's own row) is not read.
 * An anchor or candidate id outside [0, V) marks the request invalid: its path
 * entries become -1, its scores NaN, and *status gets bit 1.
 */
int df2o_selector_walk(const int32_t* anchors, int32_t R, int32_t Bsz, const int32_t* ids,
                       const float* vals, const float* G, const uint16_t* A, const uint16_t* Bc,
                       int64_t V, int32_t K, int32_t r, int32_t* path, float* path_score,
                       double* margin, int32_t* status)
{
    if (R < 0 || Bsz < 2 || K < 1 || r < 1 || V < 1 || K > V) return DF2O_INVALID;
    int32_t bad = 0;
    int32_t q;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
    for (q = 0; q < R; ++q) {
        const int64_t T = Bsz - 1;
        int valid = anchors[q] >= 0 && anchors[q] < V;
        for (int64_t t = 1; t < Bsz && valid; ++t)
            for (int32_t j = 0; j < K; ++j) {
                int32_t b = ids[((int64_t)q * Bsz + t) * K + j];
                if (b < 0 || b >= V) valid = 0;
            }
        if (!valid) {
            for (int64_t t = 0; t < T; ++t) {
                path[q * T + t] = -1;
                path_score[q * T + t] = NAN;
                if (margin) margin[q * T + t] = NAN;
            }
            bad |= 1;
            continue;
        }
        int32_t a = anchors[q];
        for (int64_t t = 1; t < Bsz; ++t) {
            const int64_t row = (int64_t)q * Bsz + t;
            float best = -INFINITY, second = -INFINITY;
            int32_t best_id = -1;
            for (int32_t j = 0; j < K; ++j) {
                int32_t b = ids[row * K + j];
                float s = pair_score(vals[row * K + j], a, b, G + row * r, A, Bc, r);
                if (best_id < 0 || s > best || (s == best && b < best_id)) {
                    if (best_id >= 0) second = best;
                    best = s;
                    best_id = b;
                } else if (s > second) {
                    second = s;
                }
            }
            path[q * T + (t - 1)] = best_id;
            path_score[q * T + (t - 1)] = best;
            if (margin) margin[q * T + (t - 1)] = (K > 1) ? (double)best - (double)second : INFINITY;
            a = best_id;
        }
    }
    if (status) *status = bad;
    return DF2O_OK;
}

/*
 * Teacher-forced scores: S[p,j] = vals[p,j] + sum_i A[pred[p],i] G[p,i] B[ids[p,j],i]
 * for every row at once.  A predecessor or candidate id outside [0, V) gives NaN
 * for the affected scores and sets bit 1 of *status.
 */
int df2o_selector_pair_scores(const int32_t* pred, int64_t P, const int32_t* ids, const float* vals,
                              const float* G, const uint16_t* A, const uint16_t* Bc, int64_t V,
                              int32_t K, int32_t r, float* scores, int32_t* status)
{
    if (P < 0 || K < 1 || r < 1 || V < 1) return DF2O_INVALID;
    int32_t bad = 0;
    int64_t p;
#pragma omp parallel for schedule(dynamic, 16) reduction(| : bad)
    for (p = 0; p < P; ++p) {
        int32_t a = pred[p];
        for (int32_t j = 0; j < K; ++j) {
            int32_t b = ids[p * K + j];
            if (a < 0 || a >= V || b < 0 || b >= V) {
                scores[p * K + j] = NAN;
                bad |= 1;
                continue;
            }
            scores[p * K + j] = pair_score(vals[p * K + j], a, b, G + p * r, A, Bc, r);
        }
    }
    if (status) *status = bad;
    return DF2O_OK;
}

/*
 * The selector's training loss, forward (verl-SpeCo PR #62, "Selector training
 * objective"; vLLM Speculators "DFlash2" guide, "Training Objective"): a
 * categorical cross-entropy of the teacher-forced scores over the K candidates the
 * head kept, to which a row contributes only when its ground-truth token is one of
 * those candidates.  Row p holds the
 * teacher-forced scores S[p, 0..K-1] of its candidates ids[p, .] and the ground
 * truth y = targets[p]:
 *     label_idx[p] = the column j with ids[p, j] == y, else -1
 *     loss[p]      = log(sum_j exp(S[p, j])) - S[p, label_idx[p]]   (NaN when -1)
 * in double; the sum is taken after subtracting the row's largest score, which
 * leaves the value unchanged and keeps exp in range.  y < 0 means the row has no
 * target; y >= V sets bit 1 of *status (label -1, loss NaN).
 */
int df2o_selector_ce(const float* scores, const int32_t* ids, const int32_t* targets, int64_t P, int32_t K,
                     int64_t V, float* loss, int32_t* label_idx, int32_t* status)
{
    if (P < 0 || K < 1 || V < 1) return DF2O_INVALID;
    int32_t bad = 0;
    int64_t p;
#pragma omp parallel for schedule(static) reduction(| : bad)
    for (p = 0; p < P; ++p) {
        const int32_t y = targets[p];
        int32_t js = -1;
        if (y >= V) bad |= 1;
        if (y >= 0 && y < V)
            for (int32_t j = 0; j < K; ++j)
                if (ids[p * K + j] == y) {
                    js = j;
                    break;
                }
        label_idx[p] = js;
        if (js < 0) {
            loss[p] = NAN;
            continue;
        }
        double m = -INFINITY;
        for (int32_t j = 0; j < K; ++j)
            if ((double)scores[p * K + j] > m) m = (double)scores[p * K + j];
        double sum = 0.0;
        for (int32_t j = 0; j < K; ++j) sum += exp((double)scores[p * K + j] - m);
        loss[p] = (float)(log(sum) + m - (double)scores[p * K + js]);
    }
    if (status) *status = bad;
    return DF2O_OK;
}

/* ------------------------------------------------------------- lattice -- */

/* 1 when the anchor and every candidate id of rows 1 .. Bsz-1 of request q lie in [0, V). */
static int request_ids_valid(const int32_t* anchors, int32_t q, int32_t Bsz, const int32_t* ids,
                             int64_t V, int32_t K)
{
    if (anchors[q] < 0 || anchors[q] >= V) return 0;
    for (int64_t t = 1; t < Bsz; ++t)
        for (int32_t j = 0; j < K; ++j) {
            int32_t b = ids[((int64_t)q * Bsz + t) * K + j];
            if (b < 0 || b >= V) return 0;
        }
    return 1;
}

/*
 * The lattice of pair scores ("DFlash 2 Explanation", "How It Works", Problem 1:
 * every adjacent pair is scored in one parallel pass and only the final walk over
 * the finished scores is sequential).  Table slot t-1 of request q, for drafted
 * position t = 1 .. Bsz-1, holds
 *     L[q][t-1][i][j] = S_t(a_i, b_j),   b_j = ids[q, t, j],
 * where a_i is the i-th predecessor candidate: ids[q, t-1, i] for t >= 2, and for
 * t = 1 the anchor alone in row i = 0 (rows 1 .. K-1 of slot 0 are NaN).
 * Layout [R][Bsz-1][K][K] fp32.  A request with an id outside [0, V) gets an
 * all-NaN table and sets bit 1 of *status.
 */
int df2o_selector_lattice(const int32_t* anchors, int32_t R, int32_t Bsz, const int32_t* ids,
                          const float* vals, const float* G, const uint16_t* A, const uint16_t* Bc,
                          int64_t V, int32_t K, int32_t r, float* lattice, int32_t* status)
{
    if (R < 0 || Bsz < 2 || K < 1 || r < 1 || V < 1 || K > V) return DF2O_INVALID;
    const int64_t T = Bsz - 1;
    const int64_t KK = (int64_t)K * K;
    int32_t bad = 0;
    int32_t q;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
    for (q = 0; q < R; ++q) {
        float* Lq = lattice + (int64_t)q * T * KK;
        if (!request_ids_valid(anchors, q, Bsz, ids, V, K)) {
            for (int64_t e = 0; e < T * KK; ++e) Lq[e] = NAN;
            bad |= 1;
            continue;
        }
        for (int64_t t = 1; t < Bsz; ++t) {
            const int64_t row = (int64_t)q * Bsz + t;
            float* Lt = Lq + (t - 1) * KK;
            for (int32_t i = 0; i < K; ++i) {
                int32_t a;
                if (t == 1) {
                    if (i > 0) {
                        for (int32_t j = 0; j < K; ++j) Lt[(int64_t)i * K + j] = NAN;
                        continue;
                    }
                    a = anchors[q];
                } else {
                    a = ids[(row - 1) * K + i];
                }
                for (int32_t j = 0; j < K; ++j)
                    Lt[(int64_t)i * K + j] =
                        pair_score(vals[row * K + j], a, ids[row * K + j], G + row * r, A, Bc, r);
            }
        }
    }
    if (status) *status = bad;
    return DF2O_OK;
}

/*
 * The walk over a finished lattice, request q.  The state is the row i of the
 * current predecessor (i = 0, the anchor, at t = 1).  For t = 1 .. Bsz-1 the
 * step reads row i of slot t-1 and picks a column j, which becomes the next row:
 *   greedy (uniforms == NULL): the largest score, equal scores to the lower
 *     token id; margin = best - second best (+inf when K == 1).
 *   sampling: a draw from softmax(L[t-1][i][.] / temperature) by the inverse CDF
 *     in candidate-list order with u = uniforms[q, t-1] in [0, 1): with
 *     w_j = exp((L_j - max_j' L_j') / temperature), the smallest j whose running
 *     sum w_0 + .. + w_j exceeds u * sum(w).  margin = distance of u to the nearer
 *     end of the chosen interval, in probability units (the ends 0 and 1 do not
 *     count; +inf when neither end counts).
 * path = ids[q, t, j] and path_score = L[t-1][i][j].  A request with a candidate
 * id outside [0, V) gets path -1, score NaN, margin NaN and sets bit 1 of *status.
 */
int df2o_lattice_walk(const float* lattice, const int32_t* ids, int32_t R, int32_t Bsz, int32_t K,
                      int64_t V, const float* uniforms, double temperature, int32_t* path,
                      float* path_score, double* margin, int32_t* status)
{
    if (R < 0 || Bsz < 2 || K < 1 || V < 1) return DF2O_INVALID;
    if (uniforms && !(temperature > 0.0)) return DF2O_INVALID;
    const int64_t T = Bsz - 1;
    const int64_t KK = (int64_t)K * K;
    int32_t bad = 0;
    int failed = 0;
    int32_t q;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
    for (q = 0; q < R; ++q) {
        int valid = 1;
        for (int64_t t = 1; t < Bsz && valid; ++t)
            for (int32_t j = 0; j < K; ++j) {
                int32_t b = ids[((int64_t)q * Bsz + t) * K + j];
                if (b < 0 || b >= V) valid = 0;
            }
        if (!valid) {
            for (int64_t t = 0; t < T; ++t) {
                path[q * T + t] = -1;
                path_score[q * T + t] = NAN;
                if (margin) margin[q * T + t] = NAN;
            }
            bad |= 1;
            continue;
        }
        double* w = uniforms ? (double*)malloc((size_t)K * sizeof(double)) : NULL;
        if (uniforms && !w) {
#pragma omp atomic write
            failed = 1;
            continue;
        }
        int32_t i = 0;
        for (int64_t t = 1; t < Bsz; ++t) {
            const int32_t* cand = ids + ((int64_t)q * Bsz + t) * K;
            const float* Lrow = lattice + ((int64_t)q * T + (t - 1)) * KK + (int64_t)i * K;
            int32_t pick = -1;
            double mg;
            if (!uniforms) {
                float best = -INFINITY, second = -INFINITY;
                for (int32_t j = 0; j < K; ++j) {
                    float s = Lrow[j];
                    if (pick < 0 || s > best || (s == best && cand[j] < cand[pick])) {
                        if (pick >= 0) second = best;
                        best = s;
                        pick = j;
                    } else if (second < s) {
                        second = s;
                    }
                }
                mg = (K > 1) ? (double)best - (double)second : INFINITY;
            } else {
                double mx = -INFINITY, total = 0.0;
                for (int32_t j = 0; j < K; ++j)
                    if ((double)Lrow[j] > mx) mx = (double)Lrow[j];
                for (int32_t j = 0; j < K; ++j) {
                    w[j] = exp(((double)Lrow[j] - mx) / temperature);
                    total += w[j];
                }
                const double u = (double)uniforms[q * T + (t - 1)];
                double below = 0.0;  /* running sum of the weights before j */
                for (int32_t j = 0; j < K; ++j) {
                    if (below + w[j] > u * total) {
                        pick = j;
                        break;
                    }
                    below += w[j];
                }
                if (pick < 0) /* u * total rounded up to the full sum: the last nonzero weight */
                    for (int32_t j = K - 1; j >= 0 && pick < 0; --j)
                        if (w[j] > 0.0) pick = j;
                double lo = 0.0;
                for (int32_t j = 0; j < pick; ++j) lo += w[j];
                const double hi = lo + w[pick];
                mg = INFINITY;
                if (pick > 0) mg = u - lo / total;
                if (pick < K - 1 && hi / total - u < mg) mg = hi / total - u;
            }
            path[q * T + (t - 1)] = cand[pick];
            path_score[q * T + (t - 1)] = Lrow[pick];
            if (margin) margin[q * T + (t - 1)] = mg;
            i = pick;
        }
        free(w);
    }
    if (status) *status = bad;
    return failed ? DF2O_NOMEM : DF2O_OK;
}

/* ---------------------------------------------------------------- conv -- */

static int conv_args_ok(int64_t P, int32_t C, int32_t Bsz, int32_t taps, int32_t g)
{
    return P >= 0 && C >= 1 && Bsz >= 1 && g >= 1 && C % g == 0 && taps >= 1 && taps <= Bsz &&
           P % Bsz == 0;
}

/*
 * Prepare (before the sublayer), row p with in-block position t = p mod Bsz:
 *   d[io][j][gi] = sum_c W_proj[(io*taps + j)*G + gi][c] * x[p][c]
 *   y[p][c]      = sum_{j < taps, t-j >= 0} (base[0][j][c] + d[0][j][c/g]) * x[p-j][c]
 *   dyn_out[p][j][gi] = d[1][j][gi]   (the kernel correction finish applies)
 * y has x's type; x_is_f32 selects fp32 (else bf16) activations.
 */
int df2o_conv_prepare(const void* x, int x_is_f32, int64_t P, int32_t C, int32_t Bsz, int32_t taps,
                      int32_t g, const uint16_t* W_proj, const float* base, void* y, float* dyn_out)
{
    if (!conv_args_ok(P, C, Bsz, taps, g)) return DF2O_INVALID;
    const int32_t G = C / g;
    const int64_t NP = 2LL * taps * G;
    int failed = 0;
    int64_t p;
#pragma omp parallel for schedule(dynamic, 4)
    for (p = 0; p < P; ++p) {
        double* d = (double*)malloc((size_t)NP * sizeof(double));
        if (!d) {
#pragma omp atomic write
            failed = 1;
            continue;
        }
        for (int64_t n = 0; n < NP; ++n) {
            double acc = 0.0;
            for (int32_t c = 0; c < C; ++c)
                acc += bf16_value(W_proj[n * C + c]) * act_value(x, x_is_f32, p * C + c);
            d[n] = acc;
        }
        for (int32_t j = 0; j < taps; ++j)
            for (int32_t gi = 0; gi < G; ++gi)
                dyn_out[(p * taps + j) * G + gi] = (float)d[((int64_t)1 * taps + j) * G + gi];
        const int64_t t = p % Bsz;
        for (int32_t c = 0; c < C; ++c) {
            double acc = 0.0;
            for (int32_t j = 0; j < taps; ++j) {
                if (t - j < 0) continue;
                double k = (double)base[((int64_t)0 * taps + j) * C + c] +
                           d[((int64_t)0 * taps + j) * G + c / g];
                acc += k * act_value(x, x_is_f32, (p - j) * C + c);
            }
            act_store(y, x_is_f32, p * C + c, acc);
        }
        free(d);
    }
    return failed ? DF2O_NOMEM : DF2O_OK;
}

/*
 * Finish (after the sublayer), with the correction prepare emitted:
 *   y[p][c] = sum_{j < taps, t-j >= 0} (base[1][j][c] + dyn_out[p][j][c/g]) * z[p-j][c]
 */
int df2o_conv_finish(const void* z, int z_is_f32, int64_t P, int32_t C, int32_t Bsz, int32_t taps,
                     int32_t g, const float* dyn_out, const float* base, void* y)
{
    if (!conv_args_ok(P, C, Bsz, taps, g)) return DF2O_INVALID;
    const int32_t G = C / g;
    int64_t p;
#pragma omp parallel for schedule(dynamic, 16)
    for (p = 0; p < P; ++p) {
        const int64_t t = p % Bsz;
        for (int32_t c = 0; c < C; ++c) {
            double acc = 0.0;
            for (int32_t j = 0; j < taps; ++j) {
                if (t - j < 0) continue;
                double k = (double)base[((int64_t)1 * taps + j) * C + c] +
                           (double)dyn_out[(p * taps + j) * G + c / g];
                acc += k * act_value(z, z_is_f32, (p - j) * C + c);
            }
            act_store(y, z_is_f32, p * C + c, acc);
        }
    }
    return DF2O_OK;
}

/*
 * The two convs that meet between consecutive sublayers of a draft layer: the
 * finish of one sublayer, then the prepare of the next (vLLM Speculators "DFlash2"
 * guide, "Local Convolution": each attention and MLP sublayer has a conv on its
 * input side and one on its output side).  The pages do not state the residual wiring between the
 * two.  Reading: h = finish(z), plus the residual stream when one is given (the sum
 * rounded to the activation dtype, as a separate elementwise add would round it),
 * then prepare(h) with the next sublayer's projection and base kernels.  Writes
 * h, y_next and dyn_next.
 */
int df2o_conv_finish_prepare(const void* z, int is_f32, int64_t P, int32_t C, int32_t Bsz, int32_t taps,
                             int32_t g, const float* dyn_out, const float* base, const void* residual,
                             void* h, const uint16_t* W_proj, const float* base_next, void* y_next,
                             float* dyn_next)
{
    int rc = df2o_conv_finish(z, is_f32, P, C, Bsz, taps, g, dyn_out, base, h);
    if (rc != DF2O_OK) return rc;
    if (residual) {
        for (int64_t i = 0; i < P * (int64_t)C; ++i)
            act_store(h, is_f32, i, act_value(h, is_f32, i) + act_value(residual, is_f32, i));
    }
    return df2o_conv_prepare(h, is_f32, P, C, Bsz, taps, g, W_proj, base_next, y_next, dyn_next);
}
