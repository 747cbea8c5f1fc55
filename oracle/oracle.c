/*
 * oracle.c -- plain, slow CPU reference ("the oracle") for the DFlash2
 * candidate-selector head.
 *
 * TEST INFRASTRUCTURE ONLY.  The tests, the package's smoke check and the
 * benchmark's CPU-baseline / reference leg may load this library.  The product
 * path (the CUDA library and its binding) never includes, links or calls it,
 * and shares no code with it.
 *
 * What it computes, step by step, with no blocking, fusion or reordering
 * beyond the definitions:
 *
 *  1. LM head.  logit[r,v] = sum_h hidden[r,h] * W_vocab[v,h].
 *     "DFlash 2: Keep Drafting Parallel", section "A Lightweight Path
 *     Selector": the unary term U_t(b) is the drafter's own logit.  Each
 *     product of two bf16 values is exact in double; the sum runs in double
 *     in increasing h and is rounded once to float32 (the float32 logits the
 *     method's engines hand to top-k).
 *  2. Top-k.  Full sort of each row by (logit desc, token id asc), first k.
 *     "DFlash2 Lands in llama.cpp", section "What llama.cpp Actually Builds
 *     for the Selector": candidates = top_k(logits); the unary scores are the
 *     candidates' logits.  Ties go to the lower token id.
 *  3. Gate.  g[r,d] = sum_h W_sel[d,h] * hidden[r,h], in double, linear with
 *     no bias: the hidden state of the current position projected through the
 *     selector projection (same section of the llama.cpp page; "context gate
 *     H(h_t)" on the DFlash 2 page).
 *  4. Lattice.  For position r = b*T + t, predecessor candidates are the
 *     previous position's candidates, or the anchor (last verified token) at
 *     t = 0; S[r,i,j] = U[r,j] + sum_d (A[prev_i,d] * g[r,d]) * B[cand_j,d]
 *     (DFlash 2 page, equation S_t(a,b) = U_t(b) + <A(a) (.) H(h_t), B(b)>;
 *     llama.cpp page, section "The Central Insight": edge = unary + pairwise).
 *     Computed in double, rounded once to float32.
 *  5. Packing.  Row r = [k candidate ids as exact floats | S[r,i,j] with the
 *     predecessor index i major] (llama.cpp page: each row holds the candidate
 *     IDs followed by the transition scores).  At t = 0 every predecessor row
 *     holds the anchor-conditioned scores.
 *  6. Walk.  j_0 = argmax_j S[(b,0),0,j]; j_t = argmax_j S[(b,t),j_{t-1},j];
 *     draft[b,t] = cand[(b,t), j_t]; the first maximum wins (llama.cpp page,
 *     the predecessor = anchor walk; DFlash 2 page: greedy follows the best
 *     successor at each step).  Decided on the float32 lattice.
 *  7. Confidence, p_min and sampling (oracle_walk_sample).  On the row the
 *     walk reads, p_j = softmax(S / temperature)_j.  Greedy takes the first
 *     maximum; sampling takes the first j whose running sum of p (in index
 *     order) exceeds the given uniform u (DFlash 2 page: sampling draws from
 *     the same scores).  The chosen transition's confidence is p_{j_t}; when it
 *     is below p_min the walk stops and emits nothing from t on ("DFlash2 Lands
 *     in llama.cpp", section "p_min Means Something Different Under DFlash2").
 *     Computed in double.
 *
 * bf16 tensors are passed as their uint16 bit patterns.  Every function
 * returns 0 on success and a negative code on bad arguments or non-finite
 * values.  Build: gcc -O2 -fopenmp -ffp-contract=off (no fused multiply-add,
 * so x86 and Arm give the same bits).
 */
#include <math.h>
#include <stdint.h>
#ifdef _OPENMP
#include <omp.h>
#endif
#include <stdlib.h>
#include <string.h>

/* Threads the OpenMP loops below use (1 without OpenMP). */
int oracle_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Threads for the following calls (n >= 1); returns the previous count.  Only the
 * baseline timing uses it, to time the oracle on one core as well as on all of them. */
int oracle_set_threads(int n)
{
    const int prev = oracle_threads();
#ifdef _OPENMP
    if (n >= 1)
        omp_set_num_threads(n);
#else
    (void)n;
#endif
    return prev;
}

static double bf16_to_double(uint16_t bits)
{
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Step 1: float32 logits (double accumulation, one rounding).  logits64 may be NULL. */
int oracle_logits(const uint16_t *hidden, const uint16_t *W_vocab, int64_t R, int64_t H, int64_t V,
                  float *logits, double *logits64)
{
    if (!hidden || !W_vocab || !logits || R < 0 || H <= 0 || V <= 0)
        return -1;
#pragma omp parallel for collapse(2) schedule(static)
    for (int64_t r = 0; r < R; ++r) {
        for (int64_t v = 0; v < V; ++v) {
            const uint16_t *hr = hidden + r * H;
            const uint16_t *wv = W_vocab + v * H;
            double acc = 0.0;
            for (int64_t h = 0; h < H; ++h)
                acc += bf16_to_double(hr[h]) * bf16_to_double(wv[h]);
            logits[r * V + v] = (float)acc;
            if (logits64)
                logits64[r * V + v] = acc;
        }
    }
    return 0;
}

typedef struct {
    float value;
    int32_t id;
} scored_token;

/* (value desc, id asc): a strict total order on distinct ids. */
static int by_value_desc_id_asc(const void *pa, const void *pb)
{
    const scored_token *a = (const scored_token *)pa;
    const scored_token *b = (const scored_token *)pb;
    if (a->value > b->value)
        return -1;
    if (a->value < b->value)
        return 1;
    return (a->id < b->id) ? -1 : (a->id > b->id) ? 1 : 0;
}

/* Step 2: top-k of each row by a full sort. */
int oracle_topk(const float *logits, int64_t R, int64_t V, int32_t k, int32_t *ids, float *vals)
{
    if (!logits || !ids || !vals || R < 0 || V <= 0 || k < 1 || k > V)
        return -1;
    for (int64_t i = 0; i < R * V; ++i)
        if (!isfinite(logits[i]))
            return -2;
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
    for (int64_t r = 0; r < R; ++r) {
        scored_token *row = (scored_token *)malloc((size_t)V * sizeof *row);
        if (!row) {
            bad |= 1;
            continue;
        }
        for (int64_t v = 0; v < V; ++v) {
            row[v].value = logits[r * V + v];
            row[v].id = (int32_t)v;
        }
        qsort(row, (size_t)V, sizeof *row, by_value_desc_id_asc);
        for (int32_t j = 0; j < k; ++j) {
            ids[r * k + j] = row[j].id;
            vals[r * k + j] = row[j].value;
        }
        free(row);
    }
    return bad ? -3 : 0;
}

/* Step 3: gate in double. */
int oracle_gate(const uint16_t *hidden, const uint16_t *W_sel, int64_t R, int64_t H, int64_t D, double *gate)
{
    if (!hidden || !W_sel || !gate || R < 0 || H <= 0 || D <= 0)
        return -1;
#pragma omp parallel for collapse(2) schedule(static)
    for (int64_t r = 0; r < R; ++r) {
        for (int64_t d = 0; d < D; ++d) {
            double acc = 0.0;
            for (int64_t h = 0; h < H; ++h)
                acc += bf16_to_double(W_sel[d * H + h]) * bf16_to_double(hidden[r * H + h]);
            gate[r * D + d] = acc;
        }
    }
    return 0;
}

/*
 * Steps 4-5: packed lattice rows, float32 [B*T, k + k*k]; lattice64 (may be
 * NULL) receives the unrounded double scores [B*T, k*k].
 */
int oracle_lattice(int64_t B, int64_t T, int32_t k, int64_t V, int64_t D, const int32_t *cand_ids,
                   const float *unary, const double *gate, const uint16_t *pred_cb, const uint16_t *succ_cb,
                   const int32_t *anchor, float *lattice, double *lattice64)
{
    if (B < 0 || T <= 0 || k < 1 || V <= 0 || D <= 0 || !cand_ids || !unary || !gate || !pred_cb || !succ_cb ||
        !anchor || !lattice)
        return -1;
    for (int64_t b = 0; b < B; ++b)
        if (anchor[b] < 0 || anchor[b] >= V)
            return -2;
    for (int64_t i = 0; i < B * T * k; ++i)
        if (cand_ids[i] < 0 || cand_ids[i] >= V)
            return -2;
    const int64_t width = (int64_t)k + (int64_t)k * k;
#pragma omp parallel for collapse(2) schedule(static)
    for (int64_t b = 0; b < B; ++b) {
        for (int64_t t = 0; t < T; ++t) {
            const int64_t r = b * T + t;
            float *row = lattice + r * width;
            for (int32_t j = 0; j < k; ++j)
                row[j] = (float)cand_ids[r * k + j];
            for (int32_t i = 0; i < k; ++i) {
                const int64_t prev = (t == 0) ? anchor[b] : cand_ids[(r - 1) * k + i];
                for (int32_t j = 0; j < k; ++j) {
                    const int64_t cand = cand_ids[r * k + j];
                    double pairwise = 0.0;
                    for (int64_t d = 0; d < D; ++d)
                        pairwise += (bf16_to_double(pred_cb[prev * D + d]) * gate[r * D + d]) *
                                    bf16_to_double(succ_cb[cand * D + d]);
                    const double s = (double)unary[r * k + j] + pairwise;
                    row[k + (int64_t)i * k + j] = (float)s;
                    if (lattice64)
                        lattice64[r * (int64_t)k * k + (int64_t)i * k + j] = s;
                }
            }
        }
    }
    return 0;
}

/* Step 6: greedy walk on the packed float32 lattice.  choice (may be NULL) gets j_t. */
int oracle_walk(int64_t B, int64_t T, int32_t k, const float *lattice, int32_t *draft, int32_t *choice)
{
    if (B < 0 || T <= 0 || k < 1 || !lattice || !draft)
        return -1;
    const int64_t width = (int64_t)k + (int64_t)k * k;
    for (int64_t b = 0; b < B; ++b) {
        int32_t jprev = 0; /* position 0: every predecessor row holds the anchor's scores */
        for (int64_t t = 0; t < T; ++t) {
            const float *row = lattice + (b * T + t) * width;
            const float *scores = row + k + (int64_t)jprev * k;
            int32_t best = 0;
            for (int32_t j = 1; j < k; ++j)
                if (scores[j] > scores[best])
                    best = j;
            draft[b * T + t] = (int32_t)row[best];
            if (choice)
                choice[b * T + t] = best;
            jprev = best;
        }
    }
    return 0;
}

/*
 * Step 7: walk with confidence, p_min early stop and optional sampling on the
 * packed float32 lattice.  uniforms [B*T] in [0,1) selects sampling (NULL:
 * greedy).  Outputs draft [B*T] (-1 from the stop on), n_draft [B] (tokens
 * emitted), confidence [B*T] (p of the chosen transition up to and including
 * the stopping step, 0 after it).  temperature must be > 0.
 */
int oracle_walk_sample(int64_t B, int64_t T, int32_t k, const float *lattice, double temperature, double p_min,
                       const float *uniforms, int32_t *draft, int32_t *n_draft, double *confidence)
{
    if (B < 0 || T <= 0 || k < 1 || !lattice || !draft || !n_draft || !confidence || !(temperature > 0.0))
        return -1;
    const int64_t width = (int64_t)k + (int64_t)k * k;
    double *p = (double *)malloc((size_t)k * sizeof *p);
    if (!p)
        return -3;
    for (int64_t b = 0; b < B; ++b) {
        int32_t jprev = 0;
        int stopped = 0;
        n_draft[b] = (int32_t)T;
        for (int64_t t = 0; t < T; ++t) {
            const int64_t r = b * T + t;
            if (stopped) {
                draft[r] = -1;
                confidence[r] = 0.0;
                continue;
            }
            const float *row = lattice + r * width;
            const float *scores = row + k + (int64_t)jprev * k;
            double m = scores[0];
            for (int32_t j = 1; j < k; ++j)
                if (scores[j] > m)
                    m = scores[j];
            double z = 0.0;
            for (int32_t j = 0; j < k; ++j) {
                p[j] = exp(((double)scores[j] - m) / temperature);
                z += p[j];
            }
            for (int32_t j = 0; j < k; ++j)
                p[j] /= z;
            int32_t pick = 0;
            if (uniforms) {
                const double u = uniforms[r];
                double run = 0.0;
                pick = k - 1; /* if rounding leaves the total at or below u: the last candidate with weight */
                while (pick > 0 && p[pick] == 0.0)
                    --pick;
                for (int32_t j = 0; j < k; ++j) {
                    run += p[j];
                    if (run > u) {
                        pick = j;
                        break;
                    }
                }
            } else {
                for (int32_t j = 1; j < k; ++j)
                    if (scores[j] > scores[pick])
                        pick = j;
            }
            confidence[r] = p[pick];
            if (p[pick] < p_min) {
                stopped = 1;
                n_draft[b] = (int32_t)t;
                draft[r] = -1;
                continue;
            }
            draft[r] = (int32_t)row[pick];
            jprev = pick;
        }
    }
    free(p);
    return 0;
}

/*
 * Grouped two-tap dynamic depthwise convolution ("DFlash 2: Keep Drafting Parallel",
 * section "A Lightweight Local Convolution": Conv_k(x)_t = k_{t,0} (.) x_t + k_{t,1} (.)
 * x_{t-1}, each coefficient a learned base plus a correction shared by every 16
 * channels, the first position reading the last verified token; "DFlash2 Lands in
 * llama.cpp", section "Dynamic Local Convolution": static per-channel weight plus a
 * per-group dynamic weight, block-local shift).  In double:
 *   xn(v)   = v                                   without normalisation (gamma NULL)
 *           = v / sqrt(mean(v^2) + eps) * gamma   RMS-normalised row (a zero row stays zero)
 *   y[r,c]  = (base[0,c] + dyn[r,0,c/G]) * xn(x[r])[c] + (base[1,c] + dyn[r,1,c/G]) * xn(prev)[c]
 *   prev    = x[r-1] for t > 0; x_prev[b] at t = 0 (a zero row if x_prev is NULL).
 * x, x_prev, base, gamma: bf16 bits; dyn: float [B*T, 2, C/G]; y: double [B*T, C].
 */
int oracle_dynamic_conv(int64_t B, int64_t T, int64_t C, int64_t G, const uint16_t *x, const uint16_t *x_prev,
                        const uint16_t *base, const float *dyn, const uint16_t *gamma, double eps, double *y)
{
    if (B < 0 || T <= 0 || C <= 0 || G <= 0 || C % G != 0 || !x || !base || !dyn || !y || eps < 0.0)
        return -1;
    const int64_t groups = C / G;
    double *cur = (double *)malloc((size_t)C * sizeof *cur);
    double *prv = (double *)malloc((size_t)C * sizeof *prv);
    if (!cur || !prv) {
        free(cur);
        free(prv);
        return -3;
    }
    for (int64_t b = 0; b < B; ++b) {
        for (int64_t t = 0; t < T; ++t) {
            const int64_t r = b * T + t;
            for (int64_t c = 0; c < C; ++c) {
                cur[c] = bf16_to_double(x[r * C + c]);
                if (t > 0)
                    prv[c] = bf16_to_double(x[(r - 1) * C + c]);
                else
                    prv[c] = x_prev ? bf16_to_double(x_prev[b * C + c]) : 0.0;
            }
            if (gamma) {
                double sc = 0.0, sp = 0.0;
                for (int64_t c = 0; c < C; ++c) {
                    sc += cur[c] * cur[c];
                    sp += prv[c] * prv[c];
                }
                /* an all-zero row normalises to zero (even with eps = 0) */
                const double ic = (sc > 0.0 || eps > 0.0) ? 1.0 / sqrt(sc / (double)C + eps) : 0.0;
                const double ip = (sp > 0.0 || eps > 0.0) ? 1.0 / sqrt(sp / (double)C + eps) : 0.0;
                for (int64_t c = 0; c < C; ++c) {
                    const double gm = bf16_to_double(gamma[c]);
                    cur[c] = cur[c] * ic * gm;
                    prv[c] = prv[c] * ip * gm;
                }
            }
            for (int64_t c = 0; c < C; ++c) {
                const int64_t g = c / G;
                const double k0 = bf16_to_double(base[c]) + (double)dyn[(r * 2 + 0) * groups + g];
                const double k1 = bf16_to_double(base[C + c]) + (double)dyn[(r * 2 + 1) * groups + g];
                y[r * C + c] = k0 * cur[c] + k1 * prv[c];
            }
        }
    }
    free(cur);
    free(prv);
    return 0;
}
