/*
 * moe_oracle.c -- TEST INFRASTRUCTURE, NOT PRODUCT CODE.
 *
 * A plain, slow, obviously-correct CPU statement of the forward pass of a
 * sparsely-gated Mixture-of-Experts SwiGLU FFN layer, in double precision, one
 * token at a time.  Only the test-suite, the smoke check and the benchmark's
 * CPU-baseline leg may load it.  It shares no code, header, table or helper with
 * the CUDA library and includes nothing from it.
 *
 * Inputs arrive as float arrays holding the exact run-dtype values (bf16 and fp32
 * values are both exactly representable in float) and are widened to double
 * before any arithmetic.  Nothing is rounded in between.
 *
 * Sources (page title, then section):
 *   [P2] "技术日报 2026-04-14" (jsqmd.com):
 *        §3.1 Top-K routing (KeepTopK, Softmax, weighted sum y = sum G_i E_i),
 *        §3.2 Switch top-1 routing and capacity K_max = floor(C * N_tokens / N_experts),
 *             overflow tokens dropped,
 *        §3.3 Expert Choice: each expert takes the top tokens of its column of S,
 *        §3.4 DeepSeekMoE: shared experts added unweighted,
 *        §3.5 DeepSeek-V3 sigmoid gate s = Sigmoid(u),
 *        §4.3 bias b_i used for selection only, weights from the unbiased score,
 *        §9.1 MoELayer.forward (softmax, topk, renormalise over the selected k,
 *             shared experts summed), §9.2 AuxFreeRouter.forward.
 *   [P3] "MoE稀疏架构" (cloud.baidu.com), §4 工作原理: gate -> Top-K -> dispatch ->
 *        experts -> gate-weighted aggregation.
 *   [P4] lnwmold.com GPT-4 MoE article, §2.2: each expert is an FFN with W1, W2, W3.
 * Readings where the pages are silent:
 *   - expert = SwiGLU: E(x) = (SiLU(x W1) * (x W3)) W2, SiLU(z) = z / (1 + e^-z);
 *   - capacity for k slots per token: floor(C * T * k / E), assignments kept in
 *     token order (t ascending, then slot j ascending), the rest dropped;
 *   - ties in every selection go to the lower index (expert, or token for EC);
 *   - Expert Choice affinity S = softmax over experts of the router logits.
 *
 * Layouts (row-major):  x[T][d], W_r[d][E], W1/W3[d][f] and W2[f][d] per expert.
 *
 * Parity pins for every function live in tests/test_oracle_pins.py.
 */
#include <float.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_GATE_SOFTMAX 0
#define ORACLE_GATE_SIGMOID 1

/* Capacity of one expert: floor(C * T * k / E) ([P2] §3.2, k = 1 there; the k
 * factor is the reading above).  C <= 0 means "no limit" and returns -1. */
int64_t oracle_capacity(double C, int64_t T, int64_t k, int64_t E)
{
    if (C <= 0.0) return -1;
    return (int64_t)floor(C * (double)T * (double)k / (double)E);
}

/* Router logits of one token: u_e = sum_i x_i W_r[i][e] (+ logit_offset_e). */
static void router_logits(int d, int E, const float *x, const float *Wr,
                          const float *logit_offset, double *u)
{
    for (int e = 0; e < E; ++e) u[e] = 0.0;
    for (int i = 0; i < d; ++i) {
        const double xi = (double)x[i];
        const float *row = Wr + (size_t)i * E;
        for (int e = 0; e < E; ++e) u[e] += xi * (double)row[e];
    }
    if (logit_offset)
        for (int e = 0; e < E; ++e) u[e] += (double)logit_offset[e];
}

/* Softmax over E: p_e = exp(u_e - max) / sum_j exp(u_j - max) ([P2] §3.2). */
static void softmax(int E, const double *u, double *p)
{
    double m = -INFINITY;
    for (int e = 0; e < E; ++e) if (u[e] > m) m = u[e];
    double s = 0.0;
    for (int e = 0; e < E; ++e) { p[e] = exp(u[e] - m); s += p[e]; }
    for (int e = 0; e < E; ++e) p[e] /= s;
}

/* Sigmoid score s_e = 1 / (1 + exp(-u_e)) ([P2] §3.5). */
static void sigmoid(int E, const double *u, double *s)
{
    for (int e = 0; e < E; ++e) s[e] = 1.0 / (1.0 + exp(-u[e]));
}

/*
 * Token-choice routing for every token ([P2] §3.1, §3.2, §3.5, §4.3, §9.1, §9.2).
 *   score = softmax(u) or sigmoid(u);  key = score (+ sel_bias, selection only);
 *   k rounds: take the not-yet-chosen expert with the largest key, lowest index
 *   on ties, so slots come out in descending key order;
 *   weight_j = score of the chosen expert, divided by the sum of the k chosen
 *   scores when renorm != 0.
 * Outputs: topk_idx[T][k], topk_w[T][k], gap[T] = key of the k-th choice minus the
 * best key left unchosen (+INF when k == E), scores[T][E] (optional, may be NULL).
 */
int oracle_route_tc(int T, int d, int E, int k, const float *x, const float *Wr,
                    const float *logit_offset, int gate, const float *sel_bias,
                    int renorm, int32_t *topk_idx, double *topk_w, double *gap,
                    double *scores_out, int nthreads)
{
    if (T < 0 || d <= 0 || E <= 0 || k <= 0 || k > E) return -1;
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 16) num_threads(nthreads > 0 ? nthreads : 1)
    for (int t = 0; t < T; ++t) {
        double *u = (double *)malloc(sizeof(double) * E * 3);
        char *chosen = (char *)calloc((size_t)E, 1);
        if (!u || !chosen) { bad = 1; free(u); free(chosen); continue; }
        double *score = u + E, *key = u + 2 * E;
        router_logits(d, E, x + (size_t)t * d, Wr, logit_offset, u);
        if (gate == ORACLE_GATE_SIGMOID) sigmoid(E, u, score);
        else softmax(E, u, score);
        for (int e = 0; e < E; ++e)
            key[e] = score[e] + (sel_bias ? (double)sel_bias[e] : 0.0);

        double sum_sel = 0.0, last_key = 0.0;
        for (int j = 0; j < k; ++j) {
            int best = -1;
            for (int e = 0; e < E; ++e) {
                if (chosen[e]) continue;
                if (best < 0 || key[e] > key[best]) best = e;   /* strict: lowest index wins ties */
            }
            chosen[best] = 1;
            topk_idx[(size_t)t * k + j] = best;
            topk_w[(size_t)t * k + j] = score[best];
            sum_sel += score[best];
            last_key = key[best];
        }
        if (renorm)
            for (int j = 0; j < k; ++j) topk_w[(size_t)t * k + j] /= sum_sel;

        double best_left = -INFINITY;
        for (int e = 0; e < E; ++e)
            if (!chosen[e] && key[e] > best_left) best_left = key[e];
        gap[t] = (k == E) ? INFINITY : last_key - best_left;

        if (scores_out) memcpy(scores_out + (size_t)t * E, score, sizeof(double) * E);
        free(u);
        free(chosen);
    }
    return bad ? -2 : 0;
}

/* --- Expert Choice ([P2] §3.3) --------------------------------------------- */

static const double *g_col;   /* column being ordered (single-threaded section) */
static int g_E;

static int by_score_desc_then_token(const void *a, const void *b)
{
    const int ta = *(const int *)a, tb = *(const int *)b;
    const double sa = g_col[(size_t)ta * g_E], sb = g_col[(size_t)tb * g_E];
    if (sa > sb) return -1;
    if (sa < sb) return 1;
    return (ta < tb) ? -1 : (ta > tb);
}

static int int_asc(const void *a, const void *b)
{
    const int x = *(const int *)a, y = *(const int *)b;
    return (x < y) ? -1 : (x > y);
}

/*
 * Expert Choice routing.  S[t][e] = softmax over experts of the router logits of
 * token t.  Expert e orders all tokens by (S[t][e] descending, t ascending) and
 * takes the first cap; they are listed in ascending token order:
 *   ec_tok[e][r], ec_w[e][r] = S[ec_tok[e][r]][e].
 * gap[e] = S of the cap-th taken token minus S of the first token left out
 * (+INF when cap == T).  S_out[T][E] is optional.
 */
int oracle_route_ec(int T, int d, int E, int cap, const float *x, const float *Wr,
                    const float *logit_offset, int32_t *ec_tok, double *ec_w,
                    double *gap, double *S_out, int nthreads)
{
    if (T <= 0 || d <= 0 || E <= 0 || cap <= 0 || cap > T) return -1;
    double *S = (double *)malloc(sizeof(double) * (size_t)T * E);
    int *order = (int *)malloc(sizeof(int) * (size_t)T);
    if (!S || !order) { free(S); free(order); return -2; }
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 16) num_threads(nthreads > 0 ? nthreads : 1)
    for (int t = 0; t < T; ++t) {
        double *u = (double *)malloc(sizeof(double) * E);
        if (!u) { bad = 1; continue; }
        router_logits(d, E, x + (size_t)t * d, Wr, logit_offset, u);
        softmax(E, u, S + (size_t)t * E);
        free(u);
    }
    if (bad) { free(S); free(order); return -2; }
    for (int e = 0; e < E; ++e) {
        for (int t = 0; t < T; ++t) order[t] = t;
        g_col = S + e;
        g_E = E;
        qsort(order, (size_t)T, sizeof(int), by_score_desc_then_token);
        gap[e] = (cap == T) ? INFINITY
                            : S[(size_t)order[cap - 1] * E + e] - S[(size_t)order[cap] * E + e];
        qsort(order, (size_t)cap, sizeof(int), int_asc);
        for (int r = 0; r < cap; ++r) {
            ec_tok[(size_t)e * cap + r] = order[r];
            ec_w[(size_t)e * cap + r] = S[(size_t)order[r] * E + e];
        }
    }
    if (S_out) memcpy(S_out, S, sizeof(double) * (size_t)T * E);
    free(S);
    free(order);
    return 0;
}

/*
 * Token-choice dispatch with the capacity limit ([P2] §3.2; [P3] §4 step 3).
 * Assignments are visited in token order t = 0..T-1, and slot order j = 0..k-1
 * inside a token.  An assignment to expert e is kept while fewer than cap
 * assignments to e have been kept (cap < 0: always kept), otherwise dropped.
 *   cnt_raw[e] = assignments made to e;  kept count n_e = min(cnt_raw[e], cap);
 *   off[e] = n_0 + ... + n_{e-1}, off[E] = total kept;
 *   slot_of[t][j] = off[e] + (rank of the assignment among e's kept ones), -1 if
 *   dropped;  row_token[slot] = t.
 */
int oracle_dispatch_tc(int T, int k, int E, int64_t cap, const int32_t *topk_idx,
                       int32_t *off, int32_t *cnt_raw, int32_t *slot_of, int32_t *row_token)
{
    if (T < 0 || k <= 0 || E <= 0) return -1;
    int32_t *kept = (int32_t *)calloc((size_t)E, sizeof(int32_t));
    if (!kept) return -2;
    for (int e = 0; e < E; ++e) cnt_raw[e] = 0;
    /* pass 1: rank of each kept assignment within its expert */
    for (int t = 0; t < T; ++t) {
        for (int j = 0; j < k; ++j) {
            const int e = topk_idx[(size_t)t * k + j];
            if (e < 0 || e >= E) { free(kept); return -3; }
            cnt_raw[e] += 1;
            if (cap < 0 || kept[e] < cap) {
                slot_of[(size_t)t * k + j] = kept[e];
                kept[e] += 1;
            } else {
                slot_of[(size_t)t * k + j] = -1;
            }
        }
    }
    off[0] = 0;
    for (int e = 0; e < E; ++e) off[e + 1] = off[e] + kept[e];
    /* pass 2: rank -> global row */
    for (int t = 0; t < T; ++t) {
        for (int j = 0; j < k; ++j) {
            int32_t *s = slot_of + (size_t)t * k + j;
            if (*s < 0) continue;
            *s += off[topk_idx[(size_t)t * k + j]];
            row_token[*s] = t;
        }
    }
    free(kept);
    return 0;
}

/*
 * One SwiGLU expert applied to one token ([P4] §2.2 W1, W2, W3; SwiGLU reading):
 *   a_c = sum_i x_i W1[i][c],  b_c = sum_i x_i W3[i][c],
 *   h_c = SiLU(a_c) * b_c = a_c / (1 + exp(-a_c)) * b_c,
 *   out_r += scale * sum_c h_c W2[c][r].
 * Each sum runs over its index in ascending order.  `out` is accumulated into.
 */
void oracle_swiglu_expert(int d, int f, const float *x, const float *W1, const float *W3,
                          const float *W2, double scale, double *out)
{
    double *a = (double *)calloc((size_t)f * 2, sizeof(double));
    double *b = a + f;
    for (int i = 0; i < d; ++i) {
        const double xi = (double)x[i];
        const float *r1 = W1 + (size_t)i * f, *r3 = W3 + (size_t)i * f;
        for (int c = 0; c < f; ++c) { a[c] += xi * (double)r1[c]; b[c] += xi * (double)r3[c]; }
    }
    double *o = (double *)calloc((size_t)d, sizeof(double));
    for (int c = 0; c < f; ++c) {
        const double h = a[c] / (1.0 + exp(-a[c])) * b[c];
        const float *r2 = W2 + (size_t)c * d;
        for (int r = 0; r < d; ++r) o[r] += h * (double)r2[r];
    }
    for (int r = 0; r < d; ++r) out[r] += scale * o[r];
    free(o);
    free(a);
}

/*
 * One expert applied to n rows: out[r][:] = scale[r] * E(X[r]) (scale NULL = 1).
 * Same arithmetic as oracle_swiglu_expert, rows spread over threads.
 */
void oracle_expert_rows(int d, int f, int n, const float *X, const float *W1, const float *W3,
                        const float *W2, const double *scale, double *out, int nthreads)
{
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads > 0 ? nthreads : 1)
    for (int r = 0; r < n; ++r) {
        double *o = out + (size_t)r * d;
        for (int i = 0; i < d; ++i) o[i] = 0.0;
        oracle_swiglu_expert(d, f, X + (size_t)r * d, W1, W3, W2, scale ? scale[r] : 1.0, o);
    }
}

/*
 * Layer output of a list of tokens, token choice ([P2] §3.1 y = sum_i G_i E_i(x),
 * §3.4 and §9.1 shared experts added unweighted):
 *   y[t] = sum_{j : slot_of[t][j] >= 0} topk_w[t][j] * E_{topk_idx[t][j]}(x_t)
 *        + sum_s Shared_s(x_t)
 * taken in slot order j = 0..k-1, shared experts last.  A dropped slot adds
 * nothing (its residual belongs to the caller).  W1[e], W3[e], W2[e] point at
 * expert e's matrices (only experts the listed tokens use are read).
 */
int oracle_forward_tc(int d, int f, int k, int n_tok, const int32_t *tok, const float *x,
                      const int32_t *topk_idx, const double *topk_w, const int32_t *slot_of,
                      const float *const *W1, const float *const *W3, const float *const *W2,
                      int n_shared, int f_shared, const float *const *W1s,
                      const float *const *W3s, const float *const *W2s, double *y, int nthreads)
{
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads > 0 ? nthreads : 1)
    for (int n = 0; n < n_tok; ++n) {
        const int t = tok[n];
        const float *xt = x + (size_t)t * d;
        double *yt = y + (size_t)n * d;
        for (int r = 0; r < d; ++r) yt[r] = 0.0;
        for (int j = 0; j < k; ++j) {
            if (slot_of[(size_t)t * k + j] < 0) continue;
            const int e = topk_idx[(size_t)t * k + j];
            oracle_swiglu_expert(d, f, xt, W1[e], W3[e], W2[e], topk_w[(size_t)t * k + j], yt);
        }
        for (int s = 0; s < n_shared; ++s)
            oracle_swiglu_expert(d, f_shared, xt, W1s[s], W3s[s], W2s[s], 1.0, yt);
    }
    return 0;
}

/*
 * Layer output of a list of tokens, Expert Choice ([P2] §3.3): token t receives
 *   y[t] = sum over experts e (ascending) that took t of S[t][e] * E_e(x_t)
 *        + sum_s Shared_s(x_t);
 * a token no expert took gets only the shared part (zero without shared experts).
 */
int oracle_forward_ec(int d, int f, int E, int cap, int n_tok, const int32_t *tok,
                      const float *x, const int32_t *ec_tok, const double *ec_w,
                      const float *const *W1, const float *const *W3, const float *const *W2,
                      int n_shared, int f_shared, const float *const *W1s,
                      const float *const *W3s, const float *const *W2s, double *y, int nthreads)
{
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads > 0 ? nthreads : 1)
    for (int n = 0; n < n_tok; ++n) {
        const int t = tok[n];
        const float *xt = x + (size_t)t * d;
        double *yt = y + (size_t)n * d;
        for (int r = 0; r < d; ++r) yt[r] = 0.0;
        for (int e = 0; e < E; ++e) {
            for (int r = 0; r < cap; ++r) {
                if (ec_tok[(size_t)e * cap + r] != t) continue;
                oracle_swiglu_expert(d, f, xt, W1[e], W3[e], W2[e], ec_w[(size_t)e * cap + r], yt);
            }
        }
        for (int s = 0; s < n_shared; ++s)
            oracle_swiglu_expert(d, f_shared, xt, W1s[s], W3s[s], W2s[s], 1.0, yt);
    }
    return 0;
}

int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
