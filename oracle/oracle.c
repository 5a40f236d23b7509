/*
 * oracle.c -- plain, slow, fp64 CPU oracle for sparse paged decode attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the library's product path may call,
 * link or load this file; only the tests, the smoke check and the benchmark's
 * CPU-baseline leg use it.  It shares no code, header, helper or constant with
 * the CUDA path.
 *
 * Every function works on one sequence b and writes only that sequence's
 * outputs, so callers may run sequences on separate threads.  All arithmetic is
 * IEEE double; bf16 inputs (raw uint16 bit patterns) are widened exactly.
 *
 * Sources (the "Sparrow" project page and the "S3R" appendix pages):
 *  - block-sparse (page) attention over the KV cache during rollouts:
 *    Sparrow, "Insights" section (block-sparse attention is the studied form)
 *    and "Control Study 2" (block size 16 and above; cost model with a KV
 *    budget B and a page size, and a Top-k over pages);
 *  - the budget grows with generation length ("sparsity scheduling"):
 *    Sparrow, "Control Study 1";
 *  - dense verification of drafted tokens over the complete KV cache, k = 6:
 *    S3R abstract, Figure 6 and Table 7 ("Draft (6Tq)", "Verify (TV)").
 * The pages print no scoring rule; the page score is the Quest-style upper
 * bound from per-page, per-channel key minima and maxima (Quest appears in
 * Sparrow's reference list).  Where the pages are silent the readings are:
 *  - GQA: query head hq reads KV head hq / G; a KV head's page score is the
 *    maximum over its G query heads of the per-head bound;
 *  - selection is per (sequence, KV head); mandatory pages = the first
 *    sink_pages pages and the last local_pages pages; they count toward the
 *    budget; effective k = min(P, max(min(budget, k_max), |mandatory|));
 *  - the rest are ranked by score descending, ties to the lower page id, and
 *    the selected list is emitted in ascending page order;
 *  - softmax scale is passed in (1/sqrt(D) by the callers); lse uses the
 *    natural log; a row with no visible token has o = 0 and lse = -inf;
 *  - verify row t (absolute position len - T + t) sees tokens 0..len-T+t.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Exact widening of a bfloat16 bit pattern. */
static double widen(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static int pages_of(int len, int ps) { return (len + ps - 1) / ps; }

/* K or V element (phys page, kv head, token in page, channel). */
static double kv_at(const uint16_t *X, int H_kv, int ps, int D, long phys, int h, int t, int d)
{
    return widen(X[(((size_t)phys * H_kv + h) * ps + t) * D + d]);
}

/*
 * Step a1 -- per-page key summaries.  For every logical page of sequence b and
 * every KV head: the channel-wise minimum and maximum of the keys of the valid
 * tokens of that page (tokens at positions < len_b).  Written at the page's
 * physical slot: summ[phys][h][0][d] = min, summ[phys][h][1][d] = max.
 */
void oracle_summarize_seq(int H_kv, int D, int ps, int max_pages, const uint16_t *K,
                          const int32_t *page_table, const int32_t *seq_lens, int b,
                          double *summ)
{
    int len = seq_lens[b];
    int P = pages_of(len, ps);
    for (int p = 0; p < P; ++p) {
        long phys = page_table[(size_t)b * max_pages + p];
        int valid = len - p * ps;
        if (valid > ps) valid = ps;
        for (int h = 0; h < H_kv; ++h) {
            double *mn = summ + ((size_t)phys * H_kv + h) * 2 * D;
            double *mx = mn + D;
            for (int d = 0; d < D; ++d) {
                double lo = INFINITY, hi = -INFINITY;
                for (int t = 0; t < valid; ++t) {
                    double k = kv_at(K, H_kv, ps, D, phys, h, t, d);
                    if (k < lo) lo = k;
                    if (k > hi) hi = k;
                }
                mn[d] = lo;
                mx[d] = hi;
            }
        }
    }
}

/*
 * Step a2 -- page scores.  For query head hq and page p with summaries
 * (kmin, kmax): UB_hq(p) = sum_d max(q_d * kmin_d, q_d * kmax_d), which bounds
 * q . k from above for every key k of the page.  The KV head's score is the
 * maximum of UB over its G query heads.  scores[h][p] for p < P_b.
 */
void oracle_score_seq(int H_q, int H_kv, int D, int ps, int max_pages, const uint16_t *q,
                      const double *summ, const int32_t *page_table, const int32_t *seq_lens,
                      int b, double *scores)
{
    int G = H_q / H_kv;
    int P = pages_of(seq_lens[b], ps);
    for (int h = 0; h < H_kv; ++h) {
        for (int p = 0; p < P; ++p) {
            long phys = page_table[(size_t)b * max_pages + p];
            const double *mn = summ + ((size_t)phys * H_kv + h) * 2 * D;
            const double *mx = mn + D;
            double best = -INFINITY;
            for (int g = 0; g < G; ++g) {
                int hq = h * G + g;
                double ub = 0.0;
                for (int d = 0; d < D; ++d) {
                    double qd = widen(q[((size_t)b * H_q + hq) * D + d]);
                    double a = qd * mn[d], c = qd * mx[d];
                    ub += (a > c) ? a : c;
                }
                if (ub > best) best = ub;
            }
            scores[(size_t)h * max_pages + p] = best;
        }
    }
}

/*
 * Step a3 -- per-sequence budget in pages (the sparsity schedule: a budget
 * that grows with the sequence length).  Integer arithmetic only.
 *   mode 0 (fixed):    a pages
 *   mode 1 (linear):   ceil(max(a, ceil(len * b / c) + d) / ps)   [tokens: a = floor, b/c = slope, d = intercept]
 *   mode 2 (fraction): ceil(len * a / (b * ps))
 */
long oracle_budget_pages(int mode, long a, long b, long c, long d, int len, int ps)
{
    if (mode == 0) return a;
    if (mode == 1) {
        long lin = ((long)len * b + c - 1) / c + d;
        long tok = lin > a ? lin : a;
        return (tok + ps - 1) / ps;
    }
    return ((long)len * a + b * ps - 1) / (b * ps);
}

static int is_mandatory(int p, int P, int sink, int local)
{
    return p < sink || p >= P - local;
}

/* Number of pages the selection holds: min(P, max(min(budget, k_max), |mandatory|)). */
int oracle_k_eff(int P, long budget, int k_max, int sink, int local)
{
    int nm = 0;
    for (int p = 0; p < P; ++p) nm += is_mandatory(p, P, sink, local);
    long k = budget < k_max ? budget : k_max;
    if (k < nm) k = nm;
    if (k > P) k = P;
    return (int)k;
}

typedef struct {
    double s;
    int p;
} ranked;

static int by_score_then_id(const void *x, const void *y)
{
    const ranked *a = (const ranked *)x, *b = (const ranked *)y;
    if (a->s > b->s) return -1;
    if (a->s < b->s) return 1;
    return (a->p > b->p) - (a->p < b->p);
}

static int ascending(const void *x, const void *y)
{
    int a = *(const int *)x, b = *(const int *)y;
    return (a > b) - (a < b);
}

/*
 * Step a4 -- top-k page selection for every KV head of sequence b.  The
 * mandatory pages are taken first; the remaining pages are sorted by score
 * (descending; equal scores: lower page id first) and the first
 * k_eff - |mandatory| are added.  The list is written in ascending page order:
 * sel[h][0..nsel[h]).
 */
void oracle_select_seq(int H_kv, int ps, int max_pages, const double *scores, int len, int mode,
                       long a, long b, long c, long d, int sink, int local, int k_max,
                       int32_t *sel, int32_t *nsel)
{
    int P = pages_of(len, ps);
    long budget = oracle_budget_pages(mode, a, b, c, d, len, ps);
    int k = oracle_k_eff(P, budget, k_max, sink, local);
    ranked *cand = (ranked *)malloc(sizeof(ranked) * (P > 0 ? P : 1));
    int *pick = (int *)malloc(sizeof(int) * (P > 0 ? P : 1));
    for (int h = 0; h < H_kv; ++h) {
        int n = 0, nc = 0;
        for (int p = 0; p < P; ++p) {
            if (is_mandatory(p, P, sink, local))
                pick[n++] = p;
            else {
                cand[nc].s = scores[(size_t)h * max_pages + p];
                cand[nc].p = p;
                ++nc;
            }
        }
        qsort(cand, nc, sizeof(ranked), by_score_then_id);
        for (int i = 0; n < k && i < nc; ++i) pick[n++] = cand[i].p;
        qsort(pick, n, sizeof(int), ascending);
        for (int i = 0; i < n; ++i) sel[(size_t)h * k_max + i] = pick[i];
        nsel[h] = n;
    }
    free(cand);
    free(pick);
}

/*
 * Exact softmax attention of one query row over an explicit token list:
 * z_j = scale * q . k_j;  o = sum_j e^{z_j - m} v_j / sum_j e^{z_j - m};
 * lse = m + log(sum_j e^{z_j - m}), m = max_j z_j.  No tokens: o = 0, lse = -inf.
 */
static void attend_row(int H_kv, int ps, int D, const uint16_t *qrow, const uint16_t *K,
                       const uint16_t *V, int h, const long *tok_phys, const int *tok_slot, int n,
                       double scale, double *z, double *o, double *lse)
{
    for (int d = 0; d < D; ++d) o[d] = 0.0;
    if (n == 0) {
        *lse = -INFINITY;
        return;
    }
    double m = -INFINITY;
    for (int j = 0; j < n; ++j) {
        double acc = 0.0;
        for (int d = 0; d < D; ++d)
            acc += widen(qrow[d]) * kv_at(K, H_kv, ps, D, tok_phys[j], h, tok_slot[j], d);
        z[j] = scale * acc;
        if (z[j] > m) m = z[j];
    }
    double l = 0.0;
    for (int j = 0; j < n; ++j) {
        double w = exp(z[j] - m);
        l += w;
        for (int d = 0; d < D; ++d) o[d] += w * kv_at(V, H_kv, ps, D, tok_phys[j], h, tok_slot[j], d);
    }
    for (int d = 0; d < D; ++d) o[d] /= l;
    *lse = m + log(l);
}

/*
 * Step a5 -- sparse attention for sequence b: every query head attends,
 * exactly, over the valid tokens (position < len_b) of the pages its KV head
 * selected, sel[h][0..nsel[h]) (logical page ids).  o[hq][d], lse[hq].
 */
void oracle_sparse_attn_seq(int H_q, int H_kv, int D, int ps, int max_pages, const uint16_t *q,
                            const uint16_t *K, const uint16_t *V, const int32_t *page_table,
                            const int32_t *seq_lens, int b, const int32_t *sel,
                            const int32_t *nsel, int k_max, double scale, double *o, double *lse)
{
    int G = H_q / H_kv;
    int len = seq_lens[b];
    long *tp = (long *)malloc(sizeof(long) * ((size_t)k_max * ps + 1));
    int *ts = (int *)malloc(sizeof(int) * ((size_t)k_max * ps + 1));
    double *z = (double *)malloc(sizeof(double) * ((size_t)k_max * ps + 1));
    for (int h = 0; h < H_kv; ++h) {
        int n = 0;
        for (int i = 0; i < nsel[h]; ++i) {
            int p = sel[(size_t)h * k_max + i];
            long phys = page_table[(size_t)b * max_pages + p];
            for (int t = 0; t < ps && p * ps + t < len; ++t) {
                tp[n] = phys;
                ts[n] = t;
                ++n;
            }
        }
        for (int g = 0; g < G; ++g) {
            int hq = h * G + g;
            attend_row(H_kv, ps, D, q + ((size_t)b * H_q + hq) * D, K, V, h, tp, ts, n, scale, z,
                       o + (size_t)hq * D, lse + hq);
        }
    }
    free(tp);
    free(ts);
    free(z);
}

/*
 * Step a6 -- merge of S partial results of one row computed over disjoint
 * token sets: lse = log sum_s e^{lse_s}; o = sum_s e^{lse_s - lse} o_s.
 * Partials with lse_s = -inf contribute nothing; all empty: o = 0, lse = -inf.
 */
void oracle_merge_row(int S, int D, const double *part_o, const double *part_lse, double *o,
                      double *lse)
{
    double m = -INFINITY;
    for (int s = 0; s < S; ++s)
        if (part_lse[s] > m) m = part_lse[s];
    for (int d = 0; d < D; ++d) o[d] = 0.0;
    if (m == -INFINITY) {
        *lse = -INFINITY;
        return;
    }
    double l = 0.0;
    for (int s = 0; s < S; ++s)
        if (part_lse[s] != -INFINITY) l += exp(part_lse[s] - m);
    double L = m + log(l);
    for (int s = 0; s < S; ++s) {
        if (part_lse[s] == -INFINITY) continue;
        double w = exp(part_lse[s] - L);
        for (int d = 0; d < D; ++d) o[d] += w * part_o[(size_t)s * D + d];
    }
    *lse = L;
}

/*
 * Step a7 -- dense verification for sequence b: T query positions whose keys
 * and values are already the last T tokens of the cache.  Row t (absolute
 * position len_b - T + t) of query head hq attends over every token at
 * positions 0..len_b - T + t.  q is [B][T][H_q][D]; o[t][hq][d], lse[t][hq].
 * With T = 1 this is dense decode attention over the whole cache.
 */
void oracle_verify_seq(int T, int H_q, int H_kv, int D, int ps, int max_pages, const uint16_t *q,
                       const uint16_t *K, const uint16_t *V, const int32_t *page_table,
                       const int32_t *seq_lens, int b, double scale, double *o, double *lse)
{
    int G = H_q / H_kv;
    int len = seq_lens[b];
    long *tp = (long *)malloc(sizeof(long) * ((size_t)len + 1));
    int *ts = (int *)malloc(sizeof(int) * ((size_t)len + 1));
    double *z = (double *)malloc(sizeof(double) * ((size_t)len + 1));
    for (int j = 0; j < len; ++j) {
        tp[j] = page_table[(size_t)b * max_pages + j / ps];
        ts[j] = j % ps;
    }
    for (int t = 0; t < T; ++t) {
        int visible = len - T + t + 1;
        if (visible < 0) visible = 0;
        for (int hq = 0; hq < H_q; ++hq) {
            int h = hq / G;
            attend_row(H_kv, ps, D, q + (((size_t)b * T + t) * H_q + hq) * D, K, V, h, tp, ts,
                       visible, scale, z, o + ((size_t)t * H_q + hq) * D, lse + (size_t)t * H_q + hq);
        }
    }
    free(tp);
    free(ts);
    free(z);
}

/*
 * Row f1 -- appending tokens to the paged cache.  The T newest tokens of
 * sequence b take the positions len_b - T .. len_b - 1 (len_b already counts
 * them): position pos lives in logical page pos / ps, slot pos % ps, of the
 * physical page page_table[b][pos / ps].  k_new and v_new are [B][T][H_kv][D]
 * bf16 bit patterns, copied bit for bit into K and V.  The summaries of the
 * pages this touches are then, by definition, oracle_summarize_seq over the
 * updated cache.  Positions below 0 (len_b < T) are not written.
 */
void oracle_append_seq(int T, int H_kv, int D, int ps, int max_pages, uint16_t *K, uint16_t *V,
                       const int32_t *page_table, const int32_t *seq_lens, int b,
                       const uint16_t *k_new, const uint16_t *v_new)
{
    int len = seq_lens[b];
    for (int t = 0; t < T; ++t) {
        int pos = len - T + t;
        if (pos < 0) continue;
        long phys = page_table[(size_t)b * max_pages + pos / ps];
        for (int h = 0; h < H_kv; ++h) {
            size_t src = (((size_t)b * T + t) * H_kv + h) * D;
            size_t dst = (((size_t)phys * H_kv + h) * ps + pos % ps) * D;
            for (int d = 0; d < D; ++d) {
                K[dst + d] = k_new[src + d];
                V[dst + d] = v_new[src + d];
            }
        }
    }
}

/*
 * A draw with a uniform u in [0, 1) from non-negative weights w[0..n): the
 * smallest x whose running sum (in index order) exceeds u * sum(w) -- inverting
 * the cumulative distribution.  The last running sum is the total itself (the
 * same additions in the same order), which exceeds u * total for u < 1.  All
 * weights zero: -1.
 */
static int draw(const double *w, int n, double u)
{
    double total = 0.0;
    for (int x = 0; x < n; ++x) total += w[x];
    if (!(total > 0.0)) return -1;
    double t = u * total, run = 0.0;
    for (int x = 0; x < n; ++x) {
        run += w[x];
        if (run > t) return x;
    }
    return -1; /* not reached */
}

/* A probability as a weight: negative and NaN values weigh nothing. */
static double weight(double v) { return v > 0.0 ? v : 0.0; }

/*
 * Row f2 -- exact speculative sampling (the S3R abstract: responses come from
 * full-attention verification followed by exact speculative sampling, so they
 * follow the dense policy).  The rule is the standard one for a drafter
 * distribution p and a target distribution q over a vocabulary of n tokens:
 *   for i = 0 .. k-1, with x = draft[i]: accept iff u_acc[i] * p_i(x) < q_i(x)
 *   (accept with probability min(1, q_i(x) / p_i(x))), the product of the two
 *   floats formed exactly in double;
 *   at the first rejection j, emit a draw (u_res) from the residual
 *   max(0, q_j - p_j), or from q_j when the residual is zero everywhere;
 *   if all k drafts are accepted, emit a bonus draw (u_res) from q_k.
 * The draws are plain inverse-CDF draws in double precision.
 * p is [k][n] and q is [k+1][n] fp32.  tokens[0..k] receives the accepted
 * drafts then the emitted token, -1 after it; the return value is the number
 * of accepted drafts.
 */
int oracle_spec_accept_seq(int k, int n, const float *p, const float *q, const int32_t *draft,
                           const float *u_acc, float u_res, int32_t *tokens)
{
    int acc = 0;
    while (acc < k) {
        int x = draft[acc];
        double px = p[(size_t)acc * n + x], qx = q[(size_t)acc * n + x];
        if (!((double)u_acc[acc] * px < qx)) break;
        tokens[acc] = x;
        ++acc;
    }
    double *w = (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
    const float *qr = q + (size_t)acc * n;
    int tok = -1;
    if (acc < k) {
        const float *pr = p + (size_t)acc * n;
        for (int x = 0; x < n; ++x) w[x] = weight((double)qr[x] - (double)pr[x]);
        tok = draw(w, n, (double)u_res);
    }
    if (tok < 0) {
        for (int x = 0; x < n; ++x) w[x] = weight((double)qr[x]);
        tok = draw(w, n, (double)u_res);
    }
    free(w);
    tokens[acc] = tok;
    for (int i = acc + 1; i <= k; ++i) tokens[i] = -1;
    return acc;
}

/*
 * Row f3 -- query-dependent (top-p) page selection for every KV head of
 * sequence b: instead of a fixed number of pages, the smallest set whose
 * share of the page weight reaches top_p.  A page's weight is
 * w(p) = exp(score_scale * (score(p) - max_p' score(p'))) over the P_b
 * pages (the score is an upper bound of q.k, so w is a softmax over pages of
 * the bound logits).  The mandatory pages are taken first; then the
 * remaining pages in score order (descending; equal scores: lower id first)
 * while the selected weight is below top_p * sum_p w(p) and fewer than k_max
 * pages are held.  The list is written in ascending page order.
 */
void oracle_select_top_p_seq(int H_kv, int ps, int max_pages, const double *scores, int len,
                             double top_p, double score_scale, int sink, int local, int k_max,
                             int32_t *sel, int32_t *nsel)
{
    int P = pages_of(len, ps);
    ranked *cand = (ranked *)malloc(sizeof(ranked) * (P > 0 ? P : 1));
    int *pick = (int *)malloc(sizeof(int) * (P > 0 ? P : 1));
    for (int h = 0; h < H_kv; ++h) {
        const double *s = scores + (size_t)h * max_pages;
        double smax = -INFINITY;
        for (int p = 0; p < P; ++p)
            if (s[p] > smax) smax = s[p];
        double total = 0.0;
        for (int p = 0; p < P; ++p) total += exp(score_scale * (s[p] - smax));
        double need = top_p * total, held = 0.0;
        int n = 0, nc = 0;
        for (int p = 0; p < P; ++p) {
            if (is_mandatory(p, P, sink, local)) {
                pick[n++] = p;
                held += exp(score_scale * (s[p] - smax));
            } else {
                cand[nc].s = s[p];
                cand[nc].p = p;
                ++nc;
            }
        }
        qsort(cand, nc, sizeof(ranked), by_score_then_id);
        for (int i = 0; i < nc && held < need && n < k_max; ++i) {
            pick[n++] = cand[i].p;
            held += exp(score_scale * (cand[i].s - smax));
        }
        qsort(pick, n, sizeof(int), ascending);
        for (int i = 0; i < n; ++i) sel[(size_t)h * k_max + i] = pick[i];
        nsel[h] = n;
    }
    free(cand);
    free(pick);
}
