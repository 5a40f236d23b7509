/*
 * spd.h -- sparse paged decode attention for GB300 (sm_103a): the C ABI.
 *
 * The library computes the attention hot path of sparse rollouts over a paged
 * bf16 KV cache: per-page key summaries, query-aware page scoring with a
 * per-sequence page budget, attention over only the selected pages (split-K
 * with a log-sum-exp merge), and dense causal verification of k+1 drafted
 * positions over the whole cache.
 *
 * Sources.  Block-sparse (page) attention during rollouts with a KV budget and
 * a page size, and a Top-k over pages: the Sparrow project page, "Insights" and
 * "Control Study 2" (cost model; block size 16 and above; page size 16).  A
 * budget that grows with generation length: Sparrow, "Control Study 1"
 * (sparsity scheduling).  Sparse drafting of k = 6 tokens and dense
 * verification over the complete KV cache: the S3R abstract, Figure 6 and
 * Table 7.  The page score is a Quest-style upper bound from per-page,
 * per-channel key minima and maxima (Quest is in Sparrow's reference list;
 * the pages print no scoring rule of their own).
 *
 * Conventions shared by every call.
 *  - All tensor pointers are DEVICE pointers owned by the caller; the library
 *    never allocates, frees or synchronises (except spd_device_status).  Every
 *    call is asynchronous on `stream` (a cudaStream_t; NULL = legacy default).
 *  - bf16 values are passed as raw 16-bit patterns (spd_bf16).  K, V, q, the
 *    summaries and o must be 16-byte aligned; the KV cache base additionally
 *    must allow 16-byte row strides (D * 2 bytes, always true for D = 64, 128).
 *  - Paged KV cache: K and V are [num_phys_pages][H_kv][page_size][D] bf16, so
 *    one (physical page, KV head) tile is contiguous.  page_table is
 *    [B][max_pages_per_seq] int32 of physical page ids; seq_lens is [B] int32
 *    token counts (including the current token, or all T draft tokens).
 *    Sequence b uses logical pages 0 .. ceil(seq_lens[b] / page_size) - 1; the
 *    cache slots past seq_lens[b] in its last page are never used for a result
 *    (their contents may be anything, including NaN).
 *  - GQA: query head hq reads KV head hq / G, G = H_q / H_kv.
 *  - Softmax: logits z = softmax_scale * q.k; lse is the natural-log
 *    log-sum-exp of the scaled logits.  A row that sees no token gets o = 0,
 *    lse = -inf.
 *  - Workspace: `ws` is caller-owned device scratch of at least the size the
 *    matching *_workspace_size function returns.  The counters and flags some
 *    calls keep in it (unit queue, split tickets, the step's chain) MUST be
 *    zero before the first call that uses the buffer (zero the whole buffer
 *    once); every successful call leaves them zero again, so a buffer can be
 *    reused by any later call on the same stream.  Calls that overlap on the
 *    GPU must use different workspaces.
 *  - Errors: argument problems are reported synchronously by the returned
 *    status (nothing is launched); spd_last_error() gives a message.  Problems
 *    only the GPU can see (a page id outside [0, num_phys_pages), a selection
 *    entry out of range, a bounded wait that ran out) set bits in a device
 *    status word read by spd_device_status(); the affected rows are skipped or
 *    zeroed, and no kernel traps, asserts or spins without a bound.
 */
#ifndef SPD_H
#define SPD_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t spd_bf16; /* bfloat16 bit pattern */

typedef enum {
    SPD_OK = 0,
    SPD_ERR_INVALID_ARG = 1, /* null pointer, bad size, misaligned pointer, inconsistent shapes */
    SPD_ERR_UNSUPPORTED = 2, /* a shape outside the supported set (see spd_dims) */
    SPD_ERR_CUDA = 3,        /* a CUDA runtime or launch error; see spd_last_error() */
    SPD_ERR_WORKSPACE = 4    /* ws is NULL or ws_bytes is below the required size */
} spd_status;

/* Device status bits (spd_device_status). */
#define SPD_DEV_BAD_PAGE 0x1u  /* a page-table entry outside [0, num_phys_pages) */
#define SPD_DEV_BAD_SEL 0x2u   /* a selected page id outside the sequence, or nsel > k_max */
#define SPD_DEV_TIMEOUT 0x4u   /* a bounded wait on an asynchronous copy ran out */
#define SPD_DEV_BAD_LEN 0x8u   /* seq_lens[b] outside [0, max_pages_per_seq * page_size] (the row is
                                * then treated as empty: nothing selected, o = 0, lse = -inf), or
                                * too short for the tokens being appended */
#define SPD_DEV_BAD_TOKEN 0x10u /* spec_accept: a drafted token outside [0, n_vocab) */

/*
 * Problem shape.  Supported: D in {64, 128}; page_size in {16, 32, 64};
 * H_kv >= 1, H_q % H_kv == 0, G = H_q / H_kv <= 8; max_pages_per_seq >= 1;
 * num_phys_pages * H_kv * page_size < 2^31.  B = 0 is a valid no-op.
 */
typedef struct {
    int32_t B;                 /* sequences */
    int32_t H_q;               /* query heads */
    int32_t H_kv;              /* KV heads */
    int32_t D;                 /* head dimension */
    int32_t page_size;         /* tokens per page */
    int32_t max_pages_per_seq; /* row length of page_table */
    int64_t num_phys_pages;    /* pages in the K / V / summary arrays */
} spd_dims;

typedef enum {
    SPD_BUDGET_FIXED_PAGES = 0,   /* budget = fixed_pages */
    SPD_BUDGET_LINEAR_TOKENS = 1, /* ceil(max(min_tokens, ceil(len*slope_num/slope_den) + intercept) / page_size) */
    SPD_BUDGET_FRACTION = 2,      /* ceil(len * frac_num / (frac_den * page_size)) */
    SPD_BUDGET_TOP_P = 3          /* the smallest set holding top_p of the page weight (below) */
} spd_budget_mode;

/*
 * Per-sequence page budget (the sparsity schedule), evaluated on the device in
 * exact 64-bit integer arithmetic from len = seq_lens[b].  The first
 * sink_pages pages (the attention sink) and the last local_pages pages (the
 * local window) are always selected and count toward the budget.  The number
 * of pages selected for a (sequence, KV head) is
 *   k_eff = min(P, max(min(budget, k_max), |mandatory|)),  P = ceil(len / page_size).
 *
 * SPD_BUDGET_TOP_P makes the budget query-dependent (the pages stress that the
 * budget a query needs varies strongly: S3R abstract, Sparrow "Control Study
 * 1").  Each page gets the weight w(p) = exp(score_scale * (score(p) - max
 * score)), a softmax over pages of the bound logits; after the mandatory
 * pages, the best-scoring pages are added until the selected weight reaches
 * top_p of the total, at most k_max pages in all.  On the device the weights
 * are fp32 exponentials rounded to multiples of 2^-31 and summed as exact
 * integers, so the count is deterministic; it can differ from a real-number
 * evaluation only where the selected weight lands within that rounding of
 * the top_p share.
 */
typedef struct {
    int32_t mode; /* spd_budget_mode */
    int32_t fixed_pages;
    int64_t min_tokens, slope_num, slope_den, intercept; /* LINEAR_TOKENS (slope_den > 0) */
    int64_t frac_num, frac_den;                          /* FRACTION (frac_den > 0) */
    int32_t sink_pages, local_pages;                     /* >= 0 */
    float top_p;       /* TOP_P: share of the page weight to hold, in [0, 1] */
    float score_scale; /* TOP_P: logit scale of the scores (> 0), e.g. 1 / sqrt(D) */
} spd_budget_policy;

/* Library ABI version (major * 100 + minor). */
int32_t spd_version(void);

/* Message for the last non-OK status returned on this host thread ("" if none). */
const char *spd_last_error(void);

/*
 * Reads (and with clear != 0, resets) the device status word of the current
 * device.  Synchronises the device.  Returns SPD_ERR_CUDA if the read fails.
 */
spd_status spd_device_status(uint32_t *out, int32_t clear);

/*
 * Limit, in nanoseconds of the GPU's global timer, of every bounded wait in the
 * kernels launched after this call, from any host thread (2 s by default): an
 * mbarrier wait on an asynchronous copy, and in sparse_decode_step's chain a
 * selection waiting for its row's scores or an attention unit waiting for its
 * row's selection.  A wait that runs out sets SPD_DEV_TIMEOUT, the kernel
 * skips the rest of the affected rows and returns; the workspace of such a
 * call must be zeroed again before it is reused.  Graphs keep the limit they
 * were captured with.  ns = 0 is rejected (SPD_ERR_INVALID_ARG).
 */
spd_status spd_set_wait_limit_ns(uint64_t ns);
uint64_t spd_wait_limit_ns(void);

/* Workspace sizes in bytes (0 on invalid arguments; see spd_last_error). */
size_t spd_score_select_workspace_size(const spd_dims *dims);
size_t spd_sparse_decode_workspace_size(const spd_dims *dims, int32_t k_max, int32_t num_splits);
size_t spd_dense_verify_workspace_size(const spd_dims *dims, int32_t T, int32_t num_splits);

/*
 * pages_summarize -- per-page key summaries (Quest-style page metadata that the
 * scoring rule reads; the pages' cost model charges one scoring read per
 * generated page: Sparrow, "Control Study 2", scoring term).
 *
 * For each listed (sequence b, logical page p) and each KV head h, writes the
 * channel-wise minimum and maximum of the keys of the page's valid tokens
 * (positions < seq_lens[b]), phys = page_table[b][p]:
 *   summ[b][h][p][0][d] = min_t K[phys][h][t][d],  summ[b][h][p][1][d] = max_t ...
 * summ is bf16 [B][H_kv][max_pages_per_seq][2][D], sequence-major so that
 * scoring a (sequence, KV head) row reads one contiguous stream; bf16 min/max
 * is exact.  Sequences that share physical pages (the rollouts of one prompt
 * sharing its prefix pages) each keep their own copy of a shared page's
 * summary: the scoring reads each sharer's copy once per step either way, but
 * the copies cost memory (4 * D bytes per page and KV head per sharer) and a
 * rewritten shared page must be summarised again for every sharer (one
 * only_pages entry per (sequence, page) slot).
 * only_pages: NULL = every logical page of every sequence; otherwise n_only
 * entries, each b * max_pages_per_seq + p (a slot of page_table), e.g. the
 * page the newest token was written to.  Entries whose p is past the
 * sequence's last page are skipped.  Pages not listed are left untouched.
 */
spd_status pages_summarize(const spd_dims *dims, const spd_bf16 *K, const int32_t *page_table,
                           const int32_t *seq_lens, const int32_t *only_pages, int32_t n_only,
                           spd_bf16 *summ, void *stream);

/*
 * kv_append_refresh -- appends the T newest tokens of every sequence to the
 * paged cache and rewrites the summaries of the pages they land in, in one
 * kernel (the per-step cache update before scoring: one token per decode
 * step; after verification, the T drafted positions rewritten with the
 * target's keys and values).  KV pages: S3R Figure 1(c); the per-step scoring
 * read of the summaries: Sparrow, "Control Study 2".
 *
 * seq_lens[b] already counts the new tokens: token t (0 <= t < T) goes to
 * position pos = seq_lens[b] - T + t, i.e. slot pos % page_size of physical
 * page page_table[b][pos / page_size], for every KV head:
 *   K[phys][h][slot][:] = k_new[b][t][h][:],  V[...] = v_new[b][t][h][:]
 * (k_new, v_new bf16 [B][T][H_kv][D], copied bit for bit).  Every page that
 * receives a token gets summ[b][h][p] = min / max over all its valid tokens
 * after the write -- the same bits pages_summarize would write -- whatever
 * the summary held before.  Other pages and cache slots are untouched.
 * Supported: 1 <= T <= 4096.  A sequence with seq_lens[b] < T or
 * seq_lens[b] > max_pages_per_seq * page_size is skipped and sets
 * SPD_DEV_BAD_LEN; a page id outside [0, num_phys_pages) sets SPD_DEV_BAD_PAGE.
 * K, V, k_new, v_new and summ must be 16-byte aligned.  Sequences must not
 * share the physical pages they append to.
 */
spd_status kv_append_refresh(const spd_dims *dims, int32_t T, spd_bf16 *K, spd_bf16 *V,
                             const int32_t *page_table, const int32_t *seq_lens,
                             const spd_bf16 *k_new, const spd_bf16 *v_new, spd_bf16 *summ,
                             void *stream);

/*
 * pages_score_select -- query-aware page scoring plus budgeted top-k
 * (Sparrow, "Control Study 2": KV budget B, page size, Top-k over pages;
 * "Control Study 1": length-scheduled budget).
 *
 * q is bf16 [B][H_q][D] (the decode query); summ is the [B][H_kv][max_pages][2][D]
 * array pages_summarize maintains.  For every sequence b, KV head h and page
 * p < P_b, the score is
 *   score(p) = max_{g < G} sum_d max(q[b][hG+g][d] * kmin[d], q[b][hG+g][d] * kmax[d])
 * (an upper bound of q.k over the page's keys), accumulated in fp32 from the
 * bf16 summaries.  Then the mandatory pages plus the best-scoring remaining
 * pages (score descending, ties to the lower page id) up to k_eff are
 * selected and written in ascending page order:
 *   sel [B][H_kv][k_max] int32 logical page ids (entries past nsel untouched),
 *   nsel[B][H_kv] int32 = k_eff.
 * scores: optional fp32 [B][H_kv][max_pages_per_seq] output of the raw scores
 * (slots past P_b untouched); NULL keeps them in the workspace.
 * Requires k_max >= sink_pages + local_pages.
 */
spd_status pages_score_select(const spd_dims *dims, const spd_bf16 *q, const spd_bf16 *summ,
                              const int32_t *seq_lens,
                              const spd_budget_policy *policy, int32_t *sel, int32_t *nsel,
                              int32_t k_max, float *scores, void *ws, size_t ws_bytes,
                              void *stream);

/*
 * pages_append_score_select -- kv_append_refresh with T = 1 and
 * pages_score_select in one pass over the summaries: the warp that scores the
 * tile holding a row's last page first writes the step's token (position
 * seq_lens[b] - 1) into K and V, rebuilds that page's summary (stored to summ
 * and used for the score), then scores the tile.  Results (K, V, summ, sel,
 * nsel, scores) are bit-identical to kv_append_refresh(T = 1) followed by
 * pages_score_select; one kernel launch and one pass over the cache update
 * fewer.  k_new, v_new: bf16 [B][H_kv][D].  A sequence with seq_lens[b] = 0
 * sets SPD_DEV_BAD_LEN and is skipped; a page id outside [0, num_phys_pages)
 * sets SPD_DEV_BAD_PAGE.  Other arguments and errors as the two calls.
 */
spd_status pages_append_score_select(const spd_dims *dims, spd_bf16 *K, spd_bf16 *V,
                                     const int32_t *page_table, const int32_t *seq_lens,
                                     const spd_bf16 *k_new, const spd_bf16 *v_new, const spd_bf16 *q,
                                     spd_bf16 *summ, const spd_budget_policy *policy, int32_t *sel,
                                     int32_t *nsel, int32_t k_max, float *scores, void *ws,
                                     size_t ws_bytes, void *stream);

/*
 * sparse_decode_attn -- attention of the decode query over the selected pages
 * only (block-sparse page attention: Sparrow, "Insights" and "Control Study
 * 2"; the S3R sparse drafter of Table 7).
 *
 * For each sequence b and query head hq (KV head h = hq / G): exact softmax
 * attention over the valid tokens of pages sel[b][h][0 .. nsel[b][h]):
 *   o[b][hq][d] (bf16), lse[b][hq] (fp32, natural log; may be NULL).
 * num_splits: 0 = automatic; otherwise the selected list of each (b, h) is cut
 * into that many contiguous parts processed in parallel and merged with the
 * log-sum-exp rule of lse_merge.  The workspace must hold
 * spd_sparse_decode_workspace_size(dims, k_max, num_splits) bytes.
 */
spd_status sparse_decode_attn(const spd_dims *dims, const spd_bf16 *q, const spd_bf16 *K,
                              const spd_bf16 *V, const int32_t *page_table,
                              const int32_t *seq_lens, const int32_t *sel, const int32_t *nsel,
                              int32_t k_max, int32_t num_splits, float softmax_scale,
                              spd_bf16 *o, float *lse, void *ws, size_t ws_bytes, void *stream);

/*
 * sparse_decode_step -- one whole sparse decode step in one call: the step's
 * token appended (as kv_append_refresh with T = 1; skipped when k_new and
 * v_new are NULL), every page scored and the budgeted selection made (as
 * pages_score_select), and attention over the selected pages (as
 * sparse_decode_attn with automatic splits).  Results -- K, V, summ, sel,
 * nsel, o, lse -- are those of the separate calls.
 *
 * The three kernels are chained row by row instead of grid by grid: scoring
 * hands out its tiles in row order and counts the finished tiles of each row,
 * the selection of a row starts as soon as its count is complete, and the
 * attention units of a row (one, or several and a merge when there are few
 * rows) as soon as its selection is published (release / acquire flags in the
 * workspace; every wait is bounded and reports SPD_DEV_TIMEOUT).  The
 * workspace (spd_sparse_decode_step_workspace_size bytes) must be zero before
 * its first use and is left zero; calls that overlap on the GPU need separate
 * workspaces.  Errors as the separate calls.
 */
size_t spd_sparse_decode_step_workspace_size(const spd_dims *dims, int32_t k_max);
spd_status sparse_decode_step(const spd_dims *dims, spd_bf16 *K, spd_bf16 *V, const int32_t *page_table,
                              const int32_t *seq_lens, const spd_bf16 *k_new, const spd_bf16 *v_new,
                              const spd_bf16 *q, spd_bf16 *summ, const spd_budget_policy *policy,
                              int32_t *sel, int32_t *nsel, int32_t k_max, float softmax_scale,
                              spd_bf16 *o, float *lse, void *ws, size_t ws_bytes, void *stream);

/*
 * sparse_decode_attn_noalloc -- sparse_decode_attn for callers that cannot
 * allocate device memory.  It has no counterpart on the pages: it is the same
 * computation, with the same arguments and results as sparse_decode_attn,
 * minus the workspace.
 *
 * Who needs it: code that runs where a cudaMalloc is not allowed or not
 * wanted -- an inference engine that owns all device memory through a fixed
 * arena and gives plug-ins no workspace argument, or a latency-critical decode
 * loop that must not call cudaMalloc because it can synchronise the device
 * and stall every stream.  Such a caller still passes q, K, V, the page table,
 * the selection and the outputs; the scratch this call needs (the unit queue,
 * the split tickets and the split partials) lives in a fixed array compiled
 * into the library, SPD_NOALLOC_SCRATCH_BYTES (8 MiB) per GPU, which every GPU
 * that loads the library holds until the process exits.
 *
 * Behaviour: the first call on a device looks up that array's device address
 * (once per device, with that device current); make that first call before
 * any stream capture.  Each call clears the array's counters on `stream`
 * (cudaMemsetAsync) and never calls cudaMalloc, cudaFree or any allocating
 * library routine.  The split count is num_splits, or with num_splits = 0 the
 * automatic count lowered until the partials fit the array; if the requested
 * split count (or even one split) needs more scratch than the array holds, the
 * call returns SPD_ERR_UNSUPPORTED and launches nothing.  All calls share the
 * one array: calls that overlap on the GPU (different streams, or different
 * host threads without ordering) race and give wrong results.
 */
#define SPD_NOALLOC_SCRATCH_BYTES ((size_t)8 << 20)
spd_status sparse_decode_attn_noalloc(const spd_dims *dims, const spd_bf16 *q, const spd_bf16 *K,
                                      const spd_bf16 *V, const int32_t *page_table,
                                      const int32_t *seq_lens, const int32_t *sel,
                                      const int32_t *nsel, int32_t k_max, int32_t num_splits,
                                      float softmax_scale, spd_bf16 *o, float *lse, void *stream);

/*
 * dense_verify_attn -- dense causal verification of T drafted positions over
 * the complete KV cache (S3R abstract; Table 7 "Verify (TV)", k = 6 so T = 7).
 *
 * q is bf16 [B][T][H_q][D]; the drafted tokens' K/V are already the last T
 * tokens of each sequence.  Row t (absolute position seq_lens[b] - T + t)
 * attends over tokens 0 .. seq_lens[b] - T + t.  Outputs o bf16 [B][T][H_q][D]
 * and lse fp32 [B][T][H_q] (may be NULL).  T = 1 is dense decode attention.
 * Supported: 1 <= T and T * G <= 64.  num_splits: 0 = automatic.
 */
spd_status dense_verify_attn(const spd_dims *dims, int32_t T, const spd_bf16 *q,
                             const spd_bf16 *K, const spd_bf16 *V, const int32_t *page_table,
                             const int32_t *seq_lens, int32_t num_splits, float softmax_scale,
                             spd_bf16 *o, float *lse, void *ws, size_t ws_bytes, void *stream);

/*
 * spec_accept -- exact speculative sampling over k drafted tokens per sequence
 * (S3R abstract: responses come from full-attention verification and exact
 * speculative sampling, so they follow the dense policy; k = 6 in Table 7).
 *
 * p_draft fp32 [B][k][n_vocab]: the drafter's distribution at each drafted
 * position; q_target fp32 [B][k+1][n_vocab]: the target's distribution at the
 * same positions plus the one after the last draft (from dense_verify_attn's
 * pass); draft int32 [B][k]; u_acc fp32 [B][k] and u_res fp32 [B]: uniform
 * numbers in [0, 1) drawn by the caller.  Rows need not be normalised.
 * For each sequence: draft x at position i is accepted iff
 * u_acc[b][i] * p_i(x) < q_i(x) (product formed exactly in fp64), in order,
 * until the first rejection j.  The emitted token is a draw from integer
 * weights on a 2^-40 grid, W(x) = max(0, F(q_j(x)) - F(p_j(x))) with
 * F(v) = floor(2^40 * min(v, 1)) (0 for v <= 0 or NaN), or W(x) = F(q_j(x))
 * when that residual is zero everywhere; after k acceptances W(x) = F(q_k(x))
 * (the bonus token).  The draw is the smallest x whose running sum of W
 * exceeds floor(u_res[b] * sum(W)); all sums are exact integers, so the
 * result does not depend on summation order.  W zero everywhere: -1.  (Mass
 * below 2^-40 per token is never drawn: at most n_vocab * 2^-40 of total
 * variation from the real-number rule.)
 * Outputs: n_accepted int32 [B]; tokens int32 [B][k+1] = the accepted drafts,
 * the emitted token, then -1.  A draft outside [0, n_vocab) at or before the
 * first rejection sets SPD_DEV_BAD_TOKEN and gives that sequence
 * n_accepted = 0, tokens = -1.
 * Supported: 1 <= k <= 32, 1 <= n_vocab <= 2^21; p_draft and q_target 16-byte
 * aligned.
 */
spd_status spec_accept(int32_t B, int32_t k, int32_t n_vocab, const float *p_draft,
                       const float *q_target, const int32_t *draft, const float *u_acc,
                       const float *u_res, int32_t *n_accepted, int32_t *tokens, void *stream);

/*
 * lse_merge -- combine S partial attention results computed over disjoint
 * token sets (split-K FlashDecoding):
 *   lse = log sum_s exp(part_lse[s]),  o = sum_s exp(part_lse[s] - lse) * part_o[s].
 * part_o fp32 [S][rows][D] (each partial already normalised), part_lse fp32
 * [S][rows] (natural log; -inf marks an empty partial).  Writes o bf16
 * [rows][D] and lse fp32 [rows] (lse may be NULL).  All partials empty:
 * o = 0, lse = -inf.  Supported: S >= 1, D in {64, 128}.
 */
spd_status lse_merge(int32_t S, int32_t rows, int32_t D, const float *part_o,
                     const float *part_lse, spd_bf16 *o, float *lse, void *stream);

/*
 * spd_round -- one S3R round captured as CUDA graphs: k sparse draft steps,
 * then dense verification of the k + 1 positions and exact speculative
 * sampling, replayed with one graph launch per part (S3R Table 7: drafting
 * runs under CUDA Graphs; "Draft (6Tq)" and "Verify (TV)" are its two parts).
 *
 * Draft step s (0 <= s < k), on lengths seq_lens[s][:] (which count the token
 * the step appends):
 *   kv_append_refresh(T = 1, k_draft[s], v_draft[s]);
 *   pages_score_select(q_draft[s]) into sel / nsel (reused by every step);
 *   sparse_decode_attn(q_draft[s]) -> o_draft[s], lse_draft[s].
 * Verification, on lengths seq_lens[k][:]:
 *   kv_append_refresh(T = k + 1, k_verify, v_verify)   (rewrites the positions);
 *   dense_verify_attn(T = k + 1, q_verify) -> o_verify, lse_verify;
 *   spec_accept(...) -> n_accepted, tokens            (skipped when n_vocab = 0).
 * Layouts: seq_lens int32 [k + 1][B]; q_draft bf16 [k][B][H_q][D]; k_draft,
 * v_draft bf16 [k][B][H_kv][D]; q_verify bf16 [B][k+1][H_q][D]; k_verify,
 * v_verify bf16 [B][k+1][H_kv][D]; o_draft [k][B][H_q][D]; lse_draft
 * [k][B][H_q] (may be NULL); o_verify / lse_verify as dense_verify_attn; the
 * sampling buffers as spec_accept.  The three workspaces are sized by the
 * matching *_workspace_size calls; the split counts and softmax_scale mean
 * what they mean in those calls.
 *
 * spd_round_create validates the descriptor, makes each call once on a
 * private stream under capture (so every argument error surfaces here, with
 * nothing launched) and instantiates the graphs; the buffers must stay valid
 * and keep their addresses for the life of the round.  spd_round_launch
 * replays part 0 (draft steps), 1 (verification) or 2 (both, in order) on
 * `stream`; replaying is the same computation as making the calls.  Make one
 * ordinary call of the library on the device before the first create.
 */
typedef struct {
    spd_dims dims;
    int32_t k; /* draft steps per round, 1 <= k <= 32 */
    spd_bf16 *K, *V, *summ;
    const int32_t *page_table;
    const int32_t *seq_lens;
    const spd_bf16 *q_draft, *k_draft, *v_draft;
    const spd_bf16 *q_verify, *k_verify, *v_verify;
    spd_budget_policy policy;
    int32_t k_max;
    int32_t *sel, *nsel;
    spd_bf16 *o_draft;
    float *lse_draft;
    spd_bf16 *o_verify;
    float *lse_verify;
    int32_t n_vocab;
    const float *p_draft, *q_target;
    const int32_t *draft_tokens;
    const float *u_acc, *u_res;
    int32_t *n_accepted, *tokens;
    void *ws_select;
    size_t ws_select_bytes;
    void *ws_sparse;
    size_t ws_sparse_bytes;
    void *ws_verify;
    size_t ws_verify_bytes;
    int32_t sparse_splits, verify_splits;
    float softmax_scale;
} spd_round_desc;

typedef struct spd_round_s spd_round;

spd_status spd_round_create(const spd_round_desc *desc, spd_round **out);
spd_status spd_round_launch(spd_round *round, int32_t part, void *stream);
void spd_round_destroy(spd_round *round);

#ifdef __cplusplus
}
#endif

#endif /* SPD_H */
