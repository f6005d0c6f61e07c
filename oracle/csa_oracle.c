/*
 * CSA forward-path oracle: plain, slow, fp64 CPU code.
 *
 * TEST INFRASTRUCTURE ONLY. Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this library. The product path
 * (the CUDA library and its Python binding) never calls it, and the two
 * share no code: no headers, helpers, tables or constants.
 *
 * What it computes, step by step, in the order the pages describe it:
 *   - compressed cu_seqlens (per-segment floor(len / cmp_ratio));
 *   - the segment-clamped sliding window of original-KV rows;
 *   - lightning-indexer scores over the causally visible compressed blocks
 *     of the token's own segment, and their top-k;
 *   - shared-KV MLA attention over window rows plus selected compressed
 *     rows, with a per-head attention sink;
 *   - its backward: gradients of q, of both KV streams and of the sinks,
 *     and the head-averaged attention distributions;
 *   - the indexer's KL loss against that distribution, and its gradients;
 *   - the THD compressor's grouping, overlap transform and slot pooling.
 * Every floating-point input arrives as double (bf16 inputs are widened
 * exactly by the caller); every sum, exp and log is done in double.
 *
 * Index convention: all row indices are stream-absolute (rows of the packed
 * stream, not per-sample rows), as in the miles PR 2038 report, review notes
 * ("top-k indices become stream-absolute" under THD).
 *
 * Parity pins: every function here is pinned by the not-gpu tests against
 * closed forms, worked values, brute force and an independent NumPy dense
 * oracle (see tests/test_oracle_*.py). Nothing here is "parity unpinned".
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define REF_OK 0
#define REF_ERR_ARG 1
#define REF_ERR_NOMEM 2

int csa_ref_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Threads of the parallel loops from now on (n < 1: one per processor). */
void csa_ref_set_num_threads(int n) {
#ifdef _OPENMP
    omp_set_num_threads(n > 0 ? n : omp_get_num_procs());
#else
    (void)n;
#endif
}

/* cu_seqlens must start at 0 and never decrease. */
static int check_cu(const int32_t *cu, int32_t batch, int64_t total) {
    if (!cu || batch < 0) return 0;
    if (cu[0] != 0) return 0;
    for (int32_t b = 0; b < batch; ++b)
        if (cu[b + 1] < cu[b]) return 0;
    if (total >= 0 && cu[batch] != total) return 0;
    return 1;
}

/* The segment that owns packed row t: the b with cu[b] <= t < cu[b+1]. */
static int32_t segment_of(const int32_t *cu, int32_t batch, int32_t t) {
    for (int32_t b = 0; b < batch; ++b)
        if (t >= cu[b] && t < cu[b + 1]) return b;
    return -1;
}

/*
 * Compressed cu_seqlens.
 * miles PR 2038 report, compressor.py _forward_thd docstring: the last
 * len % cmp_ratio tokens of a segment produce no compressed entry; and
 * "风险与影响" (risks), item 2, the same tail rule. A segment of length L
 * therefore owns floor(L / cmp_ratio) compressed rows, and the compressed
 * stream is packed segment after segment like the original one.
 */
int csa_ref_compress_cu_seqlens(const int32_t *cu_seqlens, int32_t batch, int32_t cmp_ratio,
                                int32_t *cu_seqlens_cmp) {
    if (!cu_seqlens || !cu_seqlens_cmp || batch < 0 || cmp_ratio < 1) return REF_ERR_ARG;
    if (!check_cu(cu_seqlens, batch, -1)) return REF_ERR_ARG;
    cu_seqlens_cmp[0] = 0;
    for (int32_t b = 0; b < batch; ++b) {
        int32_t len = cu_seqlens[b + 1] - cu_seqlens[b];
        cu_seqlens_cmp[b + 1] = cu_seqlens_cmp[b] + len / cmp_ratio;
    }
    return REF_OK;
}

/*
 * Sliding-window rows of the original KV.
 * miles PR 2038 report, thd_utils.py get_window_topk_idxs_thd: the window of
 * a token holds the window_size most recent rows of its own segment, self
 * included; it is clamped to the segment start (not to stream row 0, the
 * bug the report's motivation section lists first). Output [T, W] with the
 * rows in ascending order from the clamped start, and -1 in every slot that
 * would lie after the token itself.
 * W = ori_win_left + 1 (the sparse_flash_mla schema of the hyper-parallel
 * RFC, section 2, has ori_win_left=127, ori_win_right=0: 127 rows to the left
 * plus the token itself).
 */
static void window_row(const int32_t *cu_seqlens, int32_t batch, int32_t t, int32_t W,
                       int32_t *row_out) {
    int32_t b = segment_of(cu_seqlens, batch, t);
    int32_t seg_start = cu_seqlens[b];
    int32_t start = t - W + 1;
    if (start < seg_start) start = seg_start;
    for (int32_t i = 0; i < W; ++i) {
        int32_t row = start + i;
        row_out[i] = (row > t) ? -1 : row;
    }
}

int csa_ref_window_idx(const int32_t *cu_seqlens, int32_t batch, int32_t total_tokens,
                       int32_t ori_win_left, int32_t *idx) {
    if (!cu_seqlens || !idx || batch < 0 || total_tokens < 0 || ori_win_left < 0) return REF_ERR_ARG;
    if (!check_cu(cu_seqlens, batch, total_tokens)) return REF_ERR_ARG;
    const int32_t W = ori_win_left + 1;
    for (int32_t t = 0; t < total_tokens; ++t) window_row(cu_seqlens, batch, t, W, idx + (int64_t)t * W);
    return REF_OK;
}

/* The same rows for the listed tokens only: row i of idx for tokens[i]. */
int csa_ref_window_idx_tokens(const int32_t *cu_seqlens, int32_t batch, int32_t total_tokens,
                              int32_t ori_win_left, const int32_t *tokens, int32_t n_tokens,
                              int32_t *idx) {
    if (!cu_seqlens || !idx || !tokens || batch < 0 || total_tokens < 0 || ori_win_left < 0 ||
        n_tokens < 0)
        return REF_ERR_ARG;
    if (!check_cu(cu_seqlens, batch, total_tokens)) return REF_ERR_ARG;
    const int32_t W = ori_win_left + 1;
    for (int32_t i = 0; i < n_tokens; ++i) {
        if (tokens[i] < 0 || tokens[i] >= total_tokens) return REF_ERR_ARG;
        window_row(cu_seqlens, batch, tokens[i], W, idx + (int64_t)i * W);
    }
    return REF_OK;
}

/*
 * Visibility of compressed block j (a stream-absolute compressed row) to
 * token t of segment b.
 * Block j_local of segment b pools tokens cu[b] + j_local*r ... + r - 1
 * (miles PR 2038 report, compressor.py _forward_thd, gather_idx), so it is
 * complete once the token at local position (j_local+1)*r - 1 has been seen.
 * Reading (the pages fix only "causal" via cmp_mask_mode=3 in the
 * sparse_flash_mla schema and "own segment only" via the report's fourth
 * THD bug): visible iff j is in t's segment and (j_local+1)*r <= pos+1.
 */
static int block_visible(const int32_t *cu, const int32_t *cu_c, int32_t b, int32_t t,
                         int32_t r, int32_t j) {
    if (j < cu_c[b] || j >= cu_c[b + 1]) return 0;
    int64_t j_local = j - cu_c[b];
    int64_t pos = t - cu[b];
    return (j_local + 1) * (int64_t)r <= pos + 1;
}

typedef struct {
    double s;
    int32_t j;
} cand_t;

/* Order: higher score first; on equal scores the lower block index first. */
static int cand_cmp(const void *a, const void *b) {
    const cand_t *x = (const cand_t *)a, *y = (const cand_t *)b;
    if (x->s > y->s) return -1;
    if (x->s < y->s) return 1;
    return (x->j < y->j) ? -1 : (x->j > y->j);
}

static int cand_cmp_j(const void *a, const void *b) {
    const cand_t *x = (const cand_t *)a, *y = (const cand_t *)b;
    return (x->j < y->j) ? -1 : (x->j > y->j);
}

/*
 * Lightning-indexer scores and top-k for a list of tokens.
 * hyper-parallel RFC, section 1 (lightning_indexer schema: q, k, w, topk,
 * cu_seqlens_q, cu_seqlens_k, cmp_ratio, return_value) and background item 1
 * (indexer over compressed KV); miles PR 2038 report, motivation item 4
 * (score only the query's own segment).
 * Score (reading; the pages print no formula):
 *     s(t, j) = sum_h w[t,h] * max(0, q[t,h,:] . k[j,:])
 * over the visible blocks j only. Selection: the topk highest scores, ties to
 * the lower j; fewer than topk visible -> all of them; output ascending in j,
 * padded with -1 (and -inf values).
 *
 * Rows of q / w / topk_idx / topk_val / kth / next are per listed token:
 * row i belongs to token tokens[i] (tokens == NULL: row i is token i and
 * n_tokens must equal T). kth[i] is the topk-th best score and next[i] the
 * (topk+1)-th (NaN when they do not exist), for judging near-ties.
 */
int csa_ref_indexer_topk(const double *q, const double *k, const double *w, int32_t T, int32_t Tc,
                         int32_t Hi, int32_t Di, const int32_t *cu_seqlens,
                         const int32_t *cu_seqlens_cmp, int32_t batch, int32_t cmp_ratio,
                         int32_t topk, const int32_t *tokens, int32_t n_tokens, int32_t *topk_idx,
                         double *topk_val, double *kth, double *next, int32_t *n_visible) {
    if (!q || !w || !cu_seqlens || !cu_seqlens_cmp || !topk_idx) return REF_ERR_ARG;
    if (Tc > 0 && !k) return REF_ERR_ARG;
    if (T < 0 || Tc < 0 || Hi < 1 || Di < 1 || cmp_ratio < 1 || topk < 1 || n_tokens < 0) return REF_ERR_ARG;
    if (!tokens && n_tokens != T) return REF_ERR_ARG;
    if (!check_cu(cu_seqlens, batch, T)) return REF_ERR_ARG;
    if (!check_cu(cu_seqlens_cmp, batch, Tc)) return REF_ERR_ARG;
    int err = REF_OK;
#pragma omp parallel for schedule(dynamic, 1)
    for (int32_t i = 0; i < n_tokens; ++i) {
        int32_t t = tokens ? tokens[i] : i;
        if (t < 0 || t >= T) {
            err = REF_ERR_ARG;
            continue;
        }
        int32_t b = segment_of(cu_seqlens, batch, t);
        int32_t nseg = cu_seqlens_cmp[b + 1] - cu_seqlens_cmp[b];
        cand_t *c = (cand_t *)malloc(sizeof(cand_t) * (size_t)(nseg > 0 ? nseg : 1));
        if (!c) {
            err = REF_ERR_NOMEM;
            continue;
        }
        int32_t n = 0;
        for (int32_t j = cu_seqlens_cmp[b]; j < cu_seqlens_cmp[b + 1]; ++j) {
            if (!block_visible(cu_seqlens, cu_seqlens_cmp, b, t, cmp_ratio, j)) continue;
            double s = 0.0;
            for (int32_t h = 0; h < Hi; ++h) {
                const double *qh = q + ((int64_t)i * Hi + h) * Di;
                const double *kj = k + (int64_t)j * Di;
                double dot = 0.0;
                for (int32_t d = 0; d < Di; ++d) dot += qh[d] * kj[d];
                double relu = dot > 0.0 ? dot : 0.0;
                s += w[(int64_t)i * Hi + h] * relu;
            }
            c[n].s = s;
            c[n].j = j;
            ++n;
        }
        qsort(c, (size_t)n, sizeof(cand_t), cand_cmp);
        if (kth) kth[i] = (n >= topk) ? c[topk - 1].s : NAN;
        if (next) next[i] = (n > topk) ? c[topk].s : NAN;
        if (n_visible) n_visible[i] = n;
        int32_t m = n < topk ? n : topk;
        qsort(c, (size_t)m, sizeof(cand_t), cand_cmp_j);
        for (int32_t s = 0; s < topk; ++s) {
            topk_idx[(int64_t)i * topk + s] = s < m ? c[s].j : -1;
            if (topk_val) topk_val[(int64_t)i * topk + s] = s < m ? c[s].s : -INFINITY;
        }
        free(c);
    }
    return err;
}

/*
 * Shared-KV MLA sparse attention forward with attention sinks.
 * hyper-parallel RFC, background item 2 (ori_kv band/sliding-window branch
 * plus cmp_kv compressed branch plus attention sink) and section 2
 * (sparse_flash_mla schema: q, ori_kv, cmp_kv, cmp_sparse_indices,
 * cu_seqlens_q/ori_kv/cmp_kv, sinks, softmax_scale, cmp_ratio, ori_win_left,
 * ori_win_right, return_softmax_lse); "missing arguments" analysis: the band
 * is derived from the window arguments and ori_sparse_indices is ignored.
 * Megatron-LM PR 7 (verl), environment note: head_dim = d_v = 512, so the
 * whole row is both key and value.
 *
 * For token t and head h, with keys = the window rows of ori_kv (as
 * csa_ref_window_idx) followed by the compressed rows of cmp_kv that are
 * listed in cmp_sparse_indices[t] (or, when it is NULL, every visible block:
 * the compressor-only / HCA mode), skipping -1 and any entry that is out of
 * range or not visible to t:
 *     l_i = softmax_scale * q[t,h,:] . kv_i
 *     m   = max(max_i l_i, sink_h)
 *     Z   = sum_i exp(l_i - m) + exp(sink_h - m)
 *     out[t,h,:] = sum_i exp(l_i - m) kv_i / Z
 *     lse[t,h]   = m + log(Z)
 * Readings: the sink is one logit per head, not multiplied by softmax_scale,
 * and adds to the denominator only (sinks == NULL: no sink term, which equals
 * a sink of -inf). lse is the natural log of the full denominator including
 * the sink, in scaled-logit units.
 *
 * Rows of q, cmp_sparse_indices, out and lse are per listed token as in
 * csa_ref_indexer_topk; ori_kv and cmp_kv are the full tensors.
 */
int csa_ref_sparse_mla_fwd(const double *q, const double *ori_kv, const double *cmp_kv,
                           const int32_t *cmp_sparse_indices, const int32_t *cu_seqlens,
                           const int32_t *cu_seqlens_cmp, int32_t batch, int32_t T, int32_t Tc,
                           int32_t H, int32_t D, int32_t topk, const double *sinks,
                           double softmax_scale, int32_t cmp_ratio, int32_t ori_win_left,
                           const int32_t *tokens, int32_t n_tokens, double *out, double *lse) {
    if (!q || !ori_kv || !cu_seqlens || !out) return REF_ERR_ARG;
    if (T < 0 || Tc < 0 || H < 1 || D < 1 || ori_win_left < 0 || n_tokens < 0) return REF_ERR_ARG;
    if (!tokens && n_tokens != T) return REF_ERR_ARG;
    if (!check_cu(cu_seqlens, batch, T)) return REF_ERR_ARG;
    const int use_cmp = cmp_kv != NULL && Tc > 0;
    if (use_cmp) {
        if (!cu_seqlens_cmp || cmp_ratio < 1) return REF_ERR_ARG;
        if (!check_cu(cu_seqlens_cmp, batch, Tc)) return REF_ERR_ARG;
        if (cmp_sparse_indices && topk < 1) return REF_ERR_ARG;
    }
    const int32_t W = ori_win_left + 1;
    const int32_t max_cmp = use_cmp ? (cmp_sparse_indices ? topk : Tc) : 0;
    int err = REF_OK;
#pragma omp parallel for schedule(dynamic, 1)
    for (int32_t i = 0; i < n_tokens; ++i) {
        int32_t t = tokens ? tokens[i] : i;
        if (t < 0 || t >= T) {
            err = REF_ERR_ARG;
            continue;
        }
        int32_t b = segment_of(cu_seqlens, batch, t);
        const double **rows = (const double **)malloc(sizeof(double *) * (size_t)(W + max_cmp));
        double *logit = (double *)malloc(sizeof(double) * (size_t)(W + max_cmp));
        if (!rows || !logit) {
            free(rows);
            free(logit);
            err = REF_ERR_NOMEM;
            continue;
        }
        int32_t n = 0;
        /* window branch: the most recent W rows of the own segment, self included */
        int32_t start = t - W + 1;
        if (start < cu_seqlens[b]) start = cu_seqlens[b];
        for (int32_t row = start; row <= t; ++row) rows[n++] = ori_kv + (int64_t)row * D;
        /* compressed branch */
        if (use_cmp) {
            if (cmp_sparse_indices) {
                for (int32_t s = 0; s < topk; ++s) {
                    int32_t j = cmp_sparse_indices[(int64_t)i * topk + s];
                    if (j < 0 || j >= Tc) continue;
                    if (!block_visible(cu_seqlens, cu_seqlens_cmp, b, t, cmp_ratio, j)) continue;
                    rows[n++] = cmp_kv + (int64_t)j * D;
                }
            } else {
                for (int32_t j = cu_seqlens_cmp[b]; j < cu_seqlens_cmp[b + 1]; ++j)
                    if (block_visible(cu_seqlens, cu_seqlens_cmp, b, t, cmp_ratio, j))
                        rows[n++] = cmp_kv + (int64_t)j * D;
            }
        }
        for (int32_t h = 0; h < H; ++h) {
            const double *qh = q + ((int64_t)i * H + h) * D;
            double m = -INFINITY;
            for (int32_t a = 0; a < n; ++a) {
                double dot = 0.0;
                for (int32_t d = 0; d < D; ++d) dot += qh[d] * rows[a][d];
                logit[a] = softmax_scale * dot;
                if (logit[a] > m) m = logit[a];
            }
            double sink = sinks ? sinks[h] : -INFINITY;
            if (sink > m) m = sink;
            double z = 0.0;
            for (int32_t a = 0; a < n; ++a) z += exp(logit[a] - m);
            if (sinks && sink != -INFINITY) z += exp(sink - m);
            double *oh = out + ((int64_t)i * H + h) * D;
            for (int32_t d = 0; d < D; ++d) oh[d] = 0.0;
            for (int32_t a = 0; a < n; ++a) {
                double p = exp(logit[a] - m) / z;
                for (int32_t d = 0; d < D; ++d) oh[d] += p * rows[a][d];
            }
            if (lse) lse[(int64_t)i * H + h] = m + log(z);
        }
        free(rows);
        free(logit);
    }
    return err;
}

/*
 * Backward of the shared-KV MLA attention with sinks (the gradient entry
 * point the miles PR 2038 report lists as sparse_flash_mla_grad: returns
 * d_query, d_ori_kv, d_cmp_kv, d_sinks and the head-averaged attention
 * distributions ori/cmp_softmax_l1_norm, shaped like the window and
 * compressed index lists).
 *
 * The forward is recomputed here in double from q and the KV rows (the
 * oracle does not trust a caller's out or lse). With l_a = scale q.k_a,
 * P_a = exp(l_a) / Z, P_sink = exp(sink) / Z and out = sum_a P_a v_a (v = k,
 * the same row), the loss gradient dout gives, per token t and head h:
 *   Dv      = dout . out
 *   dS_a    = P_a (dout . v_a - Dv)
 *   d_q     = scale sum_a dS_a k_a
 *   d_row_a += scale dS_a q + P_a dout        (row a as key and as value)
 *   d_sink  += -P_sink Dv
 *   l1[slot of a] += P_a / H
 * d_ori_kv [T, D], d_cmp_kv [Tc, D] and d_sinks [H] are overwritten (zeroed
 * first); ori_l1 is [n_tokens, W] in window-slot order (slot i <-> row
 * start + i, zero on the padded tail); cmp_l1 is [n_tokens, topk] in the
 * order of cmp_sparse_indices (zero where the entry is -1, out of range or
 * not visible), and is only written when cmp_sparse_indices is given.
 * Every pointer but q, dout, ori_kv, cu_seqlens, d_q and d_ori_kv may be
 * NULL where its part is absent or not wanted.
 */
int csa_ref_sparse_mla_bwd(const double *q, const double *dout, const double *ori_kv,
                           const double *cmp_kv, const int32_t *cmp_sparse_indices,
                           const int32_t *cu_seqlens, const int32_t *cu_seqlens_cmp, int32_t batch,
                           int32_t T, int32_t Tc, int32_t H, int32_t D, int32_t topk,
                           const double *sinks, double softmax_scale, int32_t cmp_ratio,
                           int32_t ori_win_left, double *d_q, double *d_ori_kv, double *d_cmp_kv,
                           double *d_sinks, double *ori_l1, double *cmp_l1) {
    if (!q || !dout || !ori_kv || !cu_seqlens || !d_q || !d_ori_kv) return REF_ERR_ARG;
    if (T < 0 || Tc < 0 || H < 1 || D < 1 || ori_win_left < 0) return REF_ERR_ARG;
    if (!check_cu(cu_seqlens, batch, T)) return REF_ERR_ARG;
    const int use_cmp = cmp_kv != NULL && Tc > 0;
    if (use_cmp) {
        if (!cu_seqlens_cmp || cmp_ratio < 1 || !d_cmp_kv) return REF_ERR_ARG;
        if (!check_cu(cu_seqlens_cmp, batch, Tc)) return REF_ERR_ARG;
        if (cmp_sparse_indices && topk < 1) return REF_ERR_ARG;
    }
    const int32_t W = ori_win_left + 1;
    const int32_t max_cmp = use_cmp ? (cmp_sparse_indices ? topk : Tc) : 0;
    memset(d_ori_kv, 0, sizeof(double) * (size_t)T * (size_t)D);
    if (use_cmp) memset(d_cmp_kv, 0, sizeof(double) * (size_t)Tc * (size_t)D);
    if (d_sinks) memset(d_sinks, 0, sizeof(double) * (size_t)H);
    if (ori_l1) memset(ori_l1, 0, sizeof(double) * (size_t)T * (size_t)W);
    if (cmp_l1 && use_cmp && cmp_sparse_indices)
        memset(cmp_l1, 0, sizeof(double) * (size_t)T * (size_t)topk);
    int err = REF_OK;
#pragma omp parallel for schedule(dynamic, 1)
    for (int32_t t = 0; t < T; ++t) {
        int32_t b = segment_of(cu_seqlens, batch, t);
        const int32_t n_max = W + max_cmp;
        const double **rows = (const double **)malloc(sizeof(double *) * (size_t)n_max);
        double **grads = (double **)malloc(sizeof(double *) * (size_t)n_max);
        double **l1 = (double **)malloc(sizeof(double *) * (size_t)n_max);
        double *logit = (double *)malloc(sizeof(double) * (size_t)n_max);
        double *prob = (double *)malloc(sizeof(double) * (size_t)n_max);
        double *ds = (double *)malloc(sizeof(double) * (size_t)n_max);
        double *o = (double *)malloc(sizeof(double) * (size_t)D);
        double *acc = (double *)malloc(sizeof(double) * (size_t)n_max * (size_t)D);
        double *sink_acc = (double *)malloc(sizeof(double) * (size_t)H);
        if (!rows || !grads || !l1 || !logit || !prob || !ds || !o || !acc || !sink_acc) {
            free(rows), free(grads), free(l1), free(logit), free(prob), free(ds), free(o);
            free(acc), free(sink_acc);
            err = REF_ERR_NOMEM;
            continue;
        }
        /* the token's keys, with where their gradient and distribution go */
        int32_t n = 0;
        int32_t start = t - W + 1;
        if (start < cu_seqlens[b]) start = cu_seqlens[b];
        for (int32_t row = start; row <= t; ++row) {
            rows[n] = ori_kv + (int64_t)row * D;
            grads[n] = d_ori_kv + (int64_t)row * D;
            l1[n] = ori_l1 ? ori_l1 + (int64_t)t * W + (row - start) : NULL;
            ++n;
        }
        if (use_cmp) {
            if (cmp_sparse_indices) {
                for (int32_t s = 0; s < topk; ++s) {
                    int32_t j = cmp_sparse_indices[(int64_t)t * topk + s];
                    if (j < 0 || j >= Tc) continue;
                    if (!block_visible(cu_seqlens, cu_seqlens_cmp, b, t, cmp_ratio, j)) continue;
                    rows[n] = cmp_kv + (int64_t)j * D;
                    grads[n] = d_cmp_kv + (int64_t)j * D;
                    l1[n] = cmp_l1 ? cmp_l1 + (int64_t)t * topk + s : NULL;
                    ++n;
                }
            } else {
                for (int32_t j = cu_seqlens_cmp[b]; j < cu_seqlens_cmp[b + 1]; ++j) {
                    if (!block_visible(cu_seqlens, cu_seqlens_cmp, b, t, cmp_ratio, j)) continue;
                    rows[n] = cmp_kv + (int64_t)j * D;
                    grads[n] = d_cmp_kv + (int64_t)j * D;
                    l1[n] = NULL;
                    ++n;
                }
            }
        }
        memset(acc, 0, sizeof(double) * (size_t)n * (size_t)D);
        for (int32_t h = 0; h < H; ++h) {
            const double *qh = q + ((int64_t)t * H + h) * D;
            const double *gh = dout + ((int64_t)t * H + h) * D;
            double *dqh = d_q + ((int64_t)t * H + h) * D;
            /* forward again: logits, max, denominator with the sink */
            double m = -INFINITY;
            for (int32_t a = 0; a < n; ++a) {
                double dot = 0.0;
                for (int32_t d = 0; d < D; ++d) dot += qh[d] * rows[a][d];
                logit[a] = softmax_scale * dot;
                if (logit[a] > m) m = logit[a];
            }
            double sink = sinks ? sinks[h] : -INFINITY;
            if (sink > m) m = sink;
            double z = 0.0;
            for (int32_t a = 0; a < n; ++a) z += exp(logit[a] - m);
            double p_sink = 0.0;
            if (sinks && sink != -INFINITY) {
                z += exp(sink - m);
                p_sink = exp(sink - m);
            }
            p_sink /= z;
            for (int32_t d = 0; d < D; ++d) o[d] = 0.0;
            for (int32_t a = 0; a < n; ++a) {
                prob[a] = exp(logit[a] - m) / z;
                for (int32_t d = 0; d < D; ++d) o[d] += prob[a] * rows[a][d];
            }
            /* Dv = dout . out; dS_a = P_a (dout . v_a - Dv) */
            double dv = 0.0;
            for (int32_t d = 0; d < D; ++d) dv += gh[d] * o[d];
            for (int32_t a = 0; a < n; ++a) {
                double dp = 0.0;
                for (int32_t d = 0; d < D; ++d) dp += gh[d] * rows[a][d];
                ds[a] = prob[a] * (dp - dv);
            }
            for (int32_t d = 0; d < D; ++d) {
                double s = 0.0;
                for (int32_t a = 0; a < n; ++a) s += ds[a] * rows[a][d];
                dqh[d] = softmax_scale * s;
            }
            for (int32_t a = 0; a < n; ++a) {
                double *ga = acc + (int64_t)a * D;
                for (int32_t d = 0; d < D; ++d)
                    ga[d] += softmax_scale * ds[a] * qh[d] + prob[a] * gh[d];
                if (l1[a]) *l1[a] += prob[a] / H;
            }
            sink_acc[h] = -p_sink * dv;
        }
        /* the rows are shared between tokens: add this token's part in turn */
#pragma omp critical(csa_ref_bwd_scatter)
        {
            for (int32_t a = 0; a < n; ++a)
                for (int32_t d = 0; d < D; ++d) grads[a][d] += acc[(int64_t)a * D + d];
            if (d_sinks)
                for (int32_t h = 0; h < H; ++h) d_sinks[h] += sink_acc[h];
        }
        free(rows), free(grads), free(l1), free(logit), free(prob), free(ds), free(o);
        free(acc), free(sink_acc);
    }
    return err;
}

/*
 * Indexer KL-loss gradient (the hyper-parallel RFC, section 3,
 * sparse_lightning_indexer_kl_loss_grad(q, k, w, sparse_indices,
 * attn_softmax_l1_norm, cu_seqlens_q, cu_seqlens_k, mask_mode=3, cmp_ratio):
 * "indexer backward + KL loss", fed with the main attention's target
 * distribution p that sparse_flash_mla_grad returns as softmax_l1_norm;
 * MindSpeed-LLM PR 4842, main changes: under TND the loss is normalised by
 * the global token count, passed as a gradient scale).
 *
 * Reading (the pages print the argument list, not the loss): for token t,
 * the entries s of sparse_indices[t] that name a row j in [0, Tc) visible to
 * t (the same causal rule as the indexer, mask_mode 3) form its set S.
 *     I_s  = sum_h w[t,h] * max(0, q[t,h,:] . k[j_s,:])   (indexer score)
 *     p_s  = a_s / sum_{u in S} a_u,   a = attn_softmax_l1_norm[t, :]
 *     pi_s = exp(I_s) / sum_{u in S} exp(I_u)
 *     loss[t] = sum_{s in S, p_s > 0} p_s (log p_s - log pi_s)
 * i.e. KL(p || softmax(I)) over the selected rows, with p the attention
 * distribution L1-normalised over the same rows. A token with no entry in S,
 * or whose entries in S carry no mass, has loss 0 and no gradient.
 * Gradients of L = grad_scale * sum_t loss[t] (p is a target, not
 * differentiated), with g_s = grad_scale (pi_s - p_s) = dL/dI_s:
 *     d_w[t,h]    = sum_s g_s max(0, a_hs)
 *     d_q[t,h,:]  = sum_s g_s w[t,h] [a_hs > 0] k[j_s,:]
 *     d_k[j_s,:] += g_s sum_h w[t,h] [a_hs > 0] q[t,h,:]
 * with a_hs = q[t,h,:] . k[j_s,:] and the ReLU's derivative 0 at 0.
 * Each entry counts on its own (a row listed twice contributes twice).
 *
 * Rows of q, w, sparse_indices, attn_l1, d_q, d_w and loss are per listed
 * token (tokens == NULL: all T tokens, row i is token i); d_k [Tc, Di] is
 * overwritten with the contributions of the listed tokens (may be NULL).
 * g_out (may be NULL) receives dL/dI_s per list entry, [n_tokens, topk],
 * zero for skipped entries.
 */
int csa_ref_indexer_kl_loss_grad(const double *q, const double *k, const double *w,
                                 const int32_t *sparse_indices, const double *attn_l1, int32_t T,
                                 int32_t Tc, int32_t Hi, int32_t Di, int32_t topk,
                                 const int32_t *cu_seqlens, const int32_t *cu_seqlens_cmp,
                                 int32_t batch, int32_t cmp_ratio, double grad_scale,
                                 const int32_t *tokens, int32_t n_tokens, double *d_q, double *d_k,
                                 double *d_w, double *loss, double *g_out) {
    if (!q || !w || !sparse_indices || !attn_l1 || !cu_seqlens || !cu_seqlens_cmp) return REF_ERR_ARG;
    if (!d_q || !d_w || !loss) return REF_ERR_ARG;
    if (Tc > 0 && !k) return REF_ERR_ARG;
    if (T < 0 || Tc < 0 || Hi < 1 || Di < 1 || topk < 1 || cmp_ratio < 1 || n_tokens < 0) return REF_ERR_ARG;
    if (!tokens && n_tokens != T) return REF_ERR_ARG;
    if (!check_cu(cu_seqlens, batch, T)) return REF_ERR_ARG;
    if (!check_cu(cu_seqlens_cmp, batch, Tc)) return REF_ERR_ARG;
    if (d_k) memset(d_k, 0, sizeof(double) * (size_t)Tc * (size_t)Di);
    int err = REF_OK;
#pragma omp parallel for schedule(dynamic, 1)
    for (int32_t i = 0; i < n_tokens; ++i) {
        int32_t t = tokens ? tokens[i] : i;
        double *dq = d_q + (int64_t)i * Hi * Di;
        double *dw = d_w + (int64_t)i * Hi;
        for (int64_t e = 0; e < (int64_t)Hi * Di; ++e) dq[e] = 0.0;
        for (int32_t h = 0; h < Hi; ++h) dw[h] = 0.0;
        loss[i] = 0.0;
        if (g_out)
            for (int32_t s = 0; s < topk; ++s) g_out[(int64_t)i * topk + s] = 0.0;
        if (t < 0 || t >= T) {
            err = REF_ERR_ARG;
            continue;
        }
        int32_t b = segment_of(cu_seqlens, batch, t);
        int32_t *rows = (int32_t *)malloc(sizeof(int32_t) * (size_t)topk);
        int32_t *slot = (int32_t *)malloc(sizeof(int32_t) * (size_t)topk);
        double *score = (double *)malloc(sizeof(double) * (size_t)topk);
        double *p = (double *)malloc(sizeof(double) * (size_t)topk);
        double *dots = (double *)malloc(sizeof(double) * (size_t)topk * (size_t)Hi);
        double *gk = (double *)malloc(sizeof(double) * (size_t)topk * (size_t)Di);
        if (!rows || !slot || !score || !p || !dots || !gk) {
            free(rows), free(slot), free(score), free(p), free(dots), free(gk);
            err = REF_ERR_NOMEM;
            continue;
        }
        /* the token's set S, its scores and its target mass */
        int32_t n = 0;
        double mass = 0.0;
        for (int32_t s = 0; s < topk; ++s) {
            int32_t j = sparse_indices[(int64_t)i * topk + s];
            if (j < 0 || j >= Tc) continue;
            if (!block_visible(cu_seqlens, cu_seqlens_cmp, b, t, cmp_ratio, j)) continue;
            rows[n] = j;
            slot[n] = s;
            p[n] = attn_l1[(int64_t)i * topk + s];
            mass += p[n];
            double sc = 0.0;
            for (int32_t h = 0; h < Hi; ++h) {
                const double *qh = q + ((int64_t)i * Hi + h) * Di;
                const double *kj = k + (int64_t)j * Di;
                double dot = 0.0;
                for (int32_t d = 0; d < Di; ++d) dot += qh[d] * kj[d];
                dots[(int64_t)n * Hi + h] = dot;
                sc += w[(int64_t)i * Hi + h] * (dot > 0.0 ? dot : 0.0);
            }
            score[n] = sc;
            ++n;
        }
        if (n > 0 && mass > 0.0) {
            /* log-softmax of the scores over S */
            double mx = -INFINITY;
            for (int32_t s = 0; s < n; ++s)
                if (score[s] > mx) mx = score[s];
            double z = 0.0;
            for (int32_t s = 0; s < n; ++s) z += exp(score[s] - mx);
            double lz = mx + log(z);
            double kl = 0.0;
            for (int32_t s = 0; s < n; ++s) {
                double ps = p[s] / mass;
                double log_pi = score[s] - lz;
                if (ps > 0.0) kl += ps * (log(ps) - log_pi);
                /* reuse score[] for g_s = dL/dI_s */
                score[s] = grad_scale * (exp(log_pi) - ps);
                if (g_out) g_out[(int64_t)i * topk + slot[s]] = score[s];
            }
            loss[i] = kl;
            for (int32_t s = 0; s < n; ++s) {
                const double g = score[s];
                const double *kj = k + (int64_t)rows[s] * Di;
                double *gks = gk + (int64_t)s * Di;
                for (int32_t d = 0; d < Di; ++d) gks[d] = 0.0;
                for (int32_t h = 0; h < Hi; ++h) {
                    double dot = dots[(int64_t)s * Hi + h];
                    dw[h] += g * (dot > 0.0 ? dot : 0.0);
                    if (!(dot > 0.0)) continue;
                    double c = g * w[(int64_t)i * Hi + h];
                    const double *qh = q + ((int64_t)i * Hi + h) * Di;
                    double *dqh = dq + (int64_t)h * Di;
                    for (int32_t d = 0; d < Di; ++d) {
                        dqh[d] += c * kj[d];
                        gks[d] += c * qh[d];
                    }
                }
            }
            if (d_k) {
#pragma omp critical(csa_ref_kl_scatter)
                for (int32_t s = 0; s < n; ++s)
                    for (int32_t d = 0; d < Di; ++d)
                        d_k[(int64_t)rows[s] * Di + d] += gk[(int64_t)s * Di + d];
            }
        }
        free(rows), free(slot), free(score), free(p), free(dots), free(gk);
    }
    return err;
}

/*
 * THD compressor: grouping, overlap transform and pooling of one compressor
 * (miles PR 2038 report, compressor.py DeepSeekV4Compressor._forward_thd and
 * _overlap_transform_thd).
 *
 * Inputs are the two projections of the packed rows, kv = x W_kv^T and
 * score = x W_gate^T ([T, Wd] fp32, Wd = 2 head_dim with overlap, head_dim
 * without; the page computes them with linear_bf16_fp32), and the absolute
 * position embedding ape [cmp_ratio, Wd] (may be NULL: zero).
 * Grouping (gather_idx): compressed row g = cu_c[b] + j of sequence b takes
 * the rows cu[b] + j r + i, i < r, of kv and score; ape[i] is added to the
 * score of slot i (reading: the page shows ape viewed as [1, ratio, 1, -1]
 * next to the grouped tensors and omits where it is added).
 * Overlap (when overlap != 0): each group becomes 2r slots of head_dim: slot
 * i < r holds the first half (columns [0, hd)) of row i of the previous
 * group of the same sequence, slot r + i the second half (columns [hd, 2hd))
 * of its own row i; the first group of a sequence has no predecessor, and
 * its slots i < r are filled with 0 (kv) and -inf (score).
 * Pooling (reading: the page omits everything after the overlap transform;
 * the -inf fill of the score only has a meaning as a softmax logit): per
 * compressed row and dimension e,
 *     out[g, e] = sum_s softmax_s(score[g, s, e]) kv[g, s, e]
 * over the group's slots. out is [Tc, head_dim], fp64 here.
 * Returns REF_ERR_ARG on inconsistent arguments.
 */
int csa_ref_compress_thd(const double *kv, const double *score, const double *ape,
                         const int32_t *cu_seqlens, const int32_t *cu_seqlens_cmp, int32_t batch,
                         int32_t T, int32_t cmp_ratio, int32_t head_dim, int32_t overlap,
                         double *out) {
    if (!kv || !score || !cu_seqlens || !cu_seqlens_cmp || !out) return REF_ERR_ARG;
    if (T < 0 || cmp_ratio < 1 || head_dim < 1 || batch < 0) return REF_ERR_ARG;
    if (!check_cu(cu_seqlens, batch, T)) return REF_ERR_ARG;
    for (int32_t b = 0; b < batch; ++b) {
        int32_t len = cu_seqlens[b + 1] - cu_seqlens[b];
        if (cu_seqlens_cmp[b + 1] - cu_seqlens_cmp[b] != len / cmp_ratio) return REF_ERR_ARG;
    }
    if (cu_seqlens_cmp[0] != 0) return REF_ERR_ARG;
    const int32_t r = cmp_ratio, hd = head_dim;
    const int32_t wd = overlap ? 2 * hd : hd;
    const int32_t slots = overlap ? 2 * r : r;
    const int32_t Tc = cu_seqlens_cmp[batch];
    int err = REF_OK;
#pragma omp parallel for schedule(static)
    for (int32_t g = 0; g < Tc; ++g) {
        int32_t b = segment_of(cu_seqlens_cmp, batch, g);
        int32_t j = g - cu_seqlens_cmp[b];
        double *sk = (double *)malloc(sizeof(double) * (size_t)slots);
        double *sv = (double *)malloc(sizeof(double) * (size_t)slots);
        if (!sk || !sv) {
            free(sk), free(sv);
            err = REF_ERR_NOMEM;
            continue;
        }
        for (int32_t e = 0; e < hd; ++e) {
            /* the group's slots for dimension e, after grouping, ape and overlap */
            for (int32_t i = 0; i < r; ++i) {
                int64_t own = cu_seqlens[b] + (int64_t)j * r + i;
                if (overlap) {
                    if (j == 0) {
                        sv[i] = 0.0;
                        sk[i] = -INFINITY;
                    } else {
                        int64_t prev = own - r;
                        sv[i] = kv[prev * wd + e];
                        sk[i] = score[prev * wd + e] + (ape ? ape[(int64_t)i * wd + e] : 0.0);
                    }
                    sv[r + i] = kv[own * wd + hd + e];
                    sk[r + i] = score[own * wd + hd + e] + (ape ? ape[(int64_t)i * wd + hd + e] : 0.0);
                } else {
                    sv[i] = kv[own * wd + e];
                    sk[i] = score[own * wd + e] + (ape ? ape[(int64_t)i * wd + e] : 0.0);
                }
            }
            double m = -INFINITY;
            for (int32_t s = 0; s < slots; ++s)
                if (sk[s] > m) m = sk[s];
            double z = 0.0, acc = 0.0;
            for (int32_t s = 0; s < slots; ++s) {
                if (sk[s] == -INFINITY) continue;
                double p = exp(sk[s] - m);
                z += p;
                acc += p * sv[s];
            }
            out[(int64_t)g * hd + e] = acc / z;
        }
        free(sk), free(sv);
    }
    return err;
}
