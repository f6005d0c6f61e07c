/*
 * csa.h -- C ABI of the GB300 (sm_103a) forward path of DeepSeek-V4
 * Compressed Sparse Attention (CSA) and its compressor-only mode (HCA) over
 * THD-packed variable-length sequences (and fixed-shape BSND batches), on one
 * GPU; of the backward of its sparse MLA attention, the indexer's KL-loss
 * gradient and the THD compressor core that produces the compressed rows.
 *
 * Sources (web pages, cited by title and section):
 *   [miles#2038]  "PR #2038 完整报告" (radixark/miles): "Enable THD
 *                 packed-sequence training for DeepSeek-V4-Flash, with context
 *                 parallelism"; sections 功能与动机 (motivation), 关键源码片段
 *                 (key source excerpts: thd_utils.py, compressor.py), 风险与影响.
 *   [hp#RFC]      "【RFC】DeepSeek-V4 CSA/HCA 自定义算子接入与对外接口对标
 *                 torch_extension" (hyper-parallel); sections 背景 (background),
 *                 1 npu_lightning_indexer, 2 npu_sparse_flash_mla,
 *                 3 npu_sparse_lightning_indexer_kl_loss_grad,
 *                 4 npu_sparse_flash_mla_grad, 缺失入参的用途分析
 *                 (analysis of the missing arguments).
 *   [MS#4842]     MindSpeed-LLM PR 4842; section 主要改动 (main changes):
 *                 LayerCompressMode {NO_COMPRESS, COMPRESSOR_ONLY, INDEXER};
 *                 the indexer loss's num_seqs (global token count) under TND.
 *   [MLM#7]       "feat(deepseek_v4): faithful THD context-parallel path for DS4
 *                 CSA" (verl Megatron-LM PR 7); section Environment note:
 *                 head_dim = d_v = 512.
 *
 * Conventions shared by every call
 *   - Layout is THD ("TND"): tokens of all sequences concatenated along the
 *     first axis; cu_seqlens[batch+1] (int32, device memory, starting at 0,
 *     non-decreasing) holds the sequence starts, as in [miles#2038] ThdLayout.
 *     Every tensor is row-major and contiguous.
 *   - Row indices (window rows, compressed rows, top-k output) are
 *     stream-absolute rows of the packed tensors ([miles#2038], review notes).
 *   - bf16 tensors are passed as csa_bf16_t (the raw 16-bit bfloat16 pattern).
 *   - All pointers are DEVICE pointers unless stated otherwise; all sizes are
 *     host integers. The caller owns and allocates every buffer, including
 *     workspaces; the library allocates no device memory per call and never
 *     synchronises the stream.
 *   - Every call is asynchronous and stream-ordered on `stream`
 *     (a cudaStream_t; NULL is the legacy default stream).
 *   - Argument checks that need only host values run synchronously: a call
 *     that returns anything but CSA_OK has launched nothing. Checks that would
 *     need device data (cu_seqlens contents) are not made; kernels never read
 *     or write outside the extents the host sizes imply, whatever the device
 *     data holds, and record an inconsistency they meet in a device error word
 *     read by csa_device_error().
 */
#ifndef CSA_GB300_H_
#define CSA_GB300_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
struct CUstream_st;
typedef struct CUstream_st *csa_stream_t;

/* Raw bfloat16 bit pattern. */
typedef uint16_t csa_bf16_t;

typedef enum {
    CSA_OK = 0,
    CSA_ERR_NULL = 1,         /* a required pointer is NULL                       */
    CSA_ERR_SHAPE = 2,        /* sizes are negative or inconsistent               */
    CSA_ERR_UNSUPPORTED = 3,  /* a valid request the library does not implement */
    CSA_ERR_WORKSPACE = 4,    /* workspace too small or misaligned                */
    CSA_ERR_CUDA = 5,         /* a CUDA runtime/driver call or launch failed      */
    CSA_ERR_DEVICE_CHECK = 6, /* a kernel met inconsistent device data            */
    CSA_ERR_TIMEOUT = 7       /* a bounded device-side wait gave up               */
} csa_status_t;

/* Static string for a status code (never NULL). */
const char *csa_status_string(csa_status_t status);

/*
 * Compressed cu_seqlens.            [miles#2038] compressor.py _forward_thd
 * docstring and 风险与影响 item 2: the trailing len % cmp_ratio tokens of a
 * sequence produce no compressed row, so sequence b owns floor(len_b/cmp_ratio)
 * rows of the compressed stream:
 *     cu_seqlens_cmp[0] = 0,
 *     cu_seqlens_cmp[b+1] = cu_seqlens_cmp[b] + floor(len_b / cmp_ratio).
 * cu_seqlens      [batch+1] int32 in.
 * cu_seqlens_cmp  [batch+1] int32 out (may not alias cu_seqlens).
 * Errors: NULL pointer -> CSA_ERR_NULL; batch < 0 -> CSA_ERR_SHAPE;
 * cmp_ratio < 1 -> CSA_ERR_UNSUPPORTED. batch == 0 writes cu_seqlens_cmp[0]=0.
 */
csa_status_t csa_compress_cu_seqlens(const int32_t *cu_seqlens, int32_t batch, int32_t cmp_ratio,
                                     int32_t *cu_seqlens_cmp, csa_stream_t stream);

/*
 * Segment-clamped sliding-window rows.   [miles#2038] thd_utils.py
 * get_window_topk_idxs_thd; [hp#RFC] section 2 (ori_win_left=127,
 * ori_win_right=0 defaults; band mask ori_mask_mode=4).
 * With W = ori_win_left + 1 and token t in sequence b:
 *     start = max(t - W + 1, cu_seqlens[b]);
 *     idx[t, i] = start + i  if start + i <= t  else -1     (0 <= i < W)
 * i.e. the W most recent rows of t's own sequence, self included, ascending,
 * -1 padded at the tail.
 * cu_seqlens [batch+1] int32 in (cu_seqlens[batch] must equal total_tokens).
 * idx        [total_tokens, W] int32 out.
 * Errors: NULL -> CSA_ERR_NULL; negative sizes -> CSA_ERR_SHAPE;
 * ori_win_right != 0 -> CSA_ERR_UNSUPPORTED (only the causal band exists).
 * total_tokens == 0 launches nothing. A token not covered by cu_seqlens
 * (inconsistent device data) gets an all -1 row and sets the device error.
 */
csa_status_t csa_window_idx(const int32_t *cu_seqlens, int32_t batch, int32_t total_tokens,
                            int32_t ori_win_left, int32_t ori_win_right, int32_t *idx,
                            csa_stream_t stream);

/*
 * Bytes of device workspace csa_indexer_topk needs for these sizes
 * (0 when it needs none). The value depends on host sizes only.
 */
size_t csa_indexer_topk_workspace_size(int32_t total_tokens, int32_t total_cmp, int32_t index_heads,
                                       int32_t index_dim, int32_t topk);

/*
 * Lightning-indexer score + per-sequence causal top-k over compressed KV.
 * [hp#RFC] section 1 (lightning_indexer(q, k, w, topk, cu_seqlens_q,
 * cu_seqlens_k, cmp_ratio, return_value)) and background item 1;
 * [miles#2038] 功能与动机 item 4 (score only the query's own sequence).
 * Score of token t for compressed row j (the pages give no formula; reading):
 *     s(t, j) = sum_h w[t,h] * max(0, q[t,h,:] . k[j,:])      (fp32 accumulate)
 * taken over the rows j visible to t: j in t's own sequence b and
 *     (j - cu_seqlens_cmp[b] + 1) * cmp_ratio <= (t - cu_seqlens_q[b]) + 1,
 * i.e. the compressed row is complete (its last pooled token is at or
 * before t). Output per token: the topk highest-scoring visible rows, ties
 * to the lower row, emitted in ascending row order; fewer than topk visible
 * -> all of them, then -1 (topk_val: -inf) padding.
 * q        [T, Hi, Di] bf16      k  [Tc, Di] bf16        w [T, Hi] fp32
 * cu_seqlens_q [batch+1], cu_seqlens_cmp_kv [batch+1] int32 (the latter as
 *          produced by csa_compress_cu_seqlens with the same cmp_ratio).
 * topk_idx [T, topk] int32 out; topk_val [T, topk] fp32 out or NULL.
 * workspace: device buffer of at least csa_indexer_topk_workspace_size(...)
 *          bytes, 256-byte aligned (may be NULL when that size is 0).
 * Errors: NULL -> CSA_ERR_NULL (k may be NULL only when Tc == 0);
 * negative sizes or topk < 1 -> CSA_ERR_SHAPE; Di not in {64, 128},
 * Hi not in [1, 64], cmp_ratio < 2 -> CSA_ERR_UNSUPPORTED; workspace too
 * small -> CSA_ERR_WORKSPACE. Tc == 0 fills topk_idx with -1.
 */
csa_status_t csa_indexer_topk(const csa_bf16_t *q, const csa_bf16_t *k, const float *w,
                              int32_t total_tokens, int32_t total_cmp, int32_t index_heads,
                              int32_t index_dim, const int32_t *cu_seqlens_q,
                              const int32_t *cu_seqlens_cmp_kv, int32_t batch, int32_t cmp_ratio,
                              int32_t topk, int32_t *topk_idx, float *topk_val, void *workspace,
                              size_t workspace_bytes, csa_stream_t stream);

/*
 * Shared-KV MLA sparse attention forward with attention sinks.
 * [hp#RFC] background item 2 (ori_kv band / sliding-window branch + cmp_kv
 * compressed branch + attention sink) and section 2 (sparse_flash_mla
 * schema; ori_sparse_indices takes no part: the band comes from the window
 * arguments); [MLM#7] environment note (head_dim = d_v = 512: the whole
 * 512-wide row is both key and value); [MS#4842] LayerCompressMode.
 * For token t, head h, keys = the window rows of ori_kv (as csa_window_idx)
 * followed by the compressed rows listed in cmp_sparse_indices[t] (entries
 * that are -1, out of [0, Tc) or not visible to t are skipped), or, when
 * cmp_sparse_indices is NULL, every compressed row visible to t
 * (COMPRESSOR_ONLY / HCA mode); cmp_kv == NULL or Tc == 0 means window only:
 *     l_i = softmax_scale * q[t,h,:] . kv_i
 *     m   = max(max_i l_i, sink_h)
 *     Z   = sum_i exp(l_i - m) + exp(sink_h - m)
 *     out[t,h,:] = sum_i exp(l_i - m) kv_i / Z              (bf16, RNE)
 *     lse[t,h]   = m + ln Z                                  (fp32)
 * The sink is one logit per head, not scaled by softmax_scale; sinks == NULL
 * is the same as every sink being -inf.
 * q [T, H, D] bf16; ori_kv [T, D] bf16; cmp_kv [Tc, D] bf16 or NULL;
 * cmp_sparse_indices [T, topk] int32 or NULL; cu_seqlens_* [batch+1] int32;
 * sinks [H] fp32 or NULL; out [T, H, D] bf16; softmax_lse [T, H] fp32,
 * written only when return_softmax_lse != 0 (may be NULL otherwise).
 * Errors: NULL q/ori_kv/cu_seqlens_q/out -> CSA_ERR_NULL (cu_seqlens_cmp_kv
 * is required when cmp_kv is used); negative sizes -> CSA_ERR_SHAPE;
 * D != 512, H not in [1, 64], ori_win_right != 0, ori_win_left > 1023,
 * cmp_ratio < 2 while cmp_kv is used, topk > 1024 with cmp_sparse_indices,
 * or cu_seqlens_ori_kv neither NULL nor equal to cu_seqlens_q (prefix KV)
 * -> CSA_ERR_UNSUPPORTED. q, ori_kv, cmp_kv and out must be 16-byte aligned.
 */
csa_status_t csa_sparse_mla_fwd(const csa_bf16_t *q, const csa_bf16_t *ori_kv,
                                const csa_bf16_t *cmp_kv, const int32_t *cmp_sparse_indices,
                                const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_ori_kv,
                                const int32_t *cu_seqlens_cmp_kv, int32_t batch,
                                int32_t total_tokens, int32_t total_cmp, int32_t heads,
                                int32_t head_dim, int32_t topk, const float *sinks,
                                float softmax_scale, int32_t cmp_ratio, int32_t ori_win_left,
                                int32_t ori_win_right, csa_bf16_t *out, float *softmax_lse,
                                int32_t return_softmax_lse, csa_stream_t stream);

/*
 * Backward of csa_sparse_mla_fwd.
 * [miles#2038] report and [hp#RFC] section 4 (npu_sparse_flash_mla_grad:
 * from q, dout, the forward's attn_out and softmax_lse it returns d_query,
 * d_ori_kv, d_cmp_kv, d_sinks, and ori/cmp_softmax_l1_norm, the attention
 * distribution averaged over heads, shaped like the window and compressed
 * index lists). Keys, masks, sinks and scale exactly as csa_sparse_mla_fwd;
 * with P_a = exp(softmax_scale q.kv_a - lse), P_sink = exp(sink - lse) and
 * Dv = dout . out, per token t and head h:
 *     dS_a  = P_a (dout[t,h,:] . kv_a - Dv)
 *     d_q[t,h,:]      = softmax_scale sum_a dS_a kv_a
 *     d_row(kv_a)    += softmax_scale dS_a q[t,h,:] + P_a dout[t,h,:]
 *     d_sinks[h]     -= P_sink Dv
 *     l1[t, slot(a)] += P_a / H
 * (the row's gradient counts it both as key and as value: it is one row).
 * Inputs: q, dout, out [T, H, D] bf16 (out and softmax_lse [T, H] fp32 are
 * what csa_sparse_mla_fwd returned for the same arguments); the rest as
 * csa_sparse_mla_fwd. Outputs, all fp32 and overwritten:
 *   d_q [T, H, D];  d_ori_kv [T, D];  d_cmp_kv [Tc, D] (when cmp_kv is used);
 *   d_sinks [H] (when sinks is given; may be NULL to skip);
 *   ori_softmax_l1_norm [T, ori_win_left + 1] or NULL: slot i is window row
 *     max(t - ori_win_left, segment start) + i, zero past the token itself;
 *   cmp_softmax_l1_norm [T, topk] or NULL: slot i follows
 *     cmp_sparse_indices[t, i], zero where that entry is skipped; only with
 *     cmp_sparse_indices (with every visible row there is no list).
 * The KV-row gradients are sums over tokens made with fp32 atomics, so their
 * last bits depend on the order the tokens finish in.
 * Errors: as csa_sparse_mla_fwd, plus NULL dout/out/softmax_lse/d_q/d_ori_kv
 * (or d_cmp_kv when cmp_kv is used) -> CSA_ERR_NULL. q, dout, ori_kv,
 * cmp_kv, d_ori_kv and d_cmp_kv must be 16-byte aligned, out 4-byte aligned
 * (else CSA_ERR_UNSUPPORTED).
 */
csa_status_t csa_sparse_mla_bwd(const csa_bf16_t *q, const csa_bf16_t *dout, const csa_bf16_t *out,
                                const float *softmax_lse, const csa_bf16_t *ori_kv,
                                const csa_bf16_t *cmp_kv, const int32_t *cmp_sparse_indices,
                                const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_ori_kv,
                                const int32_t *cu_seqlens_cmp_kv, int32_t batch,
                                int32_t total_tokens, int32_t total_cmp, int32_t heads,
                                int32_t head_dim, int32_t topk, const float *sinks,
                                float softmax_scale, int32_t cmp_ratio, int32_t ori_win_left,
                                int32_t ori_win_right, float *d_q, float *d_ori_kv,
                                float *d_cmp_kv, float *d_sinks, float *ori_softmax_l1_norm,
                                float *cmp_softmax_l1_norm, csa_stream_t stream);

/*
 * Indexer KL-loss gradient: the backward of the lightning indexer against the
 * main attention's distribution.
 * [hp#RFC] section 3 (sparse_lightning_indexer_kl_loss_grad(q, k, w,
 * sparse_indices, attn_softmax_l1_norm, cu_seqlens_q, cu_seqlens_k,
 * mask_mode=3, cmp_ratio): indexer backward plus KL loss, fed with the target
 * distribution p that the attention backward returns as softmax_l1_norm);
 * [MS#4842] (under TND the loss is normalised by the global token count:
 * pass that factor as grad_scale). The pages give the arguments, not the
 * loss; the reading taken: for token t, the entries s of sparse_indices[t]
 * naming a row j_s in [0, Tc) visible to t (the indexer's causal rule) form
 * its set S, and
 *     I_s     = sum_h w[t,h] max(0, a_hs),  a_hs = q[t,h,:] . k[j_s,:]
 *     p_s     = l1[t,s] / sum_{u in S} l1[t,u]
 *     loss[t] = sum_{s in S, p_s > 0} p_s (log p_s - log softmax_S(I)_s)
 * (KL(p || softmax of the indexer scores) over the selected rows). Outputs
 * are the gradients of L = grad_scale * sum_t loss[t] (p is a target):
 *     g_s         = grad_scale (softmax_S(I)_s - p_s)
 *     d_w[t,h]    = sum_s g_s max(0, a_hs)
 *     d_q[t,h,:]  = sum_s g_s w[t,h] [a_hs > 0] k[j_s,:]
 *     d_k[j_s,:] += g_s sum_h w[t,h] [a_hs > 0] q[t,h,:]
 * A token with no entry in S, or whose entries carry no mass, gets loss 0
 * and zero gradients. Each entry counts on its own.
 * q [T, Hi, Di] bf16; k [Tc, Di] bf16; w [T, Hi] fp32;
 * sparse_indices [T, topk] int32 (e.g. csa_indexer_topk's output);
 * attn_softmax_l1_norm [T, topk] fp32 (e.g. csa_sparse_mla_bwd's
 * cmp_softmax_l1_norm for the same list); cu_seqlens_q, cu_seqlens_cmp_kv
 * [batch+1] int32 as for csa_indexer_topk.
 * Outputs, fp32, overwritten: d_q [T, Hi, Di], d_k [Tc, Di], d_w [T, Hi],
 * loss [T] (unscaled KL per token; may be NULL). d_k is a sum over tokens
 * made with fp32 atomics, so its last bits depend on the order the tokens
 * finish in. Arithmetic: with Di = 128 the contractions run on the tensor
 * cores (bf16 q and k as given, fp32 accumulation; the per-entry factor
 * g_s w[t,h] [a_hs > 0] enters as the sum of two bf16 parts, about 2^-17
 * relative); with Di = 64 everything is fp32 on the CUDA cores.
 * Errors: negative sizes or topk < 1 -> CSA_ERR_SHAPE; Di not in {64, 128},
 * Hi not in [1, 64], cmp_ratio < 2, topk > 2048 -> CSA_ERR_UNSUPPORTED;
 * NULL inputs or outputs (k and d_k may be NULL only when Tc == 0) ->
 * CSA_ERR_NULL; q, k and d_k must be 16-byte aligned (else
 * CSA_ERR_UNSUPPORTED). total_tokens == 0 launches nothing.
 */
csa_status_t csa_indexer_kl_loss_grad(const csa_bf16_t *q, const csa_bf16_t *k, const float *w,
                                      const int32_t *sparse_indices,
                                      const float *attn_softmax_l1_norm, int32_t total_tokens,
                                      int32_t total_cmp, int32_t index_heads, int32_t index_dim,
                                      const int32_t *cu_seqlens_q,
                                      const int32_t *cu_seqlens_cmp_kv, int32_t batch,
                                      int32_t cmp_ratio, int32_t topk, float grad_scale,
                                      float *d_q, float *d_k, float *d_w, float *loss,
                                      csa_stream_t stream);

/*
 * THD compressor core: grouping, position embedding, overlap transform and
 * slot pooling of one DeepSeek-V4 compressor, producing the compressed rows
 * (cmp_kv, or the indexer's k) from the two projections of the packed rows.
 * [miles#2038] 关键源码片段 compressor.py (_forward_thd: per-sequence groups
 * of cmp_ratio rows, gather_idx, the len % cmp_ratio tail produces no row;
 * _overlap_transform_thd: [Tc, r, 2hd] -> [Tc, 2r, hd], the first r slots
 * from the previous group's first halves, a sequence's first group filled
 * with 0 for kv and -inf for the score). The page omits the rest; reading:
 * ape[i] is added to slot i's score before the overlap, and
 *     out[g, e] = sum_s softmax_s(score[g, s, e]) kv[g, s, e]
 * over the group's slots (r, or 2r with overlap). The linear projections
 * (linear_bf16_fp32 on the page) and any later normalisation or RoPE are the
 * caller's.
 * kv, score [T, Wd] fp32 (Wd = 2 * head_dim with overlap, head_dim without);
 * ape [cmp_ratio, Wd] fp32 or NULL (zero); cu_seqlens, cu_seqlens_cmp
 * [batch+1] int32 (the latter from csa_compress_cu_seqlens); out
 * [total_cmp, head_dim] fp32, overwritten.
 * Errors: negative sizes, head_dim < 1 or total_cmp * cmp_ratio >
 * total_tokens -> CSA_ERR_SHAPE; cmp_ratio < 1 or head_dim > 65536 ->
 * CSA_ERR_UNSUPPORTED; NULL kv/score/cu_seqlens/cu_seqlens_cmp/out ->
 * CSA_ERR_NULL. total_cmp == 0 launches nothing. A compressed row whose
 * group does not fit inside its sequence (inconsistent device offsets) is
 * written as 0 and recorded in the device error word.
 */
csa_status_t csa_compress_thd(const float *kv, const float *score, const float *ape,
                              const int32_t *cu_seqlens, const int32_t *cu_seqlens_cmp,
                              int32_t batch, int32_t total_tokens, int32_t total_cmp,
                              int32_t cmp_ratio, int32_t head_dim, int32_t overlap, float *out,
                              csa_stream_t stream);

/*
 * BSND layout (fixed-shape batch) of the forward path.
 * [hp#RFC] sections 1 and 2: the ops take a layout argument whose default is
 * "BSND" -- q [B, S, N, D], KV [B, S_kv, 1, D], compressed indices local to
 * their batch -- and seqused_q / seqused_kv declaring how many leading rows
 * of each batch are valid (rows past them are left unspecified). Here one
 * seqused array serves q and both KV streams (self-attention prefill: the
 * query rows are the KV rows), and the compressed stream of batch b holds
 * min(floor(seqused[b] / cmp_ratio), seqlen_cmp) valid rows.
 * The computation is exactly the THD one applied to each batch's valid rows
 * as one sequence: a valid row p of batch b sees the window rows
 * [max(0, p - ori_win_left), p] of its batch and the compressed rows j
 * (batch-local) with (j + 1) * cmp_ratio <= p + 1.
 * Implementation: batch b is rows [b S, (b+1) S) of the packed THD stream;
 * the call writes, in the caller's workspace, THD offsets with two sequences
 * per batch (valid rows, then padding rows) and the stream-absolute form of
 * the compressed indices, then runs the THD kernels. Outputs of padding rows
 * (p >= seqused[b]) are unspecified.
 * seqused [B] int32 (device) or NULL (every row valid); entries outside
 * [0, seqlen] are clamped and recorded in the device error word.
 *
 * csa_bsnd_mla_workspace_size: bytes of workspace csa_sparse_mla_fwd_bsnd
 * needs (topk = 0 when no index list is passed).
 * csa_sparse_mla_fwd_bsnd: as csa_sparse_mla_fwd, with q [B, S, H, D],
 *   ori_kv [B, S, D], cmp_kv [B, Sc, D] or NULL, cmp_sparse_indices
 *   [B, S, topk] batch-local rows (-1 or outside [0, Sc): skipped) or NULL
 *   (every visible compressed row), out [B, S, H, D], softmax_lse [B, S, H].
 *   workspace: at least csa_bsnd_mla_workspace_size(B, S, topk) bytes,
 *   256-byte aligned. Errors as csa_sparse_mla_fwd, plus B * S or B * Sc
 *   above INT32_MAX -> CSA_ERR_SHAPE and a short or misaligned workspace ->
 *   CSA_ERR_WORKSPACE. B * S == 0 launches nothing.
 * csa_bsnd_indexer_workspace_size / csa_indexer_topk_bsnd: as
 *   csa_indexer_topk with q [B, S, Hi, Di], k [B, Sc, Di], w [B, S, Hi];
 *   topk_idx [B, S, topk] receives batch-local rows (-1 padded), topk_val
 *   [B, S, topk] or NULL. The workspace also holds the indexer's own score
 *   spill. Errors as csa_indexer_topk, plus the shape and workspace checks
 *   above.
 */
size_t csa_bsnd_mla_workspace_size(int32_t batch, int32_t seqlen, int32_t topk);

csa_status_t csa_sparse_mla_fwd_bsnd(const csa_bf16_t *q, const csa_bf16_t *ori_kv,
                                     const csa_bf16_t *cmp_kv, const int32_t *cmp_sparse_indices,
                                     const int32_t *seqused, int32_t batch, int32_t seqlen,
                                     int32_t seqlen_cmp, int32_t heads, int32_t head_dim,
                                     int32_t topk, const float *sinks, float softmax_scale,
                                     int32_t cmp_ratio, int32_t ori_win_left,
                                     int32_t ori_win_right, csa_bf16_t *out, float *softmax_lse,
                                     int32_t return_softmax_lse, void *workspace,
                                     size_t workspace_bytes, csa_stream_t stream);

size_t csa_bsnd_indexer_workspace_size(int32_t batch, int32_t seqlen, int32_t seqlen_cmp,
                                       int32_t index_heads, int32_t index_dim, int32_t topk);

csa_status_t csa_indexer_topk_bsnd(const csa_bf16_t *q, const csa_bf16_t *k, const float *w,
                                   const int32_t *seqused, int32_t batch, int32_t seqlen,
                                   int32_t seqlen_cmp, int32_t index_heads, int32_t index_dim,
                                   int32_t cmp_ratio, int32_t topk, int32_t *topk_idx,
                                   float *topk_val, void *workspace, size_t workspace_bytes,
                                   csa_stream_t stream);

/*
 * csa_indexer_topk without a workspace, for callers that cannot allocate
 * device memory. The pages have no counterpart to this entry point.
 *
 * A token whose sequence offers more visible compressed rows than the
 * kernel keeps in shared memory spills its scores to device scratch, which
 * csa_indexer_topk takes from the caller. A plugin that a host framework
 * hands only its input and output buffers, or a runtime held to a memory
 * budget fixed at start-up, may be unable to call cudaMalloc (it can
 * synchronise the device and fragments a pool the caller does not own).
 * This variant computes exactly what csa_indexer_topk computes, with the
 * same arguments minus the workspace, and uses instead a scratch array of
 * 32 MiB that lives in the library: every GPU that loads the library holds
 * that array until the process exits. The call allocates nothing.
 *
 * Limits and sharing:
 *   - total_cmp above 2,097,152 rows (one CTA's slot, two buffers of two
 *     tokens' scores, no longer fits in the array) -> CSA_ERR_WORKSPACE; other
 *     errors as csa_indexer_topk.
 *   - When scores may spill, the grid is limited to as many CTAs as the
 *     array has slots of 4 x total_cmp floats.
 *   - Every call shares the array and leaves its contents behind; nothing in
 *     it needs to start at zero (each score is written before it is read).
 *     Calls that overlap on the GPU (e.g. on two streams at once) race on
 *     the array: order them on one stream.
 *   - The first call on a device looks up the array's device address (a
 *     one-time set-up with that device current); make that first call before
 *     any stream capture.
 */
csa_status_t csa_indexer_topk_noalloc(const csa_bf16_t *q, const csa_bf16_t *k, const float *w,
                                      int32_t total_tokens, int32_t total_cmp,
                                      int32_t index_heads, int32_t index_dim,
                                      const int32_t *cu_seqlens_q,
                                      const int32_t *cu_seqlens_cmp_kv, int32_t batch,
                                      int32_t cmp_ratio, int32_t topk, int32_t *topk_idx,
                                      float *topk_val, csa_stream_t stream);

/*
 * Synchronises `stream`, then returns and clears the device error word of the
 * current device: CSA_OK, CSA_ERR_DEVICE_CHECK or CSA_ERR_TIMEOUT.
 * `detail` (host pointer, may be NULL) receives the raw word (kernel id and
 * site in the high bits, 0 when clean).
 */
csa_status_t csa_device_error(csa_stream_t stream, int32_t *detail);

/*
 * Library control, no counterpart on the pages: the limit after which a wait
 * of the indexer and sparse-attention kernels on one of their own pipeline
 * barriers gives up (host value, nanoseconds; 0 restores the default of 2 s).
 * A wait that gives up records CSA_ERR_TIMEOUT in the device error word and
 * makes its CTA stop early: it lets its copies and tensor-core operations in
 * flight finish (those final waits keep the 2 s limit), frees its tensor
 * memory and exits, so that the launch ends and the context stays usable; the
 * outputs of such a launch are unspecified. A limit of a few microseconds
 * makes normal launches give up, which is how the timeout path is tested.
 * Applies to launches made after the call, from any host thread.
 *
 * The device addresses of the library's global arrays (the error word, the
 * no-allocation entry's scratch) are looked up once per device and CUDA
 * context and kept: after a device reset (cudaDeviceReset), the next call
 * makes them again for the new context.
 */
csa_status_t csa_set_wait_limit_ns(uint64_t limit_ns);

/*
 * Library control, no counterpart on the pages: the indexer selects each
 * token's top-k with two warps sharing 16-bit counts, and a token with more
 * visible rows than a bound (130,000) with one warp alone. `rows` lowers that
 * bound (0 restores it; values above it are ignored; negative ->
 * CSA_ERR_SHAPE), so that ordinary inputs run the one-warp path: the results
 * are the same either way, which is how that path is tested. Applies to
 * launches made after the call, from any host thread.
 */
csa_status_t csa_set_pair_select_rows(int32_t rows);

#ifdef __cplusplus
}
#endif

#endif /* CSA_GB300_H_ */
