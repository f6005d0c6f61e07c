// Internal launchers behind the C ABI. Arguments are already validated by
// csa_api.cu; every launcher returns the cudaError_t of its launch.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "csa.h"

namespace csa {

cudaError_t launch_compress_cu_seqlens(const int32_t *cu, int32_t batch, int32_t cmp_ratio,
                                       int32_t *cu_cmp, int32_t *err, cudaStream_t stream);

cudaError_t launch_window_idx(const int32_t *cu, int32_t batch, int32_t total_tokens,
                              int32_t window, int32_t *idx, int32_t *err, cudaStream_t stream);

struct IndexerArgs {
    const __nv_bfloat16 *q;  // [T, Hi, Di]
    const __nv_bfloat16 *k;  // [Tc, Di]
    const float *w;          // [T, Hi]
    const int32_t *cu_q;     // [batch+1]
    const int32_t *cu_c;     // [batch+1]
    int32_t *topk_idx;       // [T, topk]
    float *topk_val;         // [T, topk] or nullptr
    float *scratch;          // global score scratch (see indexer_workspace_bytes) or nullptr
    int32_t *err;
    int32_t T, Tc, Hi, Di, batch, cmp_ratio, topk;
    int32_t max_ctas = 0;    // grid bound when > 0 (scratch sized for that many CTAs)
    uint64_t wait_ns = 2000000000ull;  // limit of a pipeline wait (drains keep 2 s)
    int32_t pair_max = 130000;         // rows above this are selected by one warp
};

size_t indexer_workspace_bytes(int32_t T, int32_t Tc, int32_t Hi, int32_t Di, int32_t topk);
// A token whose sequence offers more visible compressed rows than this keeps
// its scores in the scratch (one slot of Tc floats per CTA) instead of
// shared memory.
int32_t indexer_scratch_rows_threshold();
// Floats of scratch one CTA uses when scores spill (its slot).
int64_t indexer_scratch_floats_per_cta(int32_t Tc);
cudaError_t launch_indexer_topk(const IndexerArgs &a, cudaStream_t stream);

struct MlaArgs {
    const __nv_bfloat16 *q;       // [T, H, D]
    const __nv_bfloat16 *ori_kv;  // [T, D]
    const __nv_bfloat16 *cmp_kv;  // [Tc, D] or nullptr (window only)
    const int32_t *cmp_idx;       // [T, topk] or nullptr (all visible)
    const int32_t *cu_q;          // [batch+1]
    const int32_t *cu_c;          // [batch+1] (required when cmp_kv is used)
    const float *sinks;           // [H] or nullptr
    __nv_bfloat16 *out;           // [T, H, D]
    float *lse;                   // [T, H] or nullptr
    int32_t *err;
    int32_t T, Tc, H, D, batch, topk, cmp_ratio, window;
    float softmax_scale;
    uint32_t epoch = 0;      // set by the launcher: token-claim epoch and slot
    int32_t claim_slot = 0;
    uint64_t wait_ns = 2000000000ull;  // limit of a pipeline wait (drains keep 2 s)
};

cudaError_t launch_sparse_mla_fwd(const MlaArgs &a, cudaStream_t stream);

struct MlaBwdArgs {
    const __nv_bfloat16 *q;       // [T, H, 512]
    const __nv_bfloat16 *dout;    // [T, H, 512]
    const __nv_bfloat16 *out;     // [T, H, 512], the forward's output
    const float *lse;             // [T, H], the forward's log-sum-exp
    const __nv_bfloat16 *ori_kv;  // [T, 512]
    const __nv_bfloat16 *cmp_kv;  // [Tc, 512] or nullptr
    const int32_t *cmp_idx;       // [T, topk] or nullptr (all visible)
    const int32_t *cu_q;          // [batch+1]
    const int32_t *cu_c;          // [batch+1] (required when cmp_kv is used)
    const float *sinks;           // [H] or nullptr
    float *d_q;                   // [T, H, 512]
    float *d_ori_kv;              // [T, 512]
    float *d_cmp_kv;              // [Tc, 512] (when cmp_kv is used)
    float *d_sinks;               // [H] or nullptr
    float *ori_l1;                // [T, window] or nullptr
    float *cmp_l1;                // [T, topk] or nullptr
    int32_t *err;
    int32_t T, Tc, H, batch, topk, cmp_ratio, window;
    float softmax_scale;
};

cudaError_t launch_sparse_mla_bwd(const MlaBwdArgs &a, cudaStream_t stream);
// The tensor-core kernel alone (outputs already zeroed where they accumulate).
cudaError_t launch_sparse_mla_bwd_tc(const MlaBwdArgs &a, cudaStream_t stream);
// Largest topk (entries of cmp_sparse_indices per token) the kernel accepts.
int32_t sparse_mla_max_topk();

struct IndexerKlArgs {
    const __nv_bfloat16 *q;  // [T, Hi, Di]
    const __nv_bfloat16 *k;  // [Tc, Di] (nullptr when Tc == 0)
    const float *w;          // [T, Hi]
    const int32_t *idx;      // [T, topk] sparse_indices
    const float *l1;         // [T, topk] attn_softmax_l1_norm
    const int32_t *cu_q;     // [batch+1]
    const int32_t *cu_c;     // [batch+1]
    float *d_q;              // [T, Hi, Di]
    float *d_k;              // [Tc, Di]
    float *d_w;              // [T, Hi]
    float *loss;             // [T] or nullptr
    int32_t *err;
    int32_t T, Tc, Hi, Di, batch, cmp_ratio, topk;
    float grad_scale;
};

cudaError_t launch_indexer_kl_grad(const IndexerKlArgs &a, cudaStream_t stream);
// The tensor-core form (index_dim 128, Hi <= 64); d_k already zeroed.
cudaError_t launch_indexer_kl_grad_tc(const IndexerKlArgs &a, cudaStream_t stream);
// Largest topk (entries of sparse_indices per token) the kernel accepts.
int32_t indexer_kl_max_topk();

struct CompressArgs {
    const float *kv;      // [T, wd] (wd = 2 hd with overlap, hd without)
    const float *score;   // [T, wd]
    const float *ape;     // [r, wd] or nullptr
    const int32_t *cu_q;  // [batch+1]
    const int32_t *cu_c;  // [batch+1]
    float *out;           // [Tc, hd]
    int32_t *err;
    int32_t T, Tc, batch, r, hd, overlap;
};

cudaError_t launch_compress_thd(const CompressArgs &a, cudaStream_t stream);

// Device error word of the current device (csa_api.cu).
int32_t *device_error_word(csa_status_t *st);

// Limit of the forward kernels' pipeline waits (csa_set_wait_limit_ns).
uint64_t pipeline_wait_limit_ns();
// Largest row the indexer's two-warp selection takes (csa_set_pair_select_rows),
// at most `bound`.
int32_t pair_select_max_rows(int32_t bound);

}  // namespace csa
