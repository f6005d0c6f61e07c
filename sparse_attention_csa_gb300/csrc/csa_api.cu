// C ABI of the CSA forward path: host-side argument checks and launches.
// The operations, their sources on the pages and the error behaviour are
// documented in include/csa.h.
#include <stdint.h>

#include <atomic>

#include "common.cuh"
#include "csa.h"
#include "internal.h"
#include "tmap.h"

namespace {

// Device error word (one per device that loads the library).
__device__ int32_t g_error_word = 0;

constexpr int kMaxDevices = 64;
int32_t *g_error_ptr[kMaxDevices] = {};
unsigned long long g_error_ctx[kMaxDevices] = {};  // context the address belongs to

// Device address of g_error_word on the current device: looked up with
// cudaGetSymbolAddress (the host-side way to name it) once per device and
// context, again after a device reset has made a new context.
int32_t *error_word(csa_status_t *st) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        *st = CSA_ERR_CUDA;
        return nullptr;
    }
    const unsigned long long ctx = csa::current_context_id();
    if (!g_error_ptr[dev] || ctx == 0 || ctx != g_error_ctx[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_error_word) != cudaSuccess) {
            *st = CSA_ERR_CUDA;
            return nullptr;
        }
        g_error_ptr[dev] = static_cast<int32_t *>(p);
        g_error_ctx[dev] = csa::current_context_id();
    }
    *st = CSA_OK;
    return g_error_ptr[dev];
}

csa_status_t from_cuda(cudaError_t e) { return e == cudaSuccess ? CSA_OK : CSA_ERR_CUDA; }

}  // namespace

namespace csa {
int32_t *device_error_word(csa_status_t *st) { return error_word(st); }

// 0: the default limit (2 s).
std::atomic<uint64_t> g_wait_limit_ns{0};

uint64_t pipeline_wait_limit_ns() {
    const uint64_t v = g_wait_limit_ns.load(std::memory_order_relaxed);
    return v ? v : 2000000000ull;
}

// 0: the default (the two-warp selection's own bound).
std::atomic<int32_t> g_pair_select_rows{0};

int32_t pair_select_max_rows(int32_t bound) {
    const int32_t v = g_pair_select_rows.load(std::memory_order_relaxed);
    return v > 0 && v < bound ? v : bound;
}
}  // namespace csa

extern "C" {

const char *csa_status_string(csa_status_t status) {
    switch (status) {
        case CSA_OK: return "CSA_OK";
        case CSA_ERR_NULL: return "CSA_ERR_NULL: a required pointer is NULL";
        case CSA_ERR_SHAPE: return "CSA_ERR_SHAPE: negative or inconsistent sizes";
        case CSA_ERR_UNSUPPORTED: return "CSA_ERR_UNSUPPORTED: request outside what this library implements";
        case CSA_ERR_WORKSPACE: return "CSA_ERR_WORKSPACE: workspace too small or misaligned";
        case CSA_ERR_CUDA: return "CSA_ERR_CUDA: a CUDA call or launch failed";
        case CSA_ERR_DEVICE_CHECK: return "CSA_ERR_DEVICE_CHECK: a kernel met inconsistent device data";
        case CSA_ERR_TIMEOUT: return "CSA_ERR_TIMEOUT: a bounded device-side wait gave up";
    }
    return "unknown csa_status_t";
}

csa_status_t csa_compress_cu_seqlens(const int32_t *cu_seqlens, int32_t batch, int32_t cmp_ratio,
                                     int32_t *cu_seqlens_cmp, csa_stream_t stream) {
    if (!cu_seqlens || !cu_seqlens_cmp) return CSA_ERR_NULL;
    if (batch < 0) return CSA_ERR_SHAPE;
    if (cmp_ratio < 1) return CSA_ERR_UNSUPPORTED;
    csa_status_t st;
    int32_t *err = error_word(&st);
    if (st != CSA_OK) return st;
    return from_cuda(csa::launch_compress_cu_seqlens(cu_seqlens, batch, cmp_ratio, cu_seqlens_cmp,
                                                     err, (cudaStream_t)stream));
}

csa_status_t csa_window_idx(const int32_t *cu_seqlens, int32_t batch, int32_t total_tokens,
                            int32_t ori_win_left, int32_t ori_win_right, int32_t *idx,
                            csa_stream_t stream) {
    if (!cu_seqlens || (!idx && total_tokens > 0)) return CSA_ERR_NULL;
    if (batch < 0 || total_tokens < 0 || ori_win_left < 0) return CSA_ERR_SHAPE;
    if (ori_win_right != 0) return CSA_ERR_UNSUPPORTED;
    if (total_tokens == 0) return CSA_OK;
    if (ori_win_left >= INT32_MAX - 1) return CSA_ERR_SHAPE;
    csa_status_t st;
    int32_t *err = error_word(&st);
    if (st != CSA_OK) return st;
    return from_cuda(csa::launch_window_idx(cu_seqlens, batch, total_tokens, ori_win_left + 1, idx,
                                            err, (cudaStream_t)stream));
}

size_t csa_indexer_topk_workspace_size(int32_t total_tokens, int32_t total_cmp, int32_t index_heads,
                                       int32_t index_dim, int32_t topk) {
    if (total_tokens < 0 || total_cmp < 0) return 0;
    return csa::indexer_workspace_bytes(total_tokens, total_cmp, index_heads, index_dim, topk);
}

csa_status_t csa_indexer_topk(const csa_bf16_t *q, const csa_bf16_t *k, const float *w,
                              int32_t total_tokens, int32_t total_cmp, int32_t index_heads,
                              int32_t index_dim, const int32_t *cu_seqlens_q,
                              const int32_t *cu_seqlens_cmp_kv, int32_t batch, int32_t cmp_ratio,
                              int32_t topk, int32_t *topk_idx, float *topk_val, void *workspace,
                              size_t workspace_bytes, csa_stream_t stream) {
    if (total_tokens < 0 || total_cmp < 0 || batch < 0 || topk < 1) return CSA_ERR_SHAPE;
    if (index_dim != 64 && index_dim != 128) return CSA_ERR_UNSUPPORTED;
    if (index_heads < 1 || index_heads > 64) return CSA_ERR_UNSUPPORTED;
    if (cmp_ratio < 2) return CSA_ERR_UNSUPPORTED;
    if (total_tokens == 0) return CSA_OK;  // nothing to do (empty buffers may be NULL)
    if (!q || !w || !cu_seqlens_q || !cu_seqlens_cmp_kv || !topk_idx) return CSA_ERR_NULL;
    if (total_cmp > 0 && !k) return CSA_ERR_NULL;
    const size_t need = csa::indexer_workspace_bytes(total_tokens, total_cmp, index_heads,
                                                     index_dim, topk);
    if (need > 0 && (!workspace || workspace_bytes < need || ((uintptr_t)workspace & 255u)))
        return CSA_ERR_WORKSPACE;
    // 16-byte vector loads of q / k rows
    if (((uintptr_t)q & 15u) || (k && ((uintptr_t)k & 15u))) return CSA_ERR_UNSUPPORTED;
    csa_status_t st;
    int32_t *err = error_word(&st);
    if (st != CSA_OK) return st;
    csa::IndexerArgs a;
    a.q = reinterpret_cast<const __nv_bfloat16 *>(q);
    a.k = reinterpret_cast<const __nv_bfloat16 *>(k);
    a.w = w;
    a.cu_q = cu_seqlens_q;
    a.cu_c = cu_seqlens_cmp_kv;
    a.topk_idx = topk_idx;
    a.topk_val = topk_val;
    a.scratch = need > 0 ? static_cast<float *>(workspace) : nullptr;
    a.err = err;
    a.T = total_tokens;
    a.Tc = total_cmp;
    a.Hi = index_heads;
    a.Di = index_dim;
    a.batch = batch;
    a.cmp_ratio = cmp_ratio;
    a.topk = topk;
    return from_cuda(csa::launch_indexer_topk(a, (cudaStream_t)stream));
}

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
                                float *cmp_softmax_l1_norm, csa_stream_t stream) {
    const bool use_cmp = cmp_kv != nullptr && total_cmp > 0;
    if (batch < 0 || total_tokens < 0 || total_cmp < 0 || heads < 1 || ori_win_left < 0)
        return CSA_ERR_SHAPE;
    if (total_tokens > 0) {  // empty buffers may be NULL
        if (!q || !dout || !out || !softmax_lse || !ori_kv || !cu_seqlens_q || !d_q || !d_ori_kv)
            return CSA_ERR_NULL;
        if (use_cmp && (!cu_seqlens_cmp_kv || !d_cmp_kv)) return CSA_ERR_NULL;
    }
    if (use_cmp && cmp_sparse_indices && topk < 1) return CSA_ERR_SHAPE;
    if (head_dim != 512) return CSA_ERR_UNSUPPORTED;
    if (heads > 64) return CSA_ERR_UNSUPPORTED;
    if (ori_win_right != 0 || ori_win_left > 1023) return CSA_ERR_UNSUPPORTED;
    if (use_cmp && cmp_ratio < 2) return CSA_ERR_UNSUPPORTED;
    if (use_cmp && cmp_sparse_indices && topk > 1024) return CSA_ERR_UNSUPPORTED;
    if (cu_seqlens_ori_kv && cu_seqlens_ori_kv != cu_seqlens_q) return CSA_ERR_UNSUPPORTED;
    if (((uintptr_t)q & 15u) || ((uintptr_t)dout & 15u) || ((uintptr_t)out & 3u) ||
        ((uintptr_t)ori_kv & 15u) || (use_cmp && ((uintptr_t)cmp_kv & 15u)))
        return CSA_ERR_UNSUPPORTED;
    if (((uintptr_t)d_ori_kv & 15u) || (use_cmp && ((uintptr_t)d_cmp_kv & 15u)))
        return CSA_ERR_UNSUPPORTED;  // the row gradients are added 16 bytes at a time
    if (total_tokens == 0) return CSA_OK;
    csa_status_t st;
    int32_t *err = error_word(&st);
    if (st != CSA_OK) return st;
    csa::MlaBwdArgs a;
    a.q = reinterpret_cast<const __nv_bfloat16 *>(q);
    a.dout = reinterpret_cast<const __nv_bfloat16 *>(dout);
    a.out = reinterpret_cast<const __nv_bfloat16 *>(out);
    a.lse = softmax_lse;
    a.ori_kv = reinterpret_cast<const __nv_bfloat16 *>(ori_kv);
    a.cmp_kv = use_cmp ? reinterpret_cast<const __nv_bfloat16 *>(cmp_kv) : nullptr;
    a.cmp_idx = use_cmp ? cmp_sparse_indices : nullptr;
    a.cu_q = cu_seqlens_q;
    a.cu_c = use_cmp ? cu_seqlens_cmp_kv : nullptr;
    a.sinks = sinks;
    a.d_q = d_q;
    a.d_ori_kv = d_ori_kv;
    a.d_cmp_kv = use_cmp ? d_cmp_kv : nullptr;
    a.d_sinks = sinks ? d_sinks : nullptr;
    a.ori_l1 = ori_softmax_l1_norm;
    a.cmp_l1 = use_cmp && cmp_sparse_indices ? cmp_softmax_l1_norm : nullptr;
    a.err = err;
    a.T = total_tokens;
    a.Tc = use_cmp ? total_cmp : 0;
    a.H = heads;
    a.batch = batch;
    a.topk = use_cmp && cmp_sparse_indices ? topk : 0;
    a.cmp_ratio = use_cmp ? cmp_ratio : 1;
    a.window = ori_win_left + 1;
    a.softmax_scale = softmax_scale;
    return from_cuda(csa::launch_sparse_mla_bwd(a, (cudaStream_t)stream));
}

csa_status_t csa_sparse_mla_fwd(const csa_bf16_t *q, const csa_bf16_t *ori_kv,
                                const csa_bf16_t *cmp_kv, const int32_t *cmp_sparse_indices,
                                const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_ori_kv,
                                const int32_t *cu_seqlens_cmp_kv, int32_t batch,
                                int32_t total_tokens, int32_t total_cmp, int32_t heads,
                                int32_t head_dim, int32_t topk, const float *sinks,
                                float softmax_scale, int32_t cmp_ratio, int32_t ori_win_left,
                                int32_t ori_win_right, csa_bf16_t *out, float *softmax_lse,
                                int32_t return_softmax_lse, csa_stream_t stream) {
    const bool use_cmp = cmp_kv != nullptr && total_cmp > 0;
    if (batch < 0 || total_tokens < 0 || total_cmp < 0 || heads < 1 || ori_win_left < 0)
        return CSA_ERR_SHAPE;
    if (total_tokens > 0) {  // empty buffers may be NULL
        if (!q || !ori_kv || !cu_seqlens_q || !out) return CSA_ERR_NULL;
        if (return_softmax_lse && !softmax_lse) return CSA_ERR_NULL;
        if (use_cmp && !cu_seqlens_cmp_kv) return CSA_ERR_NULL;
    }
    if (use_cmp && cmp_sparse_indices && topk < 1) return CSA_ERR_SHAPE;
    if (head_dim != 512) return CSA_ERR_UNSUPPORTED;
    if (heads > 64) return CSA_ERR_UNSUPPORTED;
    if (ori_win_right != 0 || ori_win_left > 1023) return CSA_ERR_UNSUPPORTED;
    if (use_cmp && cmp_ratio < 2) return CSA_ERR_UNSUPPORTED;
    if (use_cmp && cmp_sparse_indices && topk > csa::sparse_mla_max_topk())
        return CSA_ERR_UNSUPPORTED;
    if (cu_seqlens_ori_kv && cu_seqlens_ori_kv != cu_seqlens_q) return CSA_ERR_UNSUPPORTED;
    if (((uintptr_t)q & 15u) || ((uintptr_t)ori_kv & 15u) || ((uintptr_t)out & 15u) ||
        (use_cmp && ((uintptr_t)cmp_kv & 15u)))
        return CSA_ERR_UNSUPPORTED;
    if (total_tokens == 0) return CSA_OK;
    csa_status_t st;
    int32_t *err = error_word(&st);
    if (st != CSA_OK) return st;
    csa::MlaArgs a;
    a.q = reinterpret_cast<const __nv_bfloat16 *>(q);
    a.ori_kv = reinterpret_cast<const __nv_bfloat16 *>(ori_kv);
    a.cmp_kv = use_cmp ? reinterpret_cast<const __nv_bfloat16 *>(cmp_kv) : nullptr;
    a.cmp_idx = use_cmp ? cmp_sparse_indices : nullptr;
    a.cu_q = cu_seqlens_q;
    a.cu_c = use_cmp ? cu_seqlens_cmp_kv : nullptr;
    a.sinks = sinks;
    a.out = reinterpret_cast<__nv_bfloat16 *>(out);
    a.lse = return_softmax_lse ? softmax_lse : nullptr;
    a.err = err;
    a.T = total_tokens;
    a.Tc = use_cmp ? total_cmp : 0;
    a.H = heads;
    a.D = head_dim;
    a.batch = batch;
    a.topk = use_cmp && cmp_sparse_indices ? topk : 0;
    a.cmp_ratio = use_cmp ? cmp_ratio : 1;
    a.window = ori_win_left + 1;
    a.softmax_scale = softmax_scale;
    return from_cuda(csa::launch_sparse_mla_fwd(a, (cudaStream_t)stream));
}

csa_status_t csa_indexer_kl_loss_grad(const csa_bf16_t *q, const csa_bf16_t *k, const float *w,
                                      const int32_t *sparse_indices,
                                      const float *attn_softmax_l1_norm, int32_t total_tokens,
                                      int32_t total_cmp, int32_t index_heads, int32_t index_dim,
                                      const int32_t *cu_seqlens_q,
                                      const int32_t *cu_seqlens_cmp_kv, int32_t batch,
                                      int32_t cmp_ratio, int32_t topk, float grad_scale,
                                      float *d_q, float *d_k, float *d_w, float *loss,
                                      csa_stream_t stream) {
    if (total_tokens < 0 || total_cmp < 0 || batch < 0 || topk < 1) return CSA_ERR_SHAPE;
    if (index_dim != 64 && index_dim != 128) return CSA_ERR_UNSUPPORTED;
    if (index_heads < 1 || index_heads > 64) return CSA_ERR_UNSUPPORTED;
    if (cmp_ratio < 2) return CSA_ERR_UNSUPPORTED;
    if (topk > csa::indexer_kl_max_topk()) return CSA_ERR_UNSUPPORTED;
    if (total_tokens == 0) return CSA_OK;  // nothing to do (empty buffers may be NULL)
    if (!q || !w || !sparse_indices || !attn_softmax_l1_norm || !cu_seqlens_q ||
        !cu_seqlens_cmp_kv || !d_q || !d_w)
        return CSA_ERR_NULL;
    if (total_cmp > 0 && (!k || !d_k)) return CSA_ERR_NULL;
    // 16-byte loads of q / k rows and 16-byte atomic adds into d_k
    if (((uintptr_t)q & 15u) || (k && ((uintptr_t)k & 15u)) || (d_k && ((uintptr_t)d_k & 15u)))
        return CSA_ERR_UNSUPPORTED;
    csa_status_t st;
    int32_t *err = error_word(&st);
    if (st != CSA_OK) return st;
    csa::IndexerKlArgs a;
    a.q = reinterpret_cast<const __nv_bfloat16 *>(q);
    a.k = total_cmp > 0 ? reinterpret_cast<const __nv_bfloat16 *>(k) : nullptr;
    a.w = w;
    a.idx = sparse_indices;
    a.l1 = attn_softmax_l1_norm;
    a.cu_q = cu_seqlens_q;
    a.cu_c = cu_seqlens_cmp_kv;
    a.d_q = d_q;
    a.d_k = total_cmp > 0 ? d_k : nullptr;
    a.d_w = d_w;
    a.loss = loss;
    a.err = err;
    a.T = total_tokens;
    a.Tc = total_cmp;
    a.Hi = index_heads;
    a.Di = index_dim;
    a.batch = batch;
    a.cmp_ratio = cmp_ratio;
    a.topk = topk;
    a.grad_scale = grad_scale;
    return from_cuda(csa::launch_indexer_kl_grad(a, (cudaStream_t)stream));
}

csa_status_t csa_compress_thd(const float *kv, const float *score, const float *ape,
                              const int32_t *cu_seqlens, const int32_t *cu_seqlens_cmp,
                              int32_t batch, int32_t total_tokens, int32_t total_cmp,
                              int32_t cmp_ratio, int32_t head_dim, int32_t overlap, float *out,
                              csa_stream_t stream) {
    if (batch < 0 || total_tokens < 0 || total_cmp < 0 || head_dim < 1) return CSA_ERR_SHAPE;
    if ((int64_t)total_cmp * cmp_ratio > total_tokens) return CSA_ERR_SHAPE;
    if (cmp_ratio < 1 || head_dim > 65536) return CSA_ERR_UNSUPPORTED;
    if (total_cmp == 0) return CSA_OK;  // nothing to pool (empty buffers may be NULL)
    if (!kv || !score || !cu_seqlens || !cu_seqlens_cmp || !out) return CSA_ERR_NULL;
    csa_status_t st;
    int32_t *err = error_word(&st);
    if (st != CSA_OK) return st;
    csa::CompressArgs a;
    a.kv = kv;
    a.score = score;
    a.ape = ape;
    a.cu_q = cu_seqlens;
    a.cu_c = cu_seqlens_cmp;
    a.out = out;
    a.err = err;
    a.T = total_tokens;
    a.Tc = total_cmp;
    a.batch = batch;
    a.r = cmp_ratio;
    a.hd = head_dim;
    a.overlap = overlap ? 1 : 0;
    return from_cuda(csa::launch_compress_thd(a, (cudaStream_t)stream));
}

csa_status_t csa_set_wait_limit_ns(uint64_t limit_ns) {
    csa::g_wait_limit_ns.store(limit_ns, std::memory_order_relaxed);
    return CSA_OK;
}

csa_status_t csa_set_pair_select_rows(int32_t rows) {
    if (rows < 0) return CSA_ERR_SHAPE;
    csa::g_pair_select_rows.store(rows, std::memory_order_relaxed);
    return CSA_OK;
}

csa_status_t csa_device_error(csa_stream_t stream, int32_t *detail) {
    csa_status_t st;
    int32_t *err = error_word(&st);
    if (st != CSA_OK) return st;
    if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return CSA_ERR_CUDA;
    int32_t word = 0;
    if (cudaMemcpy(&word, err, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess)
        return CSA_ERR_CUDA;
    if (word != 0) {
        const int32_t zero = 0;
        if (cudaMemcpy(err, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess)
            return CSA_ERR_CUDA;
    }
    if (detail) *detail = word;
    if (word == 0) return CSA_OK;
    return ((word >> 24) == csa::kErrTimeout) ? CSA_ERR_TIMEOUT : CSA_ERR_DEVICE_CHECK;
}

}  // extern "C"
