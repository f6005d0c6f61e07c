// BSND layout (fixed-shape batch) for the forward path, mapped onto the THD
// kernels (sm_103a).
//
// The hyper-parallel RFC (sections 1 and 2) gives every op a layout argument
// whose default is "BSND": q [B, S, N, D], the KV streams [B, S_kv, 1, D],
// compressed indices batch-local, and seqused_q / seqused_kv declaring how
// many leading rows of each batch are valid (the rows past them are left
// unspecified). Packed back to back, batch b of a BSND tensor is rows
// [b S, (b+1) S) of a THD tensor, so the THD kernels run the BSND layout as
// is once three things are set up in the caller's workspace:
//   - cu_seqlens with two segments per batch: the valid rows
//     [b S, b S + used_b) and the padding rows [b S + used_b, (b+1) S);
//   - compressed cu_seqlens the same way over the compressed stream
//     [B, Sc, D]: [b Sc, b Sc + min(floor(used_b / r), Sc)) and the rest;
//   - batch-local compressed indices turned into stream-absolute rows
//     (b Sc + j for 0 <= j < Sc, else -1).
// A valid token then sees exactly its own batch's window and complete
// blocks; padding rows form segments of their own (their outputs are
// unspecified, as on the pages).
#include "common.cuh"
#include "internal.h"

namespace csa {

namespace {

constexpr size_t kAlign = 256;

size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

struct BsndWs {
    int32_t *cu = nullptr;   // [2B + 1]
    int32_t *cuc = nullptr;  // [2B + 1]
    int32_t *idx = nullptr;  // [B S, topk] or nullptr
    void *rest = nullptr;    // what follows (the indexer's own workspace)
    size_t rest_bytes = 0;
};

size_t layout_bytes(int32_t B) { return 2 * align_up(sizeof(int32_t) * (2 * (size_t)B + 1)); }

BsndWs carve(void *ws, size_t bytes, int32_t B, int64_t idx_elems) {
    BsndWs w;
    char *p = static_cast<char *>(ws);
    const size_t cu_b = align_up(sizeof(int32_t) * (2 * (size_t)B + 1));
    w.cu = reinterpret_cast<int32_t *>(p);
    w.cuc = reinterpret_cast<int32_t *>(p + cu_b);
    size_t used = 2 * cu_b;
    if (idx_elems > 0) {
        w.idx = reinterpret_cast<int32_t *>(p + used);
        used += align_up(sizeof(int32_t) * (size_t)idx_elems);
    }
    w.rest = p + used;
    w.rest_bytes = bytes > used ? bytes - used : 0;
    return w;
}

// One block: the two-segments-per-batch offsets. seqused entries outside
// [0, S] are clamped and recorded in the device error word.
__global__ void bsnd_offsets_kernel(const int32_t *__restrict__ seqused, int32_t B, int32_t S,
                                    int32_t Sc, int32_t r, int32_t *cu, int32_t *cuc,
                                    int32_t *err) {
    for (int32_t b = threadIdx.x; b < B; b += blockDim.x) {
        int32_t used = seqused ? __ldg(seqused + b) : S;
        if (used < 0 || used > S) {
            report_error(err, kErrCheck, kKerBsnd, 1);
            used = used < 0 ? 0 : S;
        }
        const int32_t c = min(used / r, Sc);
        cu[2 * b] = b * S;
        cu[2 * b + 1] = b * S + used;
        cuc[2 * b] = b * Sc;
        cuc[2 * b + 1] = b * Sc + c;
    }
    if (threadIdx.x == 0) {
        cu[2 * B] = B * S;
        cuc[2 * B] = B * Sc;
    }
}

// Batch-local compressed rows -> stream-absolute rows (-1 stays -1, and so
// does anything outside [0, Sc)).
__global__ void bsnd_idx_to_abs_kernel(const int32_t *__restrict__ local, int64_t n,
                                       int64_t per_batch, int32_t Sc, int32_t *abs_idx) {
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int32_t j = __ldg(local + i);
        const int64_t b = i / per_batch;
        abs_idx[i] = (j >= 0 && j < Sc) ? (int32_t)(b * Sc + j) : -1;
    }
}

// Stream-absolute rows -> batch-local rows, in place (-1 stays -1).
__global__ void bsnd_idx_to_local_kernel(int32_t *idx, int64_t n, int64_t per_batch,
                                         int32_t Sc) {
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int32_t j = idx[i];
        if (j >= 0) idx[i] = (int32_t)(j - (i / per_batch) * Sc);
    }
}

int grid_for(int64_t n) {
    const int64_t blocks = (n + 255) / 256;
    return (int)(blocks < 4096 ? (blocks > 0 ? blocks : 1) : 4096);
}

csa_status_t from_cuda(cudaError_t e) { return e == cudaSuccess ? CSA_OK : CSA_ERR_CUDA; }

}  // namespace

}  // namespace csa

extern "C" {

size_t csa_bsnd_mla_workspace_size(int32_t batch, int32_t seqlen, int32_t topk) {
    if (batch < 0 || seqlen < 0 || topk < 0) return 0;
    size_t n = csa::layout_bytes(batch);
    if (topk > 0) n += csa::align_up(sizeof(int32_t) * (size_t)batch * (size_t)seqlen * (size_t)topk);
    return n;
}

csa_status_t csa_sparse_mla_fwd_bsnd(const csa_bf16_t *q, const csa_bf16_t *ori_kv,
                                     const csa_bf16_t *cmp_kv, const int32_t *cmp_sparse_indices,
                                     const int32_t *seqused, int32_t batch, int32_t seqlen,
                                     int32_t seqlen_cmp, int32_t heads, int32_t head_dim,
                                     int32_t topk, const float *sinks, float softmax_scale,
                                     int32_t cmp_ratio, int32_t ori_win_left,
                                     int32_t ori_win_right, csa_bf16_t *out, float *softmax_lse,
                                     int32_t return_softmax_lse, void *workspace,
                                     size_t workspace_bytes, csa_stream_t stream) {
    const bool use_cmp = cmp_kv != nullptr && seqlen_cmp > 0;
    if (batch < 0 || seqlen < 0 || seqlen_cmp < 0 || heads < 1 || ori_win_left < 0)
        return CSA_ERR_SHAPE;
    if ((int64_t)batch * seqlen > INT32_MAX || (int64_t)batch * seqlen_cmp > INT32_MAX)
        return CSA_ERR_SHAPE;
    const int32_t T = batch * seqlen, Tc = use_cmp ? batch * seqlen_cmp : 0;
    const int32_t *list = use_cmp ? cmp_sparse_indices : nullptr;
    if (T > 0) {
        if (!q || !ori_kv || !out) return CSA_ERR_NULL;
        if (return_softmax_lse && !softmax_lse) return CSA_ERR_NULL;
    }
    if (list && topk < 1) return CSA_ERR_SHAPE;
    if (head_dim != 512) return CSA_ERR_UNSUPPORTED;
    if (heads > 64) return CSA_ERR_UNSUPPORTED;
    if (ori_win_right != 0 || ori_win_left > 1023) return CSA_ERR_UNSUPPORTED;
    if (use_cmp && cmp_ratio < 2) return CSA_ERR_UNSUPPORTED;
    if (list && topk > csa::sparse_mla_max_topk()) return CSA_ERR_UNSUPPORTED;
    if (((uintptr_t)q & 15u) || ((uintptr_t)ori_kv & 15u) || ((uintptr_t)out & 15u) ||
        (use_cmp && ((uintptr_t)cmp_kv & 15u)))
        return CSA_ERR_UNSUPPORTED;
    if (T == 0) return CSA_OK;
    const size_t need = csa_bsnd_mla_workspace_size(batch, seqlen, list ? topk : 0);
    if (!workspace || workspace_bytes < need || ((uintptr_t)workspace & 255u))
        return CSA_ERR_WORKSPACE;
    csa_status_t st;
    int32_t *err = csa::device_error_word(&st);
    if (st != CSA_OK) return st;
    cudaStream_t s = (cudaStream_t)stream;
    const int64_t n_idx = list ? (int64_t)T * topk : 0;
    csa::BsndWs w = csa::carve(workspace, workspace_bytes, batch, n_idx);
    csa::bsnd_offsets_kernel<<<1, 256, 0, s>>>(seqused, batch, seqlen, use_cmp ? seqlen_cmp : 0,
                                               use_cmp ? cmp_ratio : 1, w.cu, w.cuc, err);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return CSA_ERR_CUDA;
    if (list) {
        csa::bsnd_idx_to_abs_kernel<<<csa::grid_for(n_idx), 256, 0, s>>>(
            list, n_idx, (int64_t)seqlen * topk, seqlen_cmp, w.idx);
        if ((e = cudaGetLastError()) != cudaSuccess) return CSA_ERR_CUDA;
    }
    csa::MlaArgs a;
    a.q = reinterpret_cast<const __nv_bfloat16 *>(q);
    a.ori_kv = reinterpret_cast<const __nv_bfloat16 *>(ori_kv);
    a.cmp_kv = use_cmp ? reinterpret_cast<const __nv_bfloat16 *>(cmp_kv) : nullptr;
    a.cmp_idx = list ? w.idx : nullptr;
    a.cu_q = w.cu;
    a.cu_c = use_cmp ? w.cuc : nullptr;
    a.sinks = sinks;
    a.out = reinterpret_cast<__nv_bfloat16 *>(out);
    a.lse = return_softmax_lse ? softmax_lse : nullptr;
    a.err = err;
    a.T = T;
    a.Tc = Tc;
    a.H = heads;
    a.D = head_dim;
    a.batch = 2 * batch;
    a.topk = list ? topk : 0;
    a.cmp_ratio = use_cmp ? cmp_ratio : 1;
    a.window = ori_win_left + 1;
    a.softmax_scale = softmax_scale;
    return csa::from_cuda(csa::launch_sparse_mla_fwd(a, s));
}

size_t csa_bsnd_indexer_workspace_size(int32_t batch, int32_t seqlen, int32_t seqlen_cmp,
                                       int32_t index_heads, int32_t index_dim, int32_t topk) {
    if (batch < 0 || seqlen < 0 || seqlen_cmp < 0) return 0;
    if ((int64_t)batch * seqlen > INT32_MAX || (int64_t)batch * seqlen_cmp > INT32_MAX) return 0;
    return csa::layout_bytes(batch) +
           csa::align_up(csa::indexer_workspace_bytes(batch * seqlen, batch * seqlen_cmp,
                                                      index_heads, index_dim, topk));
}

csa_status_t csa_indexer_topk_bsnd(const csa_bf16_t *q, const csa_bf16_t *k, const float *w,
                                   const int32_t *seqused, int32_t batch, int32_t seqlen,
                                   int32_t seqlen_cmp, int32_t index_heads, int32_t index_dim,
                                   int32_t cmp_ratio, int32_t topk, int32_t *topk_idx,
                                   float *topk_val, void *workspace, size_t workspace_bytes,
                                   csa_stream_t stream) {
    if (batch < 0 || seqlen < 0 || seqlen_cmp < 0 || topk < 1) return CSA_ERR_SHAPE;
    if ((int64_t)batch * seqlen > INT32_MAX || (int64_t)batch * seqlen_cmp > INT32_MAX)
        return CSA_ERR_SHAPE;
    if (index_dim != 64 && index_dim != 128) return CSA_ERR_UNSUPPORTED;
    if (index_heads < 1 || index_heads > 64) return CSA_ERR_UNSUPPORTED;
    if (cmp_ratio < 2) return CSA_ERR_UNSUPPORTED;
    const int32_t T = batch * seqlen, Tc = batch * seqlen_cmp;
    if (T == 0) return CSA_OK;
    if (!q || !w || !topk_idx) return CSA_ERR_NULL;
    if (Tc > 0 && !k) return CSA_ERR_NULL;
    if (((uintptr_t)q & 15u) || (k && ((uintptr_t)k & 15u))) return CSA_ERR_UNSUPPORTED;
    const size_t need = csa_bsnd_indexer_workspace_size(batch, seqlen, seqlen_cmp, index_heads,
                                                        index_dim, topk);
    if (!workspace || workspace_bytes < need || ((uintptr_t)workspace & 255u))
        return CSA_ERR_WORKSPACE;
    csa_status_t st;
    int32_t *err = csa::device_error_word(&st);
    if (st != CSA_OK) return st;
    cudaStream_t s = (cudaStream_t)stream;
    csa::BsndWs ws = csa::carve(workspace, workspace_bytes, batch, 0);
    csa::bsnd_offsets_kernel<<<1, 256, 0, s>>>(seqused, batch, seqlen, seqlen_cmp, cmp_ratio,
                                               ws.cu, ws.cuc, err);
    if (cudaGetLastError() != cudaSuccess) return CSA_ERR_CUDA;
    csa::IndexerArgs a;
    a.q = reinterpret_cast<const __nv_bfloat16 *>(q);
    a.k = Tc > 0 ? reinterpret_cast<const __nv_bfloat16 *>(k) : nullptr;
    a.w = w;
    a.cu_q = ws.cu;
    a.cu_c = ws.cuc;
    a.topk_idx = topk_idx;
    a.topk_val = topk_val;
    const size_t spill = csa::indexer_workspace_bytes(T, Tc, index_heads, index_dim, topk);
    a.scratch = spill > 0 ? static_cast<float *>(ws.rest) : nullptr;
    a.err = err;
    a.T = T;
    a.Tc = Tc;
    a.Hi = index_heads;
    a.Di = index_dim;
    a.batch = 2 * batch;
    a.cmp_ratio = cmp_ratio;
    a.topk = topk;
    cudaError_t e = csa::launch_indexer_topk(a, s);
    if (e != cudaSuccess) return CSA_ERR_CUDA;
    const int64_t n = (int64_t)T * topk;
    csa::bsnd_idx_to_local_kernel<<<csa::grid_for(n), 256, 0, s>>>(topk_idx, n,
                                                                     (int64_t)seqlen * topk,
                                                                     seqlen_cmp);
    return csa::from_cuda(cudaGetLastError());
}

}  // extern "C"
