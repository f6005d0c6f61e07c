// csa_indexer_topk_noalloc: the indexer + top-k for callers that cannot
// allocate device memory. The pages have no counterpart to this entry point.
//
// csa_indexer_topk keeps a token's scores in shared memory, but a token whose
// sequence offers more visible compressed rows than fit there keeps them in a
// device scratch buffer, which that entry point takes from the caller as a
// workspace. Some callers cannot provide one: a plugin that is handed only
// its input and output buffers by a host framework, or a runtime that must
// stay inside a memory budget fixed at start-up, may not call cudaMalloc
// (which can synchronise the device and fragments a pool that someone else
// manages). This entry point takes the same inputs and outputs and uses a
// scratch array of fixed size that lives in the library itself.
#include <stdint.h>

#include "common.cuh"
#include "csa.h"
#include "internal.h"
#include "tmap.h"

namespace {

// 32 MiB of score scratch. Every GPU that loads the library holds one copy
// until the process exits.
constexpr size_t kScratchBytes = size_t(32) << 20;
constexpr int64_t kScratchFloats = int64_t(kScratchBytes / sizeof(float));
static __device__ __align__(256) float g_indexer_scratch[kScratchFloats];

constexpr int kMaxDevices = 64;
float *g_scratch_addr[kMaxDevices] = {};
unsigned long long g_scratch_ctx[kMaxDevices] = {};  // context the address belongs to

// Device address of g_indexer_scratch on the current device. In host code the
// array's name is only a host-side stand-in, so it is looked up with
// cudaGetSymbolAddress (with that device current) once per device and
// context, again after a device reset has made a new context.
csa_status_t scratch_address(float **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return CSA_ERR_CUDA;
    const unsigned long long ctx = csa::current_context_id();
    if (!g_scratch_addr[dev] || ctx == 0 || ctx != g_scratch_ctx[dev]) {
        float *p = nullptr;
        if (cudaGetSymbolAddress((void **)&p, g_indexer_scratch) != cudaSuccess || !p)
            return CSA_ERR_CUDA;
        g_scratch_addr[dev] = p;
        g_scratch_ctx[dev] = csa::current_context_id();
    }
    *out = g_scratch_addr[dev];
    return CSA_OK;
}

}  // namespace

extern "C" csa_status_t csa_indexer_topk_noalloc(
    const csa_bf16_t *q, const csa_bf16_t *k, const float *w, int32_t total_tokens,
    int32_t total_cmp, int32_t index_heads, int32_t index_dim, const int32_t *cu_seqlens_q,
    const int32_t *cu_seqlens_cmp_kv, int32_t batch, int32_t cmp_ratio, int32_t topk,
    int32_t *topk_idx, float *topk_val, csa_stream_t stream) {
    if (total_tokens < 0 || total_cmp < 0 || batch < 0 || topk < 1) return CSA_ERR_SHAPE;
    if (index_dim != 64 && index_dim != 128) return CSA_ERR_UNSUPPORTED;
    if (index_heads < 1 || index_heads > 64) return CSA_ERR_UNSUPPORTED;
    if (cmp_ratio < 2) return CSA_ERR_UNSUPPORTED;
    // One CTA's slot (the scores of a group of tokens) must fit in the array.
    if (csa::indexer_scratch_floats_per_cta(total_cmp) > kScratchFloats) return CSA_ERR_WORKSPACE;
    if (total_tokens == 0) return CSA_OK;
    if (!q || !w || !cu_seqlens_q || !cu_seqlens_cmp_kv || !topk_idx) return CSA_ERR_NULL;
    if (total_cmp > 0 && !k) return CSA_ERR_NULL;
    if (((uintptr_t)q & 15u) || (k && ((uintptr_t)k & 15u))) return CSA_ERR_UNSUPPORTED;
    csa_status_t st;
    int32_t *err = csa::device_error_word(&st);
    if (st != CSA_OK) return st;
    csa::IndexerArgs a;
    a.q = reinterpret_cast<const __nv_bfloat16 *>(q);
    a.k = reinterpret_cast<const __nv_bfloat16 *>(k);
    a.w = w;
    a.cu_q = cu_seqlens_q;
    a.cu_c = cu_seqlens_cmp_kv;
    a.topk_idx = topk_idx;
    a.topk_val = topk_val;
    a.scratch = nullptr;
    a.err = err;
    a.T = total_tokens;
    a.Tc = total_cmp;
    a.Hi = index_heads;
    a.Di = index_dim;
    a.batch = batch;
    a.cmp_ratio = cmp_ratio;
    a.topk = topk;
    if (total_cmp > csa::indexer_scratch_rows_threshold()) {
        // Scores may spill: every CTA gets its own slot, so the grid is
        // bounded by how many slots the array holds. Nothing in the slots
        // needs clearing: each score is written before it is read.
        st = scratch_address(&a.scratch);
        if (st != CSA_OK) return st;
        a.max_ctas = (int32_t)(kScratchFloats / csa::indexer_scratch_floats_per_cta(total_cmp));
    }
    return csa::launch_indexer_topk(a, (cudaStream_t)stream) == cudaSuccess ? CSA_OK : CSA_ERR_CUDA;
}
