// Backward of the shared-KV MLA sparse attention with sinks: the entry's
// launch sequence (sm_103a).
//
// The gradient call the miles PR 2038 report and the hyper-parallel RFC list
// as sparse_flash_mla_grad: from q, dout, the forward's output and
// log-sum-exp it returns d_query, d_ori_kv, d_cmp_kv, d_sinks and the
// head-averaged attention distributions ori/cmp_softmax_l1_norm. The outputs
// that are sums over tokens (the two KV-row gradients, d_sinks) and the
// compressed distribution (whose skipped entries stay zero) are zeroed here,
// then the tensor-core kernel (sparse_mla_bwd_tc.cu) runs.
#include "common.cuh"
#include "internal.h"

namespace csa {

namespace {

constexpr int kBwdMaxList = 1024;  // top-k entries kept per token
constexpr int kBwdMaxWin = 1024;   // window rows per token

__global__ void zero_f32_kernel(float *p, int64_t n) {
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x)
        p[i] = 0.0f;
}

}  // namespace

cudaError_t launch_sparse_mla_bwd(const MlaBwdArgs &a, cudaStream_t stream) {
    if (a.T == 0) return cudaSuccess;
    if (a.cmp_idx && a.topk > kBwdMaxList) return cudaErrorInvalidValue;
    if (a.window > kBwdMaxWin) return cudaErrorInvalidValue;
    const bool use_cmp = a.cmp_kv != nullptr && a.Tc > 0;
    // outputs that accumulate start at zero; the lists' unused slots stay zero
    auto zero = [&](float *p, int64_t n) -> cudaError_t {
        if (!p || n <= 0) return cudaSuccess;
        const int64_t blocks = (n + 255) / 256;
        zero_f32_kernel<<<(int)(blocks < 4096 ? blocks : 4096), 256, 0, stream>>>(p, n);
        return cudaGetLastError();
    };
    cudaError_t e;
    if ((e = zero(a.d_ori_kv, (int64_t)a.T * 512)) != cudaSuccess) return e;
    if (use_cmp && (e = zero(a.d_cmp_kv, (int64_t)a.Tc * 512)) != cudaSuccess) return e;
    if (a.sinks && (e = zero(a.d_sinks, a.H)) != cudaSuccess) return e;
    if (use_cmp && a.cmp_idx && (e = zero(a.cmp_l1, (int64_t)a.T * a.topk)) != cudaSuccess) return e;
    return launch_sparse_mla_bwd_tc(a, stream);
}

}  // namespace csa
