// Integer layout steps of the CSA path: compressed cu_seqlens and
// segment-clamped sliding-window rows.
//
// Sources: miles PR 2038 report, key source excerpts (thd_utils.py
// get_window_topk_idxs_thd; compressor.py _forward_thd docstring: the
// trailing len % cmp_ratio tokens of a sequence form no compressed row).
#include "common.cuh"
#include "internal.h"

namespace csa {

namespace {

// cu_cmp[b+1] = cu_cmp[b] + floor((cu[b+1]-cu[b]) / r). One block walks the
// sequences in chunks of NT with a block scan and a running carry (NT = 128
// for the usual few sequences, 1024 beyond).
template <int NT>
__global__ void __launch_bounds__(NT)
compress_cu_seqlens_kernel(const int32_t *__restrict__ cu, int32_t batch, int32_t r,
                           int32_t *__restrict__ cu_cmp, int32_t *err) {
    __shared__ int32_t scratch[NT / 32 + 1];
    int32_t carry = 0;
    grid_dependency_wait();
    launch_dependents();
    if (threadIdx.x == 0) cu_cmp[0] = 0;
    for (int32_t base = 0; base < batch; base += NT) {
        const int32_t b = base + threadIdx.x;
        int32_t groups = 0;
        if (b < batch) {
            int32_t len = __ldg(cu + b + 1) - __ldg(cu + b);
            if (len < 0) {
                report_error(err, kErrCheck, kKerCompress, 1);
                len = 0;
            }
            groups = len / r;
        }
        int32_t total;
        int32_t before = block_exclusive_scan<NT>(groups, scratch, &total);
        if (b < batch) cu_cmp[b + 1] = carry + before + groups;
        carry += total;
    }
}

// Each warp writes one contiguous run of tokens: the sequence of its first
// token is found by a search, later ones by stepping the sequence forward, and
// the W entries of a row are written by the 32 lanes (16-byte stores when W is
// a multiple of 4 and the output is 16-byte aligned).
__global__ void __launch_bounds__(256)
window_idx_kernel(const int32_t *__restrict__ cu, int32_t batch, int32_t T, int32_t W,
                  bool vec4, int32_t *__restrict__ idx, int32_t *err) {
    const int lane = threadIdx.x & 31;
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    const int64_t w = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int64_t per = (T + warps - 1) / warps;
    const int64_t t0 = w * per, t1 = min((int64_t)T, t0 + per);
    grid_dependency_wait();
    launch_dependents();
    if (t0 >= t1) return;
    int32_t b = -1, seg0 = 0, seg1 = 0;
    for (int64_t t = t0; t < t1; ++t) {
        if (b < 0 || t >= seg1) {  // the next non-empty sequence holding t
            b = find_segment(cu, batch, (int32_t)t);
            if (b >= 0) {
                seg0 = __ldg(cu + b);
                seg1 = __ldg(cu + b + 1);
            }
        }
        int32_t start, last;
        if (b < 0) {
            if (lane == 0) report_error(err, kErrCheck, kKerWindow, 1);
            start = 1;
            last = 0;  // empty: every slot -1
        } else {
            start = max((int32_t)t - W + 1, seg0);
            last = (int32_t)t;
        }
        int32_t *row = idx + t * (int64_t)W;
        if (vec4) {
            for (int32_t i = lane * 4; i < W; i += 128) {
                int4 v;
                v.x = (start + i <= last) ? start + i : -1;
                v.y = (start + i + 1 <= last) ? start + i + 1 : -1;
                v.z = (start + i + 2 <= last) ? start + i + 2 : -1;
                v.w = (start + i + 3 <= last) ? start + i + 3 : -1;
                *reinterpret_cast<int4 *>(row + i) = v;
            }
        } else {
            for (int32_t i = lane; i < W; i += 32) row[i] = (start + i <= last) ? start + i : -1;
        }
    }
}

}  // namespace

cudaError_t launch_compress_cu_seqlens(const int32_t *cu, int32_t batch, int32_t cmp_ratio,
                                       int32_t *cu_cmp, int32_t *err, cudaStream_t stream) {
    if (batch <= 128)
        return launch_early(compress_cu_seqlens_kernel<128>, dim3(1), dim3(128), 0, stream, cu,
                            batch, cmp_ratio, cu_cmp, err);
    return launch_early(compress_cu_seqlens_kernel<1024>, dim3(1), dim3(1024), 0, stream, cu, batch,
                        cmp_ratio, cu_cmp, err);
}

cudaError_t launch_window_idx(const int32_t *cu, int32_t batch, int32_t total_tokens,
                              int32_t window, int32_t *idx, int32_t *err, cudaStream_t stream) {
    if (total_tokens == 0) return cudaSuccess;
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    // One 256-thread block per SM at most (runs of tokens per warp): the
    // blocks then fit beside a concurrent indexer or attention CTA.
    const int warps_per_block = 8;
    int64_t blocks = ((int64_t)total_tokens + 4 * warps_per_block - 1) / (4 * warps_per_block);
    if (blocks > (int64_t)sms) blocks = (int64_t)sms;
    const bool vec4 = (window & 3) == 0 && ((uintptr_t)idx & 15u) == 0;
    return launch_early(window_idx_kernel, dim3((unsigned)blocks), dim3(32 * warps_per_block), 0,
                        stream, cu, batch, total_tokens, window, vec4, idx, err);
}

}  // namespace csa
