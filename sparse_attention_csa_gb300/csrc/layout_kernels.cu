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

constexpr int kScanThreads = 1024;

// cu_cmp[b+1] = cu_cmp[b] + floor((cu[b+1]-cu[b]) / r). One block walks the
// sequences in chunks of 1024 with a block scan and a running carry.
__global__ void __launch_bounds__(kScanThreads)
compress_cu_seqlens_kernel(const int32_t *__restrict__ cu, int32_t batch, int32_t r,
                           int32_t *__restrict__ cu_cmp, int32_t *err) {
    __shared__ int32_t scratch[kScanThreads / 32 + 1];
    int32_t carry = 0;
    if (threadIdx.x == 0) cu_cmp[0] = 0;
    for (int32_t base = 0; base < batch; base += kScanThreads) {
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
        int32_t before = block_exclusive_scan<kScanThreads>(groups, scratch, &total);
        if (b < batch) cu_cmp[b + 1] = carry + before + groups;
        carry += total;
    }
}

// One warp per token: the segment search runs once, the W entries are
// written by the 32 lanes (16-byte stores when W is a multiple of 4 and the
// output is 16-byte aligned).
__global__ void __launch_bounds__(256)
window_idx_kernel(const int32_t *__restrict__ cu, int32_t batch, int32_t T, int32_t W,
                  bool vec4, int32_t *__restrict__ idx, int32_t *err) {
    const int lane = threadIdx.x & 31;
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    for (int64_t t = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); t < T;
         t += warps) {
        const int32_t b = find_segment(cu, batch, (int32_t)t);
        int32_t start, last;
        if (b < 0) {
            if (lane == 0) report_error(err, kErrCheck, kKerWindow, 1);
            start = 1;
            last = 0;  // empty: every slot -1
        } else {
            const int32_t seg0 = __ldg(cu + b);
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
    compress_cu_seqlens_kernel<<<1, kScanThreads, 0, stream>>>(cu, batch, cmp_ratio, cu_cmp, err);
    return cudaGetLastError();
}

cudaError_t launch_window_idx(const int32_t *cu, int32_t batch, int32_t total_tokens,
                              int32_t window, int32_t *idx, int32_t *err, cudaStream_t stream) {
    if (total_tokens == 0) return cudaSuccess;
    const int warps_per_block = 8;
    int64_t blocks = ((int64_t)total_tokens + warps_per_block - 1) / warps_per_block;
    if (blocks > 152 * 64) blocks = 152 * 64;
    const bool vec4 = (window & 3) == 0 && ((uintptr_t)idx & 15u) == 0;
    window_idx_kernel<<<(unsigned)blocks, 32 * warps_per_block, 0, stream>>>(
        cu, batch, total_tokens, window, vec4, idx, err);
    return cudaGetLastError();
}

}  // namespace csa
