// THD compressor core (sm_103a): grouping, position embedding, overlap
// transform and slot pooling of one DeepSeek-V4 compressor.
//
// The miles PR 2038 report (compressor.py, _forward_thd and
// _overlap_transform_thd) groups the rows of each packed sequence: compressed
// row g = cu_c[b] + j takes rows cu[b] + j r + i (i < r) of the two
// projections kv = x W_kv^T and score = x W_gate^T; with overlap, each group
// becomes 2r slots of head_dim -- the first halves of the previous group's
// rows (missing for a sequence's first group: kv 0, score -inf) and the
// second halves of its own rows. The page omits what follows; the -inf fill
// of the score only means something as a softmax logit, so the reading here
// is the softmax over the slots, per dimension, weighting kv, with the
// position embedding ape[i] added to the score of slot i before the overlap.
//
// Design: one thread per (compressed row, dimension); a block covers 128
// dimensions of one compressed row, so each slot's read is a coalesced
// 512-byte row piece, and every input element is read once (a row's first
// half by the next group, its second half by its own group). The softmax is
// accumulated online in fp32 (running max, rescaled sum). HBM-bound: the
// bytes are the grouped rows of both projections plus the output.
#include "common.cuh"
#include "internal.h"

namespace csa {

namespace {

constexpr int kCmpThreads = 128;

__device__ __forceinline__ void pool_slot(float s, float v, float &m, float &z, float &acc) {
    if (s > m) {
        const float c = expf(m - s);  // 0 while m is still -inf
        z = z * c + 1.0f;
        acc = acc * c + v;
        m = s;
    } else {
        const float p = expf(s - m);
        z += p;
        acc = fmaf(p, v, acc);
    }
}

__global__ void __launch_bounds__(kCmpThreads) compress_thd_kernel(CompressArgs a) {
    __shared__ int32_t info[3];  // segment, its first packed row, j (group index in it)
    const int32_t g = blockIdx.x;
    if (threadIdx.x == 0) {
        const int32_t b = find_segment(a.cu_c, a.batch, g);
        info[0] = b;
        if (b >= 0) {
            info[1] = __ldg(a.cu_q + b);
            info[2] = g - __ldg(a.cu_c + b);
            // the group's rows must lie inside its sequence
            const int64_t last = (int64_t)info[1] + ((int64_t)info[2] + 1) * a.r - 1;
            if (last >= __ldg(a.cu_q + b + 1) || last >= a.T) info[0] = -1;
        }
        if (info[0] < 0) report_error(a.err, kErrCheck, kKerCompressor, 1);
    }
    __syncthreads();
    const int32_t e = blockIdx.y * kCmpThreads + threadIdx.x;
    if (e >= a.hd) return;
    float *dst = a.out + (int64_t)g * a.hd + e;
    if (info[0] < 0) {
        *dst = 0.0f;
        return;
    }
    const int64_t wd = a.overlap ? 2 * (int64_t)a.hd : a.hd;
    const int64_t first = (int64_t)info[1] + (int64_t)info[2] * a.r;  // own group's first row
    const bool has_prev = a.overlap && info[2] > 0;
    const int64_t own_col = a.overlap ? a.hd + e : e;
    float m = -INFINITY, z = 0.0f, acc = 0.0f;
    for (int32_t i = 0; i < a.r; ++i) {
        if (has_prev) {
            const int64_t row = first - a.r + i;
            const float s = __ldg(a.score + row * wd + e) + (a.ape ? __ldg(a.ape + i * wd + e) : 0.0f);
            pool_slot(s, __ldg(a.kv + row * wd + e), m, z, acc);
        }
        const int64_t row = first + i;
        const float s = __ldg(a.score + row * wd + own_col) +
                        (a.ape ? __ldg(a.ape + i * wd + own_col) : 0.0f);
        pool_slot(s, __ldg(a.kv + row * wd + own_col), m, z, acc);
    }
    *dst = acc / z;
}

}  // namespace

cudaError_t launch_compress_thd(const CompressArgs &a, cudaStream_t stream) {
    if (a.Tc == 0) return cudaSuccess;
    const dim3 grid((unsigned)a.Tc, (unsigned)((a.hd + kCmpThreads - 1) / kCmpThreads));
    compress_thd_kernel<<<grid, kCmpThreads, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace csa
