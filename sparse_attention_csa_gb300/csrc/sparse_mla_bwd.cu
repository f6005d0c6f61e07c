// Backward of the shared-KV MLA sparse attention with sinks (sm_103a).
//
// The gradient entry point of DeepSeek-V4's CSA/HCA attention as the miles PR
// 2038 report and the hyper-parallel RFC ("npu_sparse_flash_mla_grad") list
// it: from q, dout, the forward's output and log-sum-exp, it returns d_query,
// d_ori_kv, d_cmp_kv, d_sinks and the head-averaged attention distributions
// ori/cmp_softmax_l1_norm, shaped like the window and compressed index lists.
// For token t, head h and its keys a (window rows of ori_kv, then the
// selected, or every visible, row of cmp_kv; one 512-wide row is both key and
// value):
//   P_a  = exp(scale q.k_a - lse),   P_sink = exp(sink - lse)
//   Dv   = dout . out
//   dS_a = P_a (dout . k_a - Dv)
//   d_q  = scale sum_a dS_a k_a
//   d_row_a += scale dS_a q + P_a dout
//   d_sink  -= P_sink Dv
//   l1[slot of a] += P_a / H
//
// First version, on the CUDA cores in fp32. One CTA of 512 threads per token;
// heads in groups of 32 (a group's q and dout rows staged in shared memory as
// fp32), keys in tiles of 32 stored transposed ([d][key], padded) so that one
// lane owns one key in the score dot products. Each thread owns one of the 512
// dimensions for d_q (32 heads in registers) and for the rows' gradients,
// which are added to the fp32 outputs with one atomic per (key, dimension,
// head group). The distributions accumulate in shared memory over the head
// groups and are written once.
#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace csa {

namespace {

constexpr int kBwdThreads = 512;  // one per dimension
constexpr int kHG = 32;           // heads per group
constexpr int kKT = 32;           // keys per tile
constexpr int kKTStride = 33;     // floats per transposed tile row (no bank conflicts)
constexpr int kBwdMaxList = 1024; // top-k entries kept per token
constexpr int kBwdMaxWin = 1024;  // window rows per token

struct BwdSmem {
    float q[kHG][512];
    float g[kHG][512];
    float kt[512][kKTStride];
    float p[kKT][kHG];   // [key][head]
    float ds[kKT][kHG];  // [key][head]
    float l1[kBwdMaxWin + kBwdMaxList];
    int32_t rows[kBwdMaxList];  // compressed rows of the token's top-k list that count
    int32_t slots[kBwdMaxList]; // and the list entries they came from
    float dv[kHG];
    float lse[kHG];
    int32_t n_cmp;
};
static_assert(sizeof(BwdSmem) <= 232448, "shared memory budget");

__global__ void zero_f32_kernel(float *p, int64_t n) {
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x)
        p[i] = 0.0f;
}

__global__ void __launch_bounds__(kBwdThreads, 1) sparse_mla_bwd_kernel(MlaBwdArgs a) {
    extern __shared__ __align__(16) unsigned char raw[];
    BwdSmem *sm = reinterpret_cast<BwdSmem *>(raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int32_t t = blockIdx.x;
    const int32_t W = a.window;
    const bool use_cmp = a.cmp_kv != nullptr && a.Tc > 0;

    const int32_t b = find_segment(a.cu_q, a.batch, t);
    if (b < 0) {  // not covered by any sequence: report, leave zero gradients
        if (tid == 0) report_error(a.err, kErrCheck, kKerMlaBwd, 1);
        for (int i = tid; i < a.H * 512; i += kBwdThreads) a.d_q[(int64_t)t * a.H * 512 + i] = 0.0f;
        return;
    }
    const int32_t seg0 = __ldg(a.cu_q + b);
    const int32_t pos = t - seg0;
    const int32_t start = max(t - W + 1, seg0);
    const int32_t n_win = t - start + 1;
    int32_t cbase = 0, vis = 0;
    if (use_cmp) {
        cbase = __ldg(a.cu_c + b);
        vis = min((pos + 1) / a.cmp_ratio, __ldg(a.cu_c + b + 1) - cbase);
        if (cbase < 0 || vis < 0 || (int64_t)cbase + vis > a.Tc) {
            if (tid == 0) report_error(a.err, kErrCheck, kKerMlaBwd, 2);
            vis = 0;
        }
    }
    // The compressed keys: the visible entries of the top-k list, in list
    // order (warp 0 compacts), or every visible block.
    if (use_cmp && a.cmp_idx) {
        if (warp == 0) {
            int32_t n = 0;
            const int32_t *row = a.cmp_idx + (int64_t)t * a.topk;
            for (int32_t e0 = 0; e0 < a.topk; e0 += 32) {
                const int32_t e = e0 + lane;
                const int32_t j = e < a.topk ? __ldg(row + e) : -1;
                const bool ok = j >= cbase && j < cbase + vis;
                const uint32_t m = __ballot_sync(0xffffffffu, ok);
                if (ok) {
                    const int32_t at = n + __popc(m & ((1u << lane) - 1u));
                    sm->rows[at] = j;
                    sm->slots[at] = e;
                }
                n += __popc(m);
            }
            if (lane == 0) sm->n_cmp = n;
        }
    } else if (tid == 0) {
        sm->n_cmp = vis;
    }
    for (int i = tid; i < kBwdMaxWin + kBwdMaxList; i += kBwdThreads) sm->l1[i] = 0.0f;
    __syncthreads();
    const int32_t n_cmp = sm->n_cmp;
    const int32_t n_keys = n_win + n_cmp;
    const float scale = a.softmax_scale;
    const int d = tid;  // this thread's dimension

    for (int32_t h0 = 0; h0 < a.H; h0 += kHG) {
        const int nh = min(kHG, a.H - h0);
        // the group's q and dout rows, fp32; rows past the last head are zero
        for (int i = tid; i < kHG * 512; i += kBwdThreads) {
            const int h = i >> 9, dd = i & 511;
            float qv = 0.0f, gv = 0.0f;
            if (h < nh) {
                const int64_t o = ((int64_t)t * a.H + h0 + h) * 512 + dd;
                qv = __bfloat162float(a.q[o]);
                gv = __bfloat162float(a.dout[o]);
            }
            sm->q[h][dd] = qv;
            sm->g[h][dd] = gv;
        }
        // Dv = dout . out per head (one warp per head); the sink's gradient
        for (int h = warp; h < kHG; h += kBwdThreads / 32) {
            float s = 0.0f;
            if (h < nh) {
                const int64_t o = ((int64_t)t * a.H + h0 + h) * 512;
                for (int dd = lane; dd < 512; dd += 32)
                    s += __bfloat162float(a.dout[o + dd]) * __bfloat162float(a.out[o + dd]);
            }
            s = warp_sum(s);
            if (lane == 0) {
                const float lse = h < nh ? a.lse[(int64_t)t * a.H + h0 + h] : 0.0f;
                sm->dv[h] = s;
                sm->lse[h] = lse;
                if (h < nh && a.sinks && a.d_sinks) {
                    const float sk = __ldg(a.sinks + h0 + h);
                    if (sk != -INFINITY) atomicAdd(a.d_sinks + h0 + h, -expf(sk - lse) * s);
                }
            }
        }
        __syncthreads();
        // this thread's dimension of q and dout for the group's heads
        float qd[kHG], gd[kHG], dq[kHG];
#pragma unroll
        for (int h = 0; h < kHG; ++h) {
            qd[h] = sm->q[h][d];
            gd[h] = sm->g[h][d];
            dq[h] = 0.0f;
        }
        for (int32_t k0 = 0; k0 < n_keys; k0 += kKT) {
            const int nk = min(kKT, n_keys - k0);
            // the tile, transposed: kt[d][i] = row of key k0 + i, dimension d
            for (int i = warp; i < kKT; i += kBwdThreads / 32) {
                const int32_t key = k0 + i;
                const __nv_bfloat16 *src = nullptr;
                if (i < nk) {
                    if (key < n_win) src = a.ori_kv + (int64_t)(start + key) * 512;
                    else if (a.cmp_idx) src = a.cmp_kv + (int64_t)sm->rows[key - n_win] * 512;
                    else src = a.cmp_kv + (int64_t)(cbase + key - n_win) * 512;
                }
                for (int e = 0; e < 8; ++e) {
                    const int dd = 2 * lane + 64 * e;
                    float2 v = make_float2(0.0f, 0.0f);
                    if (src) v = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(src + dd));
                    sm->kt[dd][i] = v.x;
                    sm->kt[dd + 1][i] = v.y;
                }
            }
            __syncthreads();
            // scores and dout.k: warp w takes heads 2w and 2w+1, lane = key
            {
                const int i = lane;
                const int ha = 2 * warp, hb = ha + 1;
                float sa = 0.0f, sb = 0.0f, pa = 0.0f, pb = 0.0f;
                for (int dd = 0; dd < 512; dd += 4) {
                    const float4 qa = *reinterpret_cast<const float4 *>(&sm->q[ha][dd]);
                    const float4 qb = *reinterpret_cast<const float4 *>(&sm->q[hb][dd]);
                    const float4 ga = *reinterpret_cast<const float4 *>(&sm->g[ha][dd]);
                    const float4 gb = *reinterpret_cast<const float4 *>(&sm->g[hb][dd]);
                    const float k0v = sm->kt[dd][i], k1v = sm->kt[dd + 1][i];
                    const float k2v = sm->kt[dd + 2][i], k3v = sm->kt[dd + 3][i];
                    sa += qa.x * k0v + qa.y * k1v + qa.z * k2v + qa.w * k3v;
                    sb += qb.x * k0v + qb.y * k1v + qb.z * k2v + qb.w * k3v;
                    pa += ga.x * k0v + ga.y * k1v + ga.z * k2v + ga.w * k3v;
                    pb += gb.x * k0v + gb.y * k1v + gb.z * k2v + gb.w * k3v;
                }
                const bool key_ok = i < nk;
                const float Pa = (key_ok && ha < nh) ? expf(scale * sa - sm->lse[ha]) : 0.0f;
                const float Pb = (key_ok && hb < nh) ? expf(scale * sb - sm->lse[hb]) : 0.0f;
                sm->p[i][ha] = Pa;
                sm->p[i][hb] = Pb;
                sm->ds[i][ha] = Pa * (pa - sm->dv[ha]);
                sm->ds[i][hb] = Pb * (pb - sm->dv[hb]);
            }
            __syncthreads();
            // the distribution: sum of the tile's weights over the group's heads
            if (tid < nk) {
                const int32_t key = k0 + tid;
                if (key < n_win || a.cmp_idx) {
                    float s = 0.0f;
#pragma unroll
                    for (int h = 0; h < kHG; ++h) s += sm->p[tid][h];
                    sm->l1[key] += s;
                }
            }
            // d_q (registers) and the rows' gradients (atomics), dimension d
            for (int i = 0; i < nk; ++i) {
                const float kv = sm->kt[d][i];
                float gsum = 0.0f;
#pragma unroll
                for (int h4 = 0; h4 < kHG; h4 += 4) {
                    const float4 s4 = *reinterpret_cast<const float4 *>(&sm->ds[i][h4]);
                    const float4 p4 = *reinterpret_cast<const float4 *>(&sm->p[i][h4]);
                    dq[h4] += s4.x * kv;
                    dq[h4 + 1] += s4.y * kv;
                    dq[h4 + 2] += s4.z * kv;
                    dq[h4 + 3] += s4.w * kv;
                    gsum += scale * (s4.x * qd[h4] + s4.y * qd[h4 + 1] + s4.z * qd[h4 + 2] +
                                     s4.w * qd[h4 + 3]) +
                            (p4.x * gd[h4] + p4.y * gd[h4 + 1] + p4.z * gd[h4 + 2] +
                             p4.w * gd[h4 + 3]);
                }
                const int32_t key = k0 + i;
                float *dst;
                if (key < n_win) dst = a.d_ori_kv + (int64_t)(start + key) * 512;
                else if (a.cmp_idx) dst = a.d_cmp_kv + (int64_t)sm->rows[key - n_win] * 512;
                else dst = a.d_cmp_kv + (int64_t)(cbase + key - n_win) * 512;
                atomicAdd(dst + d, gsum);
            }
            __syncthreads();  // the tile and the weights are rewritten next
        }
#pragma unroll
        for (int h = 0; h < kHG; ++h)
            if (h < nh) a.d_q[((int64_t)t * a.H + h0 + h) * 512 + d] = scale * dq[h];
        __syncthreads();  // q and dout rows are rewritten by the next group
    }
    // head-averaged distributions, in the index lists' shapes
    const float inv_h = 1.0f / (float)a.H;
    if (a.ori_l1)
        for (int i = tid; i < W; i += kBwdThreads)
            a.ori_l1[(int64_t)t * W + i] = i < n_win ? sm->l1[i] * inv_h : 0.0f;
    if (a.cmp_l1 && use_cmp && a.cmp_idx)
        for (int i = tid; i < n_cmp; i += kBwdThreads)
            a.cmp_l1[(int64_t)t * a.topk + sm->slots[i]] = sm->l1[n_win + i] * inv_h;
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
    e = cudaFuncSetAttribute(sparse_mla_bwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)sizeof(BwdSmem));
    if (e != cudaSuccess) return e;
    sparse_mla_bwd_kernel<<<a.T, kBwdThreads, sizeof(BwdSmem), stream>>>(a);
    return cudaGetLastError();
}

}  // namespace csa
