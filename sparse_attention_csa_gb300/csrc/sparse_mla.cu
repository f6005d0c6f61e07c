// Shared-KV MLA sparse attention forward with attention sinks.
//
// Sources: hyper-parallel RFC "DeepSeek-V4 CSA/HCA 自定义算子接入…", background
// item 2 (ori_kv band/sliding-window branch + cmp_kv compressed branch +
// attention sink) and section 2 (sparse_flash_mla schema and defaults;
// ori_sparse_indices takes no part, the band comes from the window
// arguments); Megatron-LM PR 7 (verl) environment note (head_dim = d_v = 512:
// the 512-wide row is both key and value); MindSpeed-LLM PR 4842 main changes
// (COMPRESSOR_ONLY mode attends every visible compressed block).
//
// Per token t and head h, over keys = window rows of ori_kv, then the
// compressed rows of cmp_kv chosen by cmp_sparse_indices (or all visible):
//     l_i = scale * q.kv_i ; m = max(l, sink) ; Z = sum e^(l_i-m) + e^(sink-m)
//     out = sum e^(l_i-m) kv_i / Z ; lse = m + ln Z
// computed with an online softmax in fp32 (base-2 exponent), bf16 output.
//
// This kernel is the plain SIMT formulation: one CTA per token, keys staged in
// shared memory 32 rows at a time.
#include "common.cuh"
#include "internal.h"

namespace csa {

namespace {

constexpr int kThreads = 256;
constexpr int kD = 512;
constexpr int kChunk = 32;                 // keys per shared-memory stage
constexpr int kRowPad = kD + 8;            // bf16 elements per staged row (bank spread)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

struct Smem {
    __nv_bfloat16 q[64 * kD];
    __nv_bfloat16 kv[kChunk * kRowPad];
    float p[64 * kChunk];
    float m[64];
    float l[64];
    float alpha[64];
    int32_t row[kChunk];       // global row index, -1 masked
    int32_t src[kChunk];       // 0 = ori_kv, 1 = cmp_kv
};

__global__ void __launch_bounds__(kThreads, 1) sparse_mla_simt_kernel(MlaArgs a) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    Smem &sm = *reinterpret_cast<Smem *>(smem_raw);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int H = a.H;
    const float c = a.softmax_scale * kLog2e;

    for (int32_t t = blockIdx.x; t < a.T; t += gridDim.x) {
        const int32_t b = find_segment(a.cu_q, a.batch, t);
        if (b < 0) {
            if (tid == 0) report_error(a.err, kErrCheck, kKerMla, 1);
            continue;
        }
        const int32_t seg0 = __ldg(a.cu_q + b);
        const int32_t pos = t - seg0;
        const int32_t win_start = max(t - a.window + 1, seg0);
        const int32_t n_win = t - win_start + 1;
        int32_t cbase = 0, n_cmp = 0;
        const bool use_cmp = a.cmp_kv != nullptr && a.Tc > 0;
        if (use_cmp) {
            cbase = __ldg(a.cu_c + b);
            const int32_t seg_blocks = __ldg(a.cu_c + b + 1) - cbase;
            const int32_t vis = min((pos + 1) / a.cmp_ratio, seg_blocks);
            n_cmp = a.cmp_idx ? a.topk : vis;
            if (cbase < 0 || vis < 0 || cbase + vis > a.Tc) {
                if (tid == 0) report_error(a.err, kErrCheck, kKerMla, 2);
                n_cmp = 0;
            }
        }
        const int32_t vis_end = use_cmp ? cbase + min((pos + 1) / a.cmp_ratio,
                                                      __ldg(a.cu_c + b + 1) - cbase) : 0;
        const int32_t n_keys = n_win + n_cmp;

        __syncthreads();  // shared memory free from the previous token
        // q[t] -> shared (16-byte vectors)
        {
            const uint4 *src = reinterpret_cast<const uint4 *>(a.q + (int64_t)t * H * kD);
            uint4 *dst = reinterpret_cast<uint4 *>(sm.q);
            for (int i = tid; i < H * kD / 8; i += kThreads) dst[i] = __ldg(src + i);
        }
        if (tid < 64) {
            const float sink = (a.sinks && tid < H) ? __ldg(a.sinks + tid) : -INFINITY;
            sm.m[tid] = sink * kLog2e;                   // running max (base-2 units)
            sm.l[tid] = (sink == -INFINITY) ? 0.0f : 1.0f;  // e^(sink - m) with m = sink
        }
        // each thread owns head oh, d-range [od, od+128)
        const int oh = tid >> 2, od = (tid & 3) * 128;
        float o[128];
#pragma unroll
        for (int i = 0; i < 128; ++i) o[i] = 0.0f;

        for (int32_t k0 = 0; k0 < n_keys; k0 += kChunk) {
            // resolve this chunk's rows
            if (tid < kChunk) {
                const int32_t kk = k0 + tid;
                int32_t row = -1, src = 0;
                if (kk < n_win) {
                    row = win_start + kk;
                } else if (kk < n_keys) {
                    src = 1;
                    if (a.cmp_idx) {
                        const int32_t j = __ldg(a.cmp_idx + (int64_t)t * a.topk + (kk - n_win));
                        row = (j >= cbase && j < vis_end) ? j : -1;
                    } else {
                        row = cbase + (kk - n_win);
                    }
                }
                sm.row[tid] = row;
                sm.src[tid] = src;
            }
            __syncthreads();
            // gather rows (masked rows read as zero)
            for (int i = tid; i < kChunk * (kD / 8); i += kThreads) {
                const int r = i / (kD / 8), v = i % (kD / 8);
                const int32_t row = sm.row[r];
                uint4 x = make_uint4(0, 0, 0, 0);
                if (row >= 0) {
                    const __nv_bfloat16 *base = sm.src[r] ? a.cmp_kv : a.ori_kv;
                    x = __ldg(reinterpret_cast<const uint4 *>(base + (int64_t)row * kD) + v);
                }
                *reinterpret_cast<uint4 *>(sm.kv + r * kRowPad + v * 8) = x;
            }
            __syncthreads();
            // scores: thread -> key (lane), heads warp, warp+8, ...
            {
                const int key = lane;
                float acc[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
                const __nv_bfloat16 *kr = sm.kv + key * kRowPad;
                for (int d = 0; d < kD; d += 8) {
                    uint4 kx = *reinterpret_cast<const uint4 *>(kr + d);
                    const __nv_bfloat162 *k2 = reinterpret_cast<const __nv_bfloat162 *>(&kx);
                    float2 kf[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) kf[e] = __bfloat1622float2(k2[e]);
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const int h = warp + 8 * i;
                        if (h < H) {
                            uint4 qx = *reinterpret_cast<const uint4 *>(sm.q + h * kD + d);
                            const __nv_bfloat162 *q2 = reinterpret_cast<const __nv_bfloat162 *>(&qx);
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                float2 qf = __bfloat1622float2(q2[e]);
                                acc[i] = fmaf(qf.x, kf[e].x, acc[i]);
                                acc[i] = fmaf(qf.y, kf[e].y, acc[i]);
                            }
                        }
                    }
                }
                const bool valid = sm.row[key] >= 0;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int h = warp + 8 * i;
                    if (h < 64) sm.p[h * kChunk + key] = valid ? acc[i] * c : -INFINITY;
                }
            }
            __syncthreads();
            // online softmax: warp w updates heads w, w+8, ...
            for (int h = warp; h < H; h += 8) {
                const float v = sm.p[h * kChunk + lane];
                const float mx = warp_max(v);
                const float m_old = sm.m[h];
                const float m_new = fmaxf(m_old, mx);
                float alpha, pv;
                if (m_new == -INFINITY) {
                    alpha = 1.0f;
                    pv = 0.0f;
                } else {
                    alpha = exp2f(m_old - m_new);
                    pv = exp2f(v - m_new);
                }
                // the denominator sums fp32 p; P.V uses p rounded to bf16
                const float ps = warp_sum(pv);
                sm.p[h * kChunk + lane] = __bfloat162float(__float2bfloat16_rn(pv));
                __syncwarp();
                if (lane == 0) {
                    sm.m[h] = m_new;
                    sm.l[h] = sm.l[h] * alpha + ps;
                    sm.alpha[h] = alpha;
                }
            }
            __syncthreads();
            // O[h, d] = alpha O + sum_k p[h,k] kv[k, d]
            if (oh < H) {
                const float al = sm.alpha[oh];
#pragma unroll
                for (int i = 0; i < 128; ++i) o[i] *= al;
                for (int k = 0; k < kChunk; ++k) {
                    const float pk = sm.p[oh * kChunk + k];
                    if (pk == 0.0f) continue;
                    const __nv_bfloat16 *vr = sm.kv + k * kRowPad + od;
#pragma unroll
                    for (int d = 0; d < 128; d += 8) {
                        uint4 vx = *reinterpret_cast<const uint4 *>(vr + d);
                        const __nv_bfloat162 *v2 = reinterpret_cast<const __nv_bfloat162 *>(&vx);
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            float2 vf = __bfloat1622float2(v2[e]);
                            o[d + 2 * e] = fmaf(pk, vf.x, o[d + 2 * e]);
                            o[d + 2 * e + 1] = fmaf(pk, vf.y, o[d + 2 * e + 1]);
                        }
                    }
                }
            }
            __syncthreads();
        }
        // epilogue
        if (oh < H) {
            const float l = sm.l[oh];
            const float inv = l > 0.0f ? 1.0f / l : 0.0f;
            __nv_bfloat16 *dst = a.out + ((int64_t)t * H + oh) * kD + od;
#pragma unroll
            for (int d = 0; d < 128; d += 8) {
                uint4 vx;
                __nv_bfloat162 *v2 = reinterpret_cast<__nv_bfloat162 *>(&vx);
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    v2[e] = __floats2bfloat162_rn(o[d + 2 * e] * inv, o[d + 2 * e + 1] * inv);
                *reinterpret_cast<uint4 *>(dst + d) = vx;
            }
            if (a.lse && (tid & 3) == 0)
                a.lse[(int64_t)t * H + oh] = (sm.m[oh] + log2f(l)) * kLn2;
        }
    }
}

}  // namespace

cudaError_t launch_sparse_mla_fwd(const MlaArgs &a, cudaStream_t stream) {
    if (a.T == 0) return cudaSuccess;
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    const size_t smem = sizeof(Smem);
    e = cudaFuncSetAttribute(sparse_mla_simt_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem);
    if (e != cudaSuccess) return e;
    int ctas = a.T < sms * 8 ? a.T : sms * 8;
    sparse_mla_simt_kernel<<<ctas, kThreads, smem, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace csa
