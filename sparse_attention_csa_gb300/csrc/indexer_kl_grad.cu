// Indexer KL-loss gradient (sm_103a): the indexer's backward against the
// main attention's distribution.
//
// The hyper-parallel RFC, section 3, lists it as
// sparse_lightning_indexer_kl_loss_grad(q, k, w, sparse_indices,
// attn_softmax_l1_norm, cu_seqlens_q, cu_seqlens_k, mask_mode=3, cmp_ratio):
// "indexer backward + KL loss", fed with the distribution p that
// sparse_flash_mla_grad returns as softmax_l1_norm. MindSpeed-LLM PR 4842
// (main changes) scales the loss by the global token count under TND; here
// that factor is the caller's grad_scale.
//
// Per token t, over the entries s of sparse_indices[t] that name a visible
// row j_s (the indexer's causal rule):
//     a_hs = q[t,h,:] . k[j_s,:]                I_s = sum_h w[t,h] relu(a_hs)
//     p_s  = l1[t,s] / sum_S l1                 pi  = softmax_S(I)
//     loss[t] = sum_{p_s > 0} p_s (log p_s - log pi_s)
//     g_s  = grad_scale (pi_s - p_s)
//     d_w[t,h]    = sum_s g_s relu(a_hs)
//     d_q[t,h,:]  = sum_s g_s w[t,h] [a_hs > 0] k[j_s,:]
//     d_k[j_s,:] += g_s sum_h w[t,h] [a_hs > 0] q[t,h,:]
//
// Design: one CTA of 256 threads per token (grid-strided over tokens, two
// CTAs per SM). The token's q (Hi x Di, widened to fp32) and w sit in shared
// memory; its valid entries are compacted in order with a block scan. Rows of
// k come in chunks of 32 (bf16 -> fp32 in shared memory, rows padded by 4
// floats so that each quarter-warp's float4 reads hit 32 distinct banks).
// Pass 1 computes a and I chunk by chunk; pass 2 recomputes a with the same
// code (identical fp32 values, hence identical ReLU decisions), then
// accumulates d_w (one head per thread), d_q (32 or 16 outputs per thread in
// registers) and the chunk's row gradients, which are added to d_k with
// 16-byte atomics (a warp covers 512 contiguous bytes of one row). All
// arithmetic is fp32 on the CUDA cores.
#include "common.cuh"
#include "internal.h"

namespace csa {

namespace {

constexpr int kKlThreads = 256;
constexpr int kKlChunk = 32;      // k rows per chunk
constexpr int kKlHeads = 64;      // heads held (Hi <= 64, the rest zero)
constexpr int kKlMaxList = 2048;  // entries per token
constexpr int kKlWarps = kKlThreads / 32;

template <int DI>
struct KlSmem {
    float q[kKlHeads][DI];             // the token's q, fp32 (rows >= Hi zero)
    float k[kKlChunk][DI + 4];         // a chunk of k rows, fp32
    float a[kKlHeads][kKlChunk + 1];   // a_hs of the chunk, then the coefficients G
    float w[kKlHeads];
    int32_t rows[kKlMaxList];          // the token's valid rows, in list order
    float p[kKlMaxList];               // their targets (unnormalised)
    float g[kKlMaxList];               // scores I, then dL/dI
    float red[kKlWarps + 1];
    int32_t scan[kKlWarps + 1];
    int32_t info[4];                   // segment, cu_q[b], cu_c[b], cu_c[b+1]
};

__device__ __forceinline__ float block_sum(float v, float *red) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    v = warp_sum(v);
    if (lane == 0) red[warp] = v;
    __syncthreads();
    if (warp == 0) {
        float x = lane < kKlWarps ? red[lane] : 0.0f;
        x = warp_sum(x);
        if (lane == 0) red[kKlWarps] = x;
    }
    __syncthreads();
    const float total = red[kKlWarps];
    __syncthreads();
    return total;
}

__device__ __forceinline__ float block_max(float v, float *red) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    v = warp_max(v);
    if (lane == 0) red[warp] = v;
    __syncthreads();
    if (warp == 0) {
        float x = lane < kKlWarps ? red[lane] : -INFINITY;
        x = warp_max(x);
        if (lane == 0) red[kKlWarps] = x;
    }
    __syncthreads();
    const float total = red[kKlWarps];
    __syncthreads();
    return total;
}

// Stage rows[c0 .. c0+32) of k as fp32 (rows past n are zero).
template <int DI>
__device__ __forceinline__ void load_k_chunk(KlSmem<DI> &s, const __nv_bfloat16 *__restrict__ k,
                                             int c0, int n) {
    constexpr int kPerRow = DI / 8;  // 16-byte pieces per row
    for (int e = threadIdx.x; e < kKlChunk * kPerRow; e += kKlThreads) {
        const int c = e / kPerRow, d8 = (e % kPerRow) * 8;
        float4 lo = make_float4(0.f, 0.f, 0.f, 0.f), hi = lo;
        if (c0 + c < n) {
            const uint4 v = __ldg(reinterpret_cast<const uint4 *>(k + (int64_t)s.rows[c0 + c] * DI + d8));
            const __nv_bfloat162 *b2 = reinterpret_cast<const __nv_bfloat162 *>(&v);
            const float2 f0 = __bfloat1622float2(b2[0]), f1 = __bfloat1622float2(b2[1]);
            const float2 f2 = __bfloat1622float2(b2[2]), f3 = __bfloat1622float2(b2[3]);
            lo = make_float4(f0.x, f0.y, f1.x, f1.y);
            hi = make_float4(f2.x, f2.y, f3.x, f3.y);
        }
        *reinterpret_cast<float4 *>(&s.k[c][d8]) = lo;
        *reinterpret_cast<float4 *>(&s.k[c][d8 + 4]) = hi;
    }
}

// a[h][c] = q[h,:] . k[c,:] for the 64 heads x 32 rows of a chunk: lane c,
// heads warp + 8 i. Pass 1 and pass 2 run this same code, so their fp32
// values (and ReLU decisions) are identical.
template <int DI>
__device__ __forceinline__ void chunk_dots(KlSmem<DI> &s) {
    const int c = threadIdx.x & 31, hg = threadIdx.x >> 5;
    float acc[kKlHeads / kKlWarps];
#pragma unroll
    for (int i = 0; i < kKlHeads / kKlWarps; ++i) acc[i] = 0.0f;
#pragma unroll 4
    for (int d = 0; d < DI; d += 4) {
        const float4 kv = *reinterpret_cast<const float4 *>(&s.k[c][d]);
#pragma unroll
        for (int i = 0; i < kKlHeads / kKlWarps; ++i) {
            const float4 qv = *reinterpret_cast<const float4 *>(&s.q[hg + kKlWarps * i][d]);
            acc[i] = fmaf(qv.x, kv.x, acc[i]);
            acc[i] = fmaf(qv.y, kv.y, acc[i]);
            acc[i] = fmaf(qv.z, kv.z, acc[i]);
            acc[i] = fmaf(qv.w, kv.w, acc[i]);
        }
    }
#pragma unroll
    for (int i = 0; i < kKlHeads / kKlWarps; ++i) s.a[hg + kKlWarps * i][c] = acc[i];
}

template <int DI>
__global__ void __launch_bounds__(kKlThreads, 2) indexer_kl_grad_kernel(IndexerKlArgs args) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    KlSmem<DI> &s = *reinterpret_cast<KlSmem<DI> *>(smem_raw);
    const IndexerKlArgs &a = args;
    const int tid = threadIdx.x;
    constexpr int kGroups = kKlThreads / DI;         // head groups of the d_q mapping
    constexpr int kDq = kKlHeads / kGroups;           // d_q accumulators per thread
    constexpr int kQuads = DI / 4;                    // float4 columns of a row
    constexpr int kRowsPerPass = kKlThreads / kQuads; // rows of the d_k mapping per pass

    for (int32_t t = blockIdx.x; t < a.T; t += gridDim.x) {
        // ---- the token's segment, q and w ----
        if (tid == 0) {
            const int32_t b = find_segment(a.cu_q, a.batch, t);
            s.info[0] = b;
            if (b >= 0) {
                s.info[1] = __ldg(a.cu_q + b);
                s.info[2] = __ldg(a.cu_c + b);
                s.info[3] = __ldg(a.cu_c + b + 1);
                if (s.info[3] > a.Tc || s.info[2] < 0) {
                    report_error(a.err, kErrCheck, kKerIndexerKl, 1);
                    s.info[3] = min(s.info[3], a.Tc);
                    s.info[2] = max(s.info[2], 0);
                }
            } else {
                report_error(a.err, kErrCheck, kKerIndexerKl, 2);
            }
        }
        if (tid < kKlHeads) s.w[tid] = tid < a.Hi ? __ldg(a.w + (int64_t)t * a.Hi + tid) : 0.0f;
        {
            constexpr int kPerRow = DI / 8;
            const __nv_bfloat16 *qt = a.q + (int64_t)t * a.Hi * DI;
            for (int e = tid; e < kKlHeads * kPerRow; e += kKlThreads) {
                const int h = e / kPerRow, d8 = (e % kPerRow) * 8;
                float4 lo = make_float4(0.f, 0.f, 0.f, 0.f), hi = lo;
                if (h < a.Hi) {
                    const uint4 v = __ldg(reinterpret_cast<const uint4 *>(qt + (int64_t)h * DI + d8));
                    const __nv_bfloat162 *b2 = reinterpret_cast<const __nv_bfloat162 *>(&v);
                    const float2 f0 = __bfloat1622float2(b2[0]), f1 = __bfloat1622float2(b2[1]);
                    const float2 f2 = __bfloat1622float2(b2[2]), f3 = __bfloat1622float2(b2[3]);
                    lo = make_float4(f0.x, f0.y, f1.x, f1.y);
                    hi = make_float4(f2.x, f2.y, f3.x, f3.y);
                }
                *reinterpret_cast<float4 *>(&s.q[h][d8]) = lo;
                *reinterpret_cast<float4 *>(&s.q[h][d8 + 4]) = hi;
            }
        }
        __syncthreads();
        const int32_t b = s.info[0];

        // ---- compact the valid entries, in list order ----
        int32_t n = 0;
        float mass_part = 0.0f;
        if (b >= 0) {
            const int32_t pos = t - s.info[1], c_lo = s.info[2], c_hi = s.info[3];
            const int32_t *lst = a.idx + (int64_t)t * a.topk;
            const float *tgt = a.l1 + (int64_t)t * a.topk;
            for (int32_t base = 0; base < a.topk; base += kKlThreads) {
                const int32_t e = base + tid;
                int32_t j = -1;
                float pv = 0.0f;
                bool ok = false;
                if (e < a.topk) {
                    j = __ldg(lst + e);
                    // visible: in the segment and complete, (j_local + 1) r <= pos + 1
                    ok = j >= c_lo && j < c_hi &&
                         (int64_t)(j - c_lo + 1) * a.cmp_ratio <= (int64_t)pos + 1;
                    if (ok) pv = __ldg(tgt + e);
                }
                int32_t total = 0;
                const int32_t before = block_exclusive_scan<kKlThreads>(ok ? 1 : 0, s.scan, &total);
                if (ok) {
                    s.rows[n + before] = j;
                    s.p[n + before] = pv;
                    mass_part += pv;
                }
                n += total;
            }
        }
        const float mass = block_sum(mass_part, s.red);
        float *dq_out = a.d_q + (int64_t)t * a.Hi * DI;
        if (n == 0 || !(mass > 0.0f)) {
            // nothing selected or no target mass: zero loss, zero gradient
            for (int e = tid; e < a.Hi * DI; e += kKlThreads) dq_out[e] = 0.0f;
            if (tid < a.Hi) a.d_w[(int64_t)t * a.Hi + tid] = 0.0f;
            if (tid == 0 && a.loss) a.loss[t] = 0.0f;
            __syncthreads();
            continue;
        }
        const float inv_mass = 1.0f / mass;

        // ---- pass 1: scores ----
        for (int c0 = 0; c0 < n; c0 += kKlChunk) {
            load_k_chunk(s, a.k, c0, n);
            __syncthreads();
            chunk_dots(s);
            __syncthreads();
            if (tid < kKlChunk && c0 + tid < n) {
                float sc = 0.0f;
                for (int h = 0; h < a.Hi; ++h) sc = fmaf(s.w[h], fmaxf(s.a[h][tid], 0.0f), sc);
                s.g[c0 + tid] = sc;
            }
            __syncthreads();
        }

        // ---- log-softmax over the entries, loss, dL/dI ----
        float mx = -INFINITY;
        for (int i = tid; i < n; i += kKlThreads) mx = fmaxf(mx, s.g[i]);
        mx = block_max(mx, s.red);
        float z = 0.0f;
        for (int i = tid; i < n; i += kKlThreads) z += expf(s.g[i] - mx);
        z = block_sum(z, s.red);
        const float lz = mx + logf(z);
        float kl = 0.0f;
        for (int i = tid; i < n; i += kKlThreads) {
            const float ps = s.p[i] * inv_mass;
            const float log_pi = s.g[i] - lz;
            if (ps > 0.0f) kl += ps * (logf(ps) - log_pi);
            s.g[i] = a.grad_scale * (expf(log_pi) - ps);
        }
        kl = block_sum(kl, s.red);  // also orders the g writes before their reads
        if (tid == 0 && a.loss) a.loss[t] = kl;

        // ---- pass 2: gradients ----
        float dq[kDq];
#pragma unroll
        for (int i = 0; i < kDq; ++i) dq[i] = 0.0f;
        float dw = 0.0f;
        const int dq_d = tid % DI, dq_h0 = tid / DI;
        const int dk_d = (tid % kQuads) * 4, dk_r0 = tid / kQuads;
        for (int c0 = 0; c0 < n; c0 += kKlChunk) {
            load_k_chunk(s, a.k, c0, n);
            __syncthreads();
            chunk_dots(s);
            __syncthreads();
            const int nc = min(kKlChunk, n - c0);
            if (tid < kKlHeads)
                for (int c = 0; c < nc; ++c) dw = fmaf(s.g[c0 + c], fmaxf(s.a[tid][c], 0.0f), dw);
            __syncthreads();
            // G[h][c] = g_c w_h [a_hc > 0] (zero past the chunk's rows)
            for (int e = tid; e < kKlHeads * kKlChunk; e += kKlThreads) {
                const int h = e / kKlChunk, c = e % kKlChunk;
                const float av = s.a[h][c];
                s.a[h][c] = (c < nc && av > 0.0f) ? s.g[c0 + c] * s.w[h] : 0.0f;
            }
            __syncthreads();
            // d_q[h][d] += sum_c G[h][c] k[c][d]
#pragma unroll 4
            for (int c = 0; c < kKlChunk; ++c) {
                const float kv = s.k[c][dq_d];
#pragma unroll
                for (int i = 0; i < kDq; ++i) dq[i] = fmaf(s.a[dq_h0 + kGroups * i][c], kv, dq[i]);
            }
            // d_k[row c][d..d+3] += sum_h G[h][c] q[h][d..d+3]
#pragma unroll
            for (int r = dk_r0; r < kKlChunk; r += kRowsPerPass) {
                float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
                for (int h = 0; h < a.Hi; ++h) {
                    const float gv = s.a[h][r];
                    const float4 qv = *reinterpret_cast<const float4 *>(&s.q[h][dk_d]);
                    acc.x = fmaf(gv, qv.x, acc.x);
                    acc.y = fmaf(gv, qv.y, acc.y);
                    acc.z = fmaf(gv, qv.z, acc.z);
                    acc.w = fmaf(gv, qv.w, acc.w);
                }
                if (r < nc)
                    atomicAdd(reinterpret_cast<float4 *>(a.d_k + (int64_t)s.rows[c0 + r] * DI + dk_d), acc);
            }
            __syncthreads();  // the chunk's k rows and coefficients are rewritten next
        }
#pragma unroll
        for (int i = 0; i < kDq; ++i) {
            const int h = dq_h0 + kGroups * i;
            if (h < a.Hi) dq_out[h * DI + dq_d] = dq[i];
        }
        if (tid < a.Hi) a.d_w[(int64_t)t * a.Hi + tid] = dw;
        __syncthreads();  // shared q, w and lists are rewritten by the next token
    }
}

__global__ void zero_f32_kl_kernel(float *p, int64_t n) {
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x)
        p[i] = 0.0f;
}

template <int DI>
cudaError_t launch_kl(const IndexerKlArgs &a, int sms, cudaStream_t stream) {
    const size_t smem = sizeof(KlSmem<DI>);
    cudaError_t e = cudaFuncSetAttribute(indexer_kl_grad_kernel<DI>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const int64_t want = (int64_t)sms * 2;
    const int ctas = (int)(a.T < want ? a.T : want);
    indexer_kl_grad_kernel<DI><<<ctas, kKlThreads, smem, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace

int32_t indexer_kl_max_topk() { return kKlMaxList; }

cudaError_t launch_indexer_kl_grad(const IndexerKlArgs &a, cudaStream_t stream) {
    if (a.T == 0) return cudaSuccess;
    if (a.topk > kKlMaxList || a.Hi > kKlHeads || (a.Di != 64 && a.Di != 128))
        return cudaErrorInvalidValue;
    // d_k accumulates over tokens: it starts at zero
    if (a.Tc > 0) {
        const int64_t n = (int64_t)a.Tc * a.Di;
        const int64_t blocks = (n + 255) / 256;
        zero_f32_kl_kernel<<<(int)(blocks < 4096 ? blocks : 4096), 256, 0, stream>>>(a.d_k, n);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    return a.Di == 128 ? launch_kl<128>(a, sms, stream) : launch_kl<64>(a, sms, stream);
}

}  // namespace csa
