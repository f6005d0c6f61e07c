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
// accumulates d_w (one head per thread), d_q (a 4-head x 8- or 4-column
// register tile per thread) and the chunk's row gradients (4 or 2 rows x 4
// columns per thread), which are added to d_k with 16-byte atomics (a warp
// covers 512 contiguous bytes of one row). Every contraction reads its
// shared operands as float4 register tiles, about one load per 5-10 FMAs.
// All arithmetic is fp32 on the CUDA cores. This kernel serves index_dim 64;
// index_dim 128 runs on the tensor cores (indexer_kl_grad_tc.cu).
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
    float q[kKlHeads][DI + 4];         // the token's q, fp32 (rows >= Hi zero)
    float k[kKlChunk][DI + 4];         // a chunk of k rows, fp32
    float a[kKlHeads][kKlChunk + 1];   // a_hs of the chunk
    float g[kKlHeads][kKlChunk + 4];   // G[h][c] = g_c w_h [a_hc > 0]
    float gt[kKlChunk][kKlHeads + 4];  // the same, transposed
    float w[kKlHeads];
    int32_t rows[kKlMaxList];          // the token's valid rows, in list order
    float p[kKlMaxList];               // their targets (unnormalised)
    float dl[kKlMaxList];              // scores I, then dL/dI
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

// a[h][c] = q[h,:] . k[c,:] for the 64 heads x 32 rows of a chunk. Thread
// tile: heads 4 hb .. 4 hb + 3 and rows cb, cb + 16 (hb = tid / 16,
// cb = tid % 16). Per 4 dims it reads 4 + 2 float4 for 32 FMAs; a
// quarter-warp's k rows are 132 floats apart (distinct banks) and the two
// head blocks of a warp are 4 padded rows apart (distinct banks). Pass 1 and
// pass 2 run this same code, so their fp32 values (and ReLU decisions) are
// identical.
template <int DI>
__device__ __forceinline__ void chunk_dots(KlSmem<DI> &s) {
    const int hb = threadIdx.x >> 4, cb = threadIdx.x & 15;
    float acc[4][2];
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[i][0] = acc[i][1] = 0.0f;
#pragma unroll 4
    for (int d = 0; d < DI; d += 4) {
        float4 kv[2], qv[4];
#pragma unroll
        for (int j = 0; j < 2; ++j) kv[j] = *reinterpret_cast<const float4 *>(&s.k[cb + 16 * j][d]);
#pragma unroll
        for (int i = 0; i < 4; ++i) qv[i] = *reinterpret_cast<const float4 *>(&s.q[4 * hb + i][d]);
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                acc[i][j] = fmaf(qv[i].x, kv[j].x, acc[i][j]);
                acc[i][j] = fmaf(qv[i].y, kv[j].y, acc[i][j]);
                acc[i][j] = fmaf(qv[i].z, kv[j].z, acc[i][j]);
                acc[i][j] = fmaf(qv[i].w, kv[j].w, acc[i][j]);
            }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 2; ++j) s.a[4 * hb + i][cb + 16 * j] = acc[i][j];
}

template <int DI>
__global__ void __launch_bounds__(kKlThreads, 2) indexer_kl_grad_kernel(IndexerKlArgs args) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    KlSmem<DI> &s = *reinterpret_cast<KlSmem<DI> *>(smem_raw);
    const IndexerKlArgs &a = args;
    const int tid = threadIdx.x;
    // d_q tile: heads 4 hb .. 4 hb + 3 x columns 64 gi + 4 db + e (hb = tid / 16,
    // db = tid % 16, gi < DI / 64, e < 4)
    constexpr int kQg = DI / 64;
    // d_k tile: rows kKr cb .. kKr cb + kKr - 1 x columns 4 db .. 4 db + 3
    // (db = tid % (DI / 4), cb = tid / (DI / 4))
    constexpr int kQuads = DI / 4;
    constexpr int kKr = kKlChunk * kQuads / kKlThreads;  // 4 (Di 128) or 2 (Di 64)
    static_assert(kKr == 2 || kKr == 4, "d_k tile");

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
                s.dl[c0 + tid] = sc;
            }
            __syncthreads();
        }

        // ---- log-softmax over the entries, loss, dL/dI ----
        float mx = -INFINITY;
        for (int i = tid; i < n; i += kKlThreads) mx = fmaxf(mx, s.dl[i]);
        mx = block_max(mx, s.red);
        float z = 0.0f;
        for (int i = tid; i < n; i += kKlThreads) z += expf(s.dl[i] - mx);
        z = block_sum(z, s.red);
        const float lz = mx + logf(z);
        float kl = 0.0f;
        for (int i = tid; i < n; i += kKlThreads) {
            const float ps = s.p[i] * inv_mass;
            const float log_pi = s.dl[i] - lz;
            if (ps > 0.0f) kl += ps * (logf(ps) - log_pi);
            s.dl[i] = a.grad_scale * (expf(log_pi) - ps);
        }
        kl = block_sum(kl, s.red);  // also orders the g writes before their reads
        if (tid == 0 && a.loss) a.loss[t] = kl;

        // ---- pass 2: gradients ----
        float dq[4][4 * kQg];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int e = 0; e < 4 * kQg; ++e) dq[i][e] = 0.0f;
        float dw = 0.0f;
        const int q_hb = tid >> 4, q_db = tid & 15;
        const int k_db = tid % kQuads, k_cb = tid / kQuads;
        for (int c0 = 0; c0 < n; c0 += kKlChunk) {
            load_k_chunk(s, a.k, c0, n);
            __syncthreads();
            chunk_dots(s);
            __syncthreads();
            const int nc = min(kKlChunk, n - c0);
            if (tid < kKlHeads)
                for (int c = 0; c < nc; ++c) dw = fmaf(s.dl[c0 + c], fmaxf(s.a[tid][c], 0.0f), dw);
            // G[h][c] = g_c w_h [a_hc > 0] (zero past the chunk's rows), and its transpose
            for (int e = tid; e < kKlHeads * kKlChunk; e += kKlThreads) {
                const int h = e / kKlChunk, c = e % kKlChunk;
                const float gv = (c < nc && s.a[h][c] > 0.0f) ? s.dl[c0 + c] * s.w[h] : 0.0f;
                s.g[h][c] = gv;
                s.gt[c][h] = gv;
            }
            __syncthreads();
            // d_q[h][d] += sum_c G[h][c] k[c][d]: 3 (Di 128) or 2 float4 reads per 32 or 16 FMAs
#pragma unroll 4
            for (int c = 0; c < kKlChunk; ++c) {
                const float4 gv = *reinterpret_cast<const float4 *>(&s.gt[c][4 * q_hb]);
                const float gh[4] = {gv.x, gv.y, gv.z, gv.w};
#pragma unroll
                for (int gi = 0; gi < kQg; ++gi) {
                    const float4 kv = *reinterpret_cast<const float4 *>(&s.k[c][64 * gi + 4 * q_db]);
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        dq[i][4 * gi + 0] = fmaf(gh[i], kv.x, dq[i][4 * gi + 0]);
                        dq[i][4 * gi + 1] = fmaf(gh[i], kv.y, dq[i][4 * gi + 1]);
                        dq[i][4 * gi + 2] = fmaf(gh[i], kv.z, dq[i][4 * gi + 2]);
                        dq[i][4 * gi + 3] = fmaf(gh[i], kv.w, dq[i][4 * gi + 3]);
                    }
                }
            }
            // d_k[row c][d..d+3] += sum_h G[h][c] q[h][d..d+3] for kKr rows per thread
            {
                float4 acc[kKr];
#pragma unroll
                for (int r = 0; r < kKr; ++r) acc[r] = make_float4(0.f, 0.f, 0.f, 0.f);
                for (int h = 0; h < a.Hi; ++h) {
                    float gr[kKr];
                    if constexpr (kKr == 4) {
                        const float4 v = *reinterpret_cast<const float4 *>(&s.g[h][4 * k_cb]);
                        gr[0] = v.x, gr[1] = v.y, gr[2] = v.z, gr[3] = v.w;
                    } else {
                        const float2 v = *reinterpret_cast<const float2 *>(&s.g[h][2 * k_cb]);
                        gr[0] = v.x, gr[1] = v.y;
                    }
                    const float4 qv = *reinterpret_cast<const float4 *>(&s.q[h][4 * k_db]);
#pragma unroll
                    for (int r = 0; r < kKr; ++r) {
                        acc[r].x = fmaf(gr[r], qv.x, acc[r].x);
                        acc[r].y = fmaf(gr[r], qv.y, acc[r].y);
                        acc[r].z = fmaf(gr[r], qv.z, acc[r].z);
                        acc[r].w = fmaf(gr[r], qv.w, acc[r].w);
                    }
                }
#pragma unroll
                for (int r = 0; r < kKr; ++r) {
                    const int c = kKr * k_cb + r;
                    if (c < nc)
                        atomicAdd(reinterpret_cast<float4 *>(a.d_k + (int64_t)s.rows[c0 + c] * DI +
                                                             4 * k_db),
                                  acc[r]);
                }
            }
            __syncthreads();  // the chunk's k rows and coefficients are rewritten next
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int h = 4 * q_hb + i;
            if (h < a.Hi)
#pragma unroll
                for (int gi = 0; gi < kQg; ++gi)
#pragma unroll
                    for (int e = 0; e < 4; ++e) dq_out[h * DI + 64 * gi + 4 * q_db + e] = dq[i][4 * gi + e];
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
    // index_dim 128: the contractions on the tensor cores
    if (a.Di == 128) return launch_indexer_kl_grad_tc(a, stream);
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    return launch_kl<64>(a, sms, stream);
}

}  // namespace csa
