// Indexer KL-loss gradient on the tensor cores (sm_103a, tcgen05 + TMEM),
// index_dim 128, up to 64 heads.
//
// Same computation as indexer_kl_grad.cu (the hyper-parallel RFC, section 3,
// sparse_lightning_indexer_kl_loss_grad; the formulas are written out at the
// top of that file). Per token, the q rows of all 64 heads (zero past Hi) sit
// in shared memory in the 128-byte-swizzled K-major layout (2 chunks of 64
// dims x 64 heads); listed rows of k come in tiles of 64 (same layout, 2
// chunks of 8 KB). Per tile one thread issues:
//   S^T  = K q^T     M=64 rows x N=64 heads, K=128      TMEM cols   0..63
// (twice: pass 1 for the scores, pass 2 again for the gradients), and in
// pass 2, after the 256 threads have written G = g_row w_h [S^T > 0]:
//   d_q^T += K^T G   M=128 dims x N=64 heads, K=64 rows  TMEM cols  64..127
//   d_k    = G q     M=64 rows x N=128 dims, K=64 heads TMEM cols 128..255
// G enters the MMAs as two bf16 tiles, G_hi = bf16(G) and G_lo = bf16(G -
// G_hi), each one 128-byte row per listed row (the K-major A of d_k and the
// MN-major B of d_q^T): their sum carries G to about 2^-17 relative, so the
// gradients keep fp32-level accuracy although the operands are bf16 (q and k
// are bf16 inputs, exact as MMA operands). d_k is staged through shared
// memory and added with coalesced float4 atomics; d_w and the scores are
// reduced on the CUDA cores from the fp32 S^T in tensor memory (row r of an
// M=64 accumulator is TMEM lane 32 (r / 16) + r % 16). The scores of pass 2
// are the same MMA on the same operands as pass 1, so the ReLU decisions of
// the two passes agree. Two CTAs per SM (256 TMEM columns each).
#include <math.h>

#include "common.cuh"
#include "internal.h"
#include "tc_ptx.cuh"

namespace csa {

namespace {

constexpr int kThreads = 256;
constexpr int kRows = 64;          // listed rows per tile
constexpr int kMaxList = 2048;
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kColS = 0, kColDQ = 64, kColDK = 128;

// shared memory (offsets from a 1024-byte aligned base)
constexpr uint32_t kOffQ = 0;          // 2 x [64 heads x 128 B]
constexpr uint32_t kOffK = 16384;      // 2 x [64 rows x 128 B]
constexpr uint32_t kOffG = 32768;      // [64 rows x 128 B] bf16 G_hi
constexpr uint32_t kOffGlo = 40960;    // [64 rows x 128 B] bf16 G_lo
constexpr uint32_t kOffStage = 49152;  // [64 rows x 132] fp32 (d_k staging)
constexpr int kStageStride = 132;
constexpr uint32_t kOffMisc = kOffStage + kRows * kStageStride * 4;

struct Misc {
    uint64_t bar;
    uint32_t tmem_base;
    int32_t abort;
    int32_t info[4];  // segment, cu_q[b], cu_c[b], cu_c[b+1]
    float w[64];
    float part[2][kRows];   // score halves per row (head halves)
    float dwp[4][64];       // d_w partials per lane quarter
    float red[kThreads / 32 + 1];
    int32_t scan[kThreads / 32 + 1];
    int32_t rows[kMaxList];
    float p[kMaxList];
    float dl[kMaxList];
};
constexpr size_t kSmemBytes = kOffMisc + sizeof(Misc) + 1024;
static_assert(kSmemBytes <= 113 * 1024, "two CTAs per SM");

__device__ __forceinline__ uint32_t sw_off(uint32_t r, uint32_t u) {
    return r * 128u + ((u ^ (r & 7u)) << 4);
}

__device__ __forceinline__ float block_sum_tc(float v, float *red) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    v = warp_sum(v);
    if (lane == 0) red[warp] = v;
    __syncthreads();
    if (warp == 0) {
        float x = lane < kThreads / 32 ? red[lane] : 0.0f;
        x = warp_sum(x);
        if (lane == 0) red[kThreads / 32] = x;
    }
    __syncthreads();
    const float total = red[kThreads / 32];
    __syncthreads();
    return total;
}

__device__ __forceinline__ float block_max_tc(float v, float *red) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    v = warp_max(v);
    if (lane == 0) red[warp] = v;
    __syncthreads();
    if (warp == 0) {
        float x = lane < kThreads / 32 ? red[lane] : -INFINITY;
        x = warp_max(x);
        if (lane == 0) red[kThreads / 32] = x;
    }
    __syncthreads();
    const float total = red[kThreads / 32];
    __syncthreads();
    return total;
}

__global__ void __launch_bounds__(kThreads, 2) indexer_kl_grad_tc_kernel(IndexerKlArgs a) {
    extern __shared__ unsigned char raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(raw) + 1023) & ~(uintptr_t)1023);
    Misc *ms = reinterpret_cast<Misc *>(smem + kOffMisc);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int q4 = warp & 3, hf = warp >> 2;  // TMEM lane quarter, column half

    if (tid == 0) {
        tc::mbar_init(&ms->bar, 1);
        ms->abort = 0;
        tc::fence_mbar_init();
    }
    if (warp == 0) {
        tc::tmem_alloc(&ms->tmem_base, kTmemCols);
        tc::tmem_relinquish();
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = ms->tmem_base;
    const uint32_t lane_base = tmem + ((uint32_t)(32 * q4) << 16);

    const uint32_t s_q = tc::smem_u32(smem + kOffQ), s_k = tc::smem_u32(smem + kOffK);
    const uint32_t s_g = tc::smem_u32(smem + kOffG), s_gl = tc::smem_u32(smem + kOffGlo);
    const uint64_t d_k_km = tc::smem_desc(s_k, 16, 1024);
    const uint64_t d_q_km = tc::smem_desc(s_q, 16, 1024);
    const uint64_t d_k_mn = tc::smem_desc(s_k, 8192, 1024);
    const uint64_t d_q_mn = tc::smem_desc(s_q, 8192, 1024);
    const uint64_t d_g_km = tc::smem_desc(s_g, 16, 1024);
    const uint64_t d_g_mn = tc::smem_desc(s_g, 8192, 1024);
    const uint64_t d_gl_km = tc::smem_desc(s_gl, 16, 1024);
    const uint64_t d_gl_mn = tc::smem_desc(s_gl, 8192, 1024);
    constexpr uint32_t id_s = tc::idesc_bf16(64, 64, false, false);
    constexpr uint32_t id_dq = tc::idesc_bf16(128, 64, true, true);
    constexpr uint32_t id_dk = tc::idesc_bf16(64, 128, false, true);

    uint32_t n_commit = 0;
    bool ok = true;
    auto sync_mma = [&]() -> bool {
        if (tid == 0) tc::mma_commit(&ms->bar);
        const bool w = tc::mbar_wait(&ms->bar, n_commit & 1);
        ++n_commit;
        if (!w) {
            ms->abort = 1;
            report_error(a.err, kErrTimeout, kKerIndexerKl, 10);
        }
        __syncthreads();
        tc::tc_fence_after();
        return ms->abort == 0;
    };
    // the listed rows [r0, r0 + 64) as a swizzled K-major tile (rows past n zero)
    // (cp.async: every thread's copies in flight at once; rows past n zero)
    auto load_tile = [&](int32_t r0, int32_t n) {
        for (int i = tid; i < kRows * 16; i += kThreads) {  // (row, chunk, 16-byte unit)
            const int r = i >> 4, c = (i >> 3) & 1, u = i & 7;
            const bool in = r0 + r < n;
            const __nv_bfloat16 *src = in ? a.k + (int64_t)ms->rows[r0 + r] * 128 + 64 * c + 8 * u : a.k;
            tc::cp_async16_zfill(smem + kOffK + c * 8192 + sw_off(r, u), src, in ? 16u : 0u);
        }
        tc::cp_async_commit_wait_all();
        tc::fence_proxy_async_smem();
        __syncthreads();
    };
    auto issue_scores = [&]() {
        if (tid == 0) {
            tc::tc_fence_after();
#pragma unroll
            for (int c = 0; c < 2; ++c)
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    const uint32_t off = c * 8192 + kk * 32;
                    tc::mma_bf16(tmem + kColS, tc::desc_add(d_k_km, off), tc::desc_add(d_q_km, off),
                                 id_s, (c | kk) != 0);
                }
        }
    };

    for (int32_t t = blockIdx.x; t < a.T && ok; t += gridDim.x) {
        // ---- the token's segment, w and q ----
        if (tid == 0) {
            const int32_t b = find_segment(a.cu_q, a.batch, t);
            ms->info[0] = b;
            if (b >= 0) {
                ms->info[1] = __ldg(a.cu_q + b);
                ms->info[2] = __ldg(a.cu_c + b);
                ms->info[3] = __ldg(a.cu_c + b + 1);
                if (ms->info[3] > a.Tc || ms->info[2] < 0) {
                    report_error(a.err, kErrCheck, kKerIndexerKl, 1);
                    ms->info[3] = min(ms->info[3], a.Tc);
                    ms->info[2] = max(ms->info[2], 0);
                }
            } else {
                report_error(a.err, kErrCheck, kKerIndexerKl, 2);
            }
        }
        if (tid < 64) ms->w[tid] = tid < a.Hi ? __ldg(a.w + (int64_t)t * a.Hi + tid) : 0.0f;
        for (int i = tid; i < 64 * 16; i += kThreads) {  // (head, chunk, 16-byte unit)
            const int h = i >> 4, c = (i >> 3) & 1, u = i & 7;
            const bool in = h < a.Hi;
            const __nv_bfloat16 *src =
                in ? a.q + ((int64_t)t * a.Hi + h) * 128 + 64 * c + 8 * u : a.q;
            tc::cp_async16_zfill(smem + kOffQ + c * 8192 + sw_off(h, u), src, in ? 16u : 0u);
        }
        tc::cp_async_commit_wait_all();
        __syncthreads();
        const int32_t b = ms->info[0];

        // ---- compact the valid entries, in list order ----
        int32_t n = 0;
        float mass_part = 0.0f;
        if (b >= 0) {
            const int32_t pos = t - ms->info[1], c_lo = ms->info[2], c_hi = ms->info[3];
            const int32_t *lst = a.idx + (int64_t)t * a.topk;
            const float *tgt = a.l1 + (int64_t)t * a.topk;
            for (int32_t base = 0; base < a.topk; base += kThreads) {
                const int32_t e = base + tid;
                int32_t j = -1;
                float pv = 0.0f;
                bool in = false;
                if (e < a.topk) {
                    j = __ldg(lst + e);
                    in = j >= c_lo && j < c_hi &&
                         (int64_t)(j - c_lo + 1) * a.cmp_ratio <= (int64_t)pos + 1;
                    if (in) pv = __ldg(tgt + e);
                }
                int32_t total = 0;
                const int32_t before = block_exclusive_scan<kThreads>(in ? 1 : 0, ms->scan, &total);
                if (in) {
                    ms->rows[n + before] = j;
                    ms->p[n + before] = pv;
                    mass_part += pv;
                }
                n += total;
            }
        }
        const float mass = block_sum_tc(mass_part, ms->red);
        float *dq_out = a.d_q + (int64_t)t * a.Hi * 128;
        if (n == 0 || !(mass > 0.0f)) {
            for (int e = tid; e < a.Hi * 128; e += kThreads) dq_out[e] = 0.0f;
            if (tid < a.Hi) a.d_w[(int64_t)t * a.Hi + tid] = 0.0f;
            if (tid == 0 && a.loss) a.loss[t] = 0.0f;
            __syncthreads();
            continue;
        }
        const float inv_mass = 1.0f / mass;

        // ---- pass 1: scores from S^T ----
        for (int32_t r0 = 0; r0 < n && ok; r0 += kRows) {
            load_tile(r0, n);
            issue_scores();
            if (!(ok = sync_mma())) break;
            float sv[32];
            tc::tmem_ld32(lane_base + kColS + 32 * hf, sv);
            tc::tmem_wait_ld();
            if (lane < 16) {
                float part = 0.0f;
#pragma unroll
                for (int i = 0; i < 32; ++i) part = fmaf(ms->w[32 * hf + i], fmaxf(sv[i], 0.0f), part);
                ms->part[hf][16 * q4 + lane] = part;
            }
            tc::tc_fence_before();
            __syncthreads();
            if (tid < kRows && r0 + tid < n) ms->dl[r0 + tid] = ms->part[0][tid] + ms->part[1][tid];
            __syncthreads();  // the K tile and the partial sums are rewritten next
        }
        if (!ok) break;

        // ---- log-softmax over the entries, loss, dL/dI ----
        float mx = -INFINITY;
        for (int i = tid; i < n; i += kThreads) mx = fmaxf(mx, ms->dl[i]);
        mx = block_max_tc(mx, ms->red);
        float z = 0.0f;
        for (int i = tid; i < n; i += kThreads) z += expf(ms->dl[i] - mx);
        z = block_sum_tc(z, ms->red);
        const float lz = mx + logf(z);
        float kl = 0.0f;
        for (int i = tid; i < n; i += kThreads) {
            const float ps = ms->p[i] * inv_mass;
            const float log_pi = ms->dl[i] - lz;
            if (ps > 0.0f) kl += ps * (logf(ps) - log_pi);
            ms->dl[i] = a.grad_scale * (expf(log_pi) - ps);
        }
        kl = block_sum_tc(kl, ms->red);
        if (tid == 0 && a.loss) a.loss[t] = kl;

        // ---- pass 2: G, d_w, d_q^T (accumulated), d_k (per tile) ----
        float dw_acc = 0.0f;  // head tid (tid < 64)
        for (int32_t r0 = 0; r0 < n && ok; r0 += kRows) {
            const int nr = min(kRows, n - r0);
            load_tile(r0, n);
            issue_scores();
            if (!(ok = sync_mma())) break;
            {
                float sv[32];
                tc::tmem_ld32(lane_base + kColS + 32 * hf, sv);
                tc::tmem_wait_ld();
                const int r = 16 * q4 + lane;  // meaningful for lane < 16
                const bool row_ok = lane < 16 && r < nr;
                const float g = row_ok ? ms->dl[r0 + r] : 0.0f;
                // d_w partials: sum over this quarter's 16 rows, per head of the half
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    float v = row_ok ? g * fmaxf(sv[i], 0.0f) : 0.0f;
                    v += __shfl_xor_sync(0xffffffffu, v, 8);
                    v += __shfl_xor_sync(0xffffffffu, v, 4);
                    v += __shfl_xor_sync(0xffffffffu, v, 2);
                    v += __shfl_xor_sync(0xffffffffu, v, 1);
                    if (lane == 0) ms->dwp[q4][32 * hf + i] = v;
                }
                if (lane < 16) {
                    uint32_t gh[16], gl[16];
#pragma unroll
                    for (int i = 0; i < 32; i += 2) {
                        const int h = 32 * hf + i;
                        const float g0 = (row_ok && sv[i] > 0.0f) ? g * ms->w[h] : 0.0f;
                        const float g1 = (row_ok && sv[i + 1] > 0.0f) ? g * ms->w[h + 1] : 0.0f;
                        __nv_bfloat162 hb = __floats2bfloat162_rn(g0, g1);
                        const float2 hf2 = __bfloat1622float2(hb);
                        __nv_bfloat162 lb = __floats2bfloat162_rn(g0 - hf2.x, g1 - hf2.y);
                        gh[i >> 1] = *reinterpret_cast<uint32_t *>(&hb);
                        gl[i >> 1] = *reinterpret_cast<uint32_t *>(&lb);
                    }
#pragma unroll
                    for (int cq = 0; cq < 4; ++cq) {  // 16-byte units 4 hf .. 4 hf + 3 of row r
                        *reinterpret_cast<uint4 *>(smem + kOffG + sw_off(r, 4 * hf + cq)) =
                            make_uint4(gh[4 * cq], gh[4 * cq + 1], gh[4 * cq + 2], gh[4 * cq + 3]);
                        *reinterpret_cast<uint4 *>(smem + kOffGlo + sw_off(r, 4 * hf + cq)) =
                            make_uint4(gl[4 * cq], gl[4 * cq + 1], gl[4 * cq + 2], gl[4 * cq + 3]);
                    }
                }
            }
            tc::tc_fence_before();
            tc::fence_proxy_async_smem();
            __syncthreads();
            if (tid < 64)
                dw_acc += (ms->dwp[0][tid] + ms->dwp[1][tid]) + (ms->dwp[2][tid] + ms->dwp[3][tid]);
            if (tid == 0) {
                tc::tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)  // d_q^T += K^T G_hi: K = 64 rows
                    tc::mma_bf16(tmem + kColDQ, tc::desc_add(d_k_mn, kk * 2048),
                                 tc::desc_add(d_g_mn, kk * 2048), id_dq, (r0 > 0 || kk > 0));
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)  // d_q^T += K^T G_lo
                    tc::mma_bf16(tmem + kColDQ, tc::desc_add(d_k_mn, kk * 2048),
                                 tc::desc_add(d_gl_mn, kk * 2048), id_dq, 1);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)  // d_k = G_hi q: K = 64 heads
                    tc::mma_bf16(tmem + kColDK, tc::desc_add(d_g_km, kk * 32),
                                 tc::desc_add(d_q_mn, kk * 2048), id_dk, kk > 0);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)  // d_k += G_lo q
                    tc::mma_bf16(tmem + kColDK, tc::desc_add(d_gl_km, kk * 32),
                                 tc::desc_add(d_q_mn, kk * 2048), id_dk, 1);
            }
            if (!(ok = sync_mma())) break;
            // rows 16 q4 + lane (lane < 16), dims 64 hf .. 64 hf + 63, staged
            {
                float *stage = reinterpret_cast<float *>(smem + kOffStage);
                float v0[32], v1[32];
                tc::tmem_ld32(lane_base + kColDK + 64 * hf, v0);
                tc::tmem_ld32(lane_base + kColDK + 64 * hf + 32, v1);
                tc::tmem_wait_ld();
                if (lane < 16) {
                    float *row = stage + (16 * q4 + lane) * kStageStride + 64 * hf;
#pragma unroll
                    for (int i = 0; i < 32; i += 4) {
                        *reinterpret_cast<float4 *>(row + i) = make_float4(v0[i], v0[i + 1], v0[i + 2], v0[i + 3]);
                        *reinterpret_cast<float4 *>(row + 32 + i) =
                            make_float4(v1[i], v1[i + 1], v1[i + 2], v1[i + 3]);
                    }
                }
                tc::tc_fence_before();
                __syncthreads();
                // 64 rows x 32 float4: a warp adds 512 contiguous bytes of one row
                for (int i = tid; i < kRows * 32; i += kThreads) {
                    const int r = i >> 5, c4 = i & 31;
                    if (r < nr)
                        atomicAdd(reinterpret_cast<float4 *>(a.d_k + (int64_t)ms->rows[r0 + r] * 128 + 4 * c4),
                                  *reinterpret_cast<const float4 *>(stage + r * kStageStride + 4 * c4));
                }
                __syncthreads();  // stage, G, the K tile and TMEM columns are rewritten next
            }
        }
        if (!ok) break;
        // d_q: dims 32 q4 + lane, heads 32 hf .. 32 hf + 31
        {
            float v[32];
            tc::tmem_ld32(lane_base + kColDQ + 32 * hf, v);
            tc::tmem_wait_ld();
            const int d = 32 * q4 + lane;
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                const int h = 32 * hf + i;
                if (h < a.Hi) dq_out[h * 128 + d] = v[i];
            }
        }
        if (tid < a.Hi) a.d_w[(int64_t)t * a.Hi + tid] = dw_acc;
        tc::tc_fence_before();
        __syncthreads();  // TMEM, q, w and the lists are rewritten by the next token
        tc::tc_fence_after();
    }
    // teardown: every MMA issued has completed before tensor memory is freed
    if (tid == 0) {
        tc::mma_commit(&ms->bar);
        if (!tc::mbar_wait(&ms->bar, n_commit & 1)) report_error(a.err, kErrTimeout, kKerIndexerKl, 11);
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    if (warp == 0) tc::tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

// Di == 128 and Hi <= 64 only; d_k must already be zeroed.
cudaError_t launch_indexer_kl_grad_tc(const IndexerKlArgs &a, cudaStream_t stream) {
    if (a.T == 0) return cudaSuccess;
    if (a.Di != 128 || a.Hi > 64 || a.topk > kMaxList) return cudaErrorInvalidValue;
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(indexer_kl_grad_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    const int64_t want = 2 * (int64_t)sms;
    const int ctas = (int)(a.T < want ? a.T : want);
    indexer_kl_grad_tc_kernel<<<ctas, kThreads, kSmemBytes, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace csa
