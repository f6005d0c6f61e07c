// Lightning-indexer score + per-sequence causal top-k over compressed KV.
//
// Sources: hyper-parallel RFC "DeepSeek-V4 CSA/HCA 自定义算子接入…", section 1
// (lightning_indexer schema: q, k, w, topk, cu_seqlens_q, cu_seqlens_k,
// cmp_ratio, return_value); miles PR 2038 report, motivation item 4 (score the
// query's own sequence only) and review notes (stream-absolute indices).
// Score (the pages print no formula; reading):
//     s(t, j) = sum_h w[t,h] * max(0, q[t,h,:] . k[j,:])
// over the compressed rows j of t's own sequence whose pooled tokens all lie at
// or before t. Top-k: ties to the lower row, output in ascending row order,
// -1 / -inf padding.
//
// One CTA owns one token at a time (persistent grid). Scores live in shared
// memory (global scratch beyond kScoreCap candidates); the K-th largest is
// found by a 4-pass 8-bit radix select on order-preserving uint32 keys, and
// the winners are emitted in row order with two block scans.
#include "common.cuh"
#include "internal.h"

namespace csa {

namespace {

constexpr int kThreads = 256;
constexpr int kScoreCap = 40960;        // candidates kept in shared memory
constexpr int kMaxCtas = 1024;          // persistent grid bound (sizes the scratch)
constexpr int kMaxHi = 64, kMaxDi = 128;

struct Smem {
    float q[kMaxHi * kMaxDi];
    float w[kMaxHi];
    int32_t hist[256];
    int32_t scan[kThreads / 32 + 1];
    uint32_t sel_digit;
    int32_t sel_above;
};

template <int DI>
__device__ __forceinline__ float score_row(const Smem &sm, const __nv_bfloat16 *__restrict__ krow,
                                           int hi) {
    // row of k in registers (bf16 pairs), q broadcast from shared memory
    __nv_bfloat162 kr[DI / 2];
    const uint4 *src = reinterpret_cast<const uint4 *>(krow);
#pragma unroll
    for (int v = 0; v < DI / 8; ++v) {
        uint4 x = __ldg(src + v);
        kr[4 * v + 0] = *reinterpret_cast<__nv_bfloat162 *>(&x.x);
        kr[4 * v + 1] = *reinterpret_cast<__nv_bfloat162 *>(&x.y);
        kr[4 * v + 2] = *reinterpret_cast<__nv_bfloat162 *>(&x.z);
        kr[4 * v + 3] = *reinterpret_cast<__nv_bfloat162 *>(&x.w);
    }
    float s = 0.0f;
    for (int h = 0; h < hi; ++h) {
        const float2 *qh = reinterpret_cast<const float2 *>(sm.q + h * DI);
        float dot = 0.0f;
#pragma unroll
        for (int p = 0; p < DI / 2; ++p) {
            float2 qq = qh[p];
            float2 kk = __bfloat1622float2(kr[p]);
            dot = fmaf(qq.x, kk.x, dot);
            dot = fmaf(qq.y, kk.y, dot);
        }
        s = fmaf(sm.w[h], fmaxf(dot, 0.0f), s);
    }
    return s;
}

// Returns the exact key of the K-th largest element (radix select, MSB first)
// and, through *take_eq, how many elements equal to it belong to the top K.
__device__ uint32_t radix_select(Smem &sm, const float *sc, int32_t n, int32_t K,
                                 int32_t *take_eq) {
    uint32_t prefix = 0, mask = 0;
    int32_t k_rem = K;
    const int lane = threadIdx.x & 31;
#pragma unroll 1
    for (int pass = 0; pass < 4; ++pass) {
        const int shift = 24 - 8 * pass;
        for (int i = threadIdx.x; i < 256; i += kThreads) sm.hist[i] = 0;
        __syncthreads();
        for (int32_t i = threadIdx.x; i < n; i += kThreads) {
            uint32_t u = float_key(sc[i]);
            if ((u & mask) == prefix) atomicAdd(&sm.hist[(u >> shift) & 255u], 1);
        }
        __syncthreads();
        if (threadIdx.x < 32) {
            // lane L holds digits 255-8L .. 248-8L (descending)
            int32_t c[8], local = 0;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                c[i] = sm.hist[255 - (lane * 8 + i)];
                local += c[i];
            }
            int32_t incl = local;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                int32_t y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += y;
            }
            int32_t above = incl - local;  // elements with a larger digit than this lane's first
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                if (above < k_rem && k_rem <= above + c[i]) {
                    sm.sel_digit = 255u - (uint32_t)(lane * 8 + i);
                    sm.sel_above = above;
                }
                above += c[i];
            }
        }
        __syncthreads();
        const uint32_t d = sm.sel_digit;
        k_rem -= sm.sel_above;
        prefix |= d << shift;
        mask |= 255u << shift;
        __syncthreads();
    }
    *take_eq = k_rem;
    return prefix;
}

// Writes the selected rows of one token in ascending order.
__device__ void emit_topk(Smem &sm, const float *sc, int32_t n, int32_t K, int32_t base,
                          int32_t *__restrict__ idx_row, float *__restrict__ val_row) {
    if (n <= K) {
        for (int32_t i = threadIdx.x; i < K; i += kThreads) {
            idx_row[i] = i < n ? base + i : -1;
            if (val_row) val_row[i] = i < n ? sc[i] : -INFINITY;
        }
        return;
    }
    int32_t take_eq;
    const uint32_t tau = radix_select(sm, sc, n, K, &take_eq);
    const int32_t per = (n + kThreads - 1) / kThreads;
    const int32_t c0 = min(n, (int32_t)threadIdx.x * per), c1 = min(n, c0 + per);
    int32_t gt = 0, eq = 0;
    for (int32_t i = c0; i < c1; ++i) {
        uint32_t u = float_key(sc[i]);
        gt += u > tau;
        eq += u == tau;
    }
    int32_t total;
    const int32_t eq_before = block_exclusive_scan<kThreads>(eq, sm.scan, &total);
    const int32_t my_eq = max(0, min(eq, take_eq - eq_before));
    int32_t pos = block_exclusive_scan<kThreads>(gt + my_eq, sm.scan, &total);
    int32_t eq_seen = 0;
    for (int32_t i = c0; i < c1; ++i) {
        uint32_t u = float_key(sc[i]);
        bool take = u > tau;
        if (u == tau) {
            take = eq_seen < my_eq;
            ++eq_seen;
        }
        if (take && pos < K) {  // exactly K are taken; the bound only guards the row
            idx_row[pos] = base + i;
            if (val_row) val_row[pos] = sc[i];
            ++pos;
        }
    }
}

template <int DI>
__global__ void __launch_bounds__(kThreads, 1) indexer_topk_kernel(IndexerArgs a) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    Smem &sm = *reinterpret_cast<Smem *>(smem_raw);
    float *sc_smem = reinterpret_cast<float *>(smem_raw + sizeof(Smem));
    for (int32_t t = blockIdx.x; t < a.T; t += gridDim.x) {
        int32_t *idx_row = a.topk_idx + (int64_t)t * a.topk;
        float *val_row = a.topk_val ? a.topk_val + (int64_t)t * a.topk : nullptr;
        const int32_t b = find_segment(a.cu_q, a.batch, t);
        int32_t n = 0, base = 0;
        if (b < 0) {
            if (threadIdx.x == 0) report_error(a.err, kErrCheck, kKerIndexer, 1);
        } else if (a.Tc > 0) {
            const int32_t pos = t - __ldg(a.cu_q + b);
            base = __ldg(a.cu_c + b);
            const int32_t seg_blocks = __ldg(a.cu_c + b + 1) - base;
            n = min((pos + 1) / a.cmp_ratio, seg_blocks);
            if (base < 0 || n < 0 || base + n > a.Tc) {
                if (threadIdx.x == 0) report_error(a.err, kErrCheck, kKerIndexer, 2);
                n = 0;
            }
        }
        if (n == 0) {
            for (int32_t i = threadIdx.x; i < a.topk; i += kThreads) {
                idx_row[i] = -1;
                if (val_row) val_row[i] = -INFINITY;
            }
            continue;
        }
        float *sc = n <= kScoreCap ? sc_smem : a.scratch + (int64_t)blockIdx.x * a.Tc;
        if (n > kScoreCap && a.scratch == nullptr) {
            if (threadIdx.x == 0) report_error(a.err, kErrCheck, kKerIndexer, 3);
            continue;
        }
        __syncthreads();  // previous token done with shared memory
        const __nv_bfloat16 *qt = a.q + (int64_t)t * a.Hi * DI;
        for (int i = threadIdx.x; i < a.Hi * DI; i += kThreads) sm.q[i] = __bfloat162float(qt[i]);
        for (int i = threadIdx.x; i < a.Hi; i += kThreads) sm.w[i] = a.w[(int64_t)t * a.Hi + i];
        __syncthreads();
        for (int32_t j = threadIdx.x; j < n; j += kThreads)
            sc[j] = score_row<DI>(sm, a.k + (int64_t)(base + j) * DI, a.Hi);
        __syncthreads();
        emit_topk(sm, sc, n, a.topk, base, idx_row, val_row);
        __syncthreads();
    }
}

}  // namespace

int32_t indexer_scratch_rows_threshold() { return kScoreCap; }

size_t indexer_workspace_bytes(int32_t T, int32_t Tc, int32_t, int32_t, int32_t) {
    if (Tc <= kScoreCap || T <= 0) return 0;
    const int64_t ctas = T < kMaxCtas ? T : kMaxCtas;
    return (size_t)ctas * (size_t)Tc * sizeof(float);
}

cudaError_t launch_indexer_topk(const IndexerArgs &a, cudaStream_t stream) {
    if (a.T == 0) return cudaSuccess;
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    int ctas = a.T < sms ? a.T : sms;
    if (ctas > kMaxCtas) ctas = kMaxCtas;
    if (a.max_ctas > 0 && ctas > a.max_ctas) ctas = a.max_ctas;
    const size_t smem = sizeof(Smem) + (size_t)kScoreCap * sizeof(float);
    if (a.Di == 64) {
        e = cudaFuncSetAttribute(indexer_topk_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        indexer_topk_kernel<64><<<ctas, kThreads, smem, stream>>>(a);
    } else {
        e = cudaFuncSetAttribute(indexer_topk_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        indexer_topk_kernel<128><<<ctas, kThreads, smem, stream>>>(a);
    }
    return cudaGetLastError();
}

}  // namespace csa
