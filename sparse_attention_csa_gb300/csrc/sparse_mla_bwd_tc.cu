// Backward of the shared-KV MLA sparse attention with sinks on the tensor
// cores (sm_103a, tcgen05 + TMEM).
//
// What it computes is stated with the entry point (the gradient call the miles
// PR 2038 report and the hyper-parallel RFC list as sparse_flash_mla_grad):
// with P_a = exp(scale q.k_a - lse), P_sink = exp(sink - lse), Dv = dout.out,
//   dS_a = P_a (dout.k_a - Dv),   d_q = scale sum_a dS_a k_a,
//   d_row_a += scale dS_a q + P_a dout,   d_sink -= P_sink Dv,
//   l1[slot of a] += P_a / H.
//
// Design. A persistent grid, one CTA (256 threads) per SM, tokens strided over
// the CTAs. Per token, q and dout rows of all 64 heads (zero past H) sit in
// shared memory in the 128-byte-swizzled K-major layout the forward uses for Q
// (8 chunks of 64 dims x 64 rows). Keys go by tiles of 64 rows (the same
// layout, 8 KB chunks). Per tile, one thread issues:
//   S^T  = K q^T     M=64 keys x N=64 heads, K=512     TMEM cols   0..63
//   dP^T = K dout^T  same shape                        TMEM cols  64..127
// The 256 threads turn them into P and scale*dS (bf16, one 128-byte row per
// key: the K-major A operand and the MN-major B operand below), then:
//   dq^T += K^T (scale dS^T)  M=128 dims x N=64 heads, K=64 keys, four dim
//                             slabs, accumulated over the token's tiles
//                                                      TMEM cols 128..383
//   dkv  = (scale dS^T) q + P^T dout  M=64 keys x N=128 dims, K=64 heads, a
//                             quarter of the 512 dims at a time
//                                                      TMEM cols 384..511
// Each quarter is read out of TMEM and added to the fp32 row gradients with
// float4 atomics straight from registers (rows are shared between tokens),
// while the next quarter's MMAs run; the next key tile's copies go in flight
// as soon as this tile's dq^T MMAs are done with the key buffer.
// M=64 accumulators put row r in TMEM lane 32 (r / 16) + r % 16. Every wait is
// bounded; on a timeout the CTA records the error, drains its MMAs and frees
// TMEM.
#include <math.h>

#include "common.cuh"
#include "internal.h"
#include "tc_ptx.cuh"

namespace csa {

namespace {

constexpr int kTcThreads = 256;
constexpr int kTcKeys = 64;          // keys per tile
constexpr int kTcMaxList = 1024;     // top-k entries kept per token
constexpr int kTcMaxWin = 1024;      // window rows per token
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0, kColDP = 64, kColDQ = 128, kColDK = 384;
constexpr float kLog2eBwd = 1.4426950408889634f;

// Shared memory (offsets from a 1024-byte aligned base).
constexpr uint32_t kOffQ = 0;                  // 8 x [64 heads x 128 B]
constexpr uint32_t kOffG = 65536;              // dout, same layout
constexpr uint32_t kOffK = 131072;             // 8 x [64 keys x 128 B]
constexpr uint32_t kOffP = 196608;             // [64 keys x 128 B] bf16 P
constexpr uint32_t kOffDS = 204800;            // [64 keys x 128 B] bf16 scale*dS
constexpr uint32_t kOffMisc = 212992;

struct TcMisc {
    uint64_t bar;
    uint32_t tmem_base;
    int32_t n_cmp;
    int32_t abort;
    float dv[64];
    float lse2[64];  // lse in base 2
    float l1[kTcMaxWin + kTcMaxList];
    int32_t rows[kTcMaxList];
    int32_t slots[kTcMaxList];
};
constexpr size_t kTcSmemBytes = kOffMisc + sizeof(TcMisc) + 1024;
static_assert(kTcSmemBytes <= 232448, "shared memory budget");

// byte offset of 16-byte unit u (0..7) of row r in a 128-byte-swizzled chunk
__device__ __forceinline__ uint32_t sw_off(uint32_t r, uint32_t u) {
    return r * 128u + ((u ^ (r & 7u)) << 4);
}


__global__ void __launch_bounds__(kTcThreads, 1) sparse_mla_bwd_tc_kernel(MlaBwdArgs a) {
    extern __shared__ unsigned char raw[];
    unsigned char *smem =
        reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~(uintptr_t)1023);
    TcMisc *ms = reinterpret_cast<TcMisc *>(smem + kOffMisc);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int q4 = warp & 3, hf = warp >> 2;  // TMEM lane quarter, column half
    const bool use_cmp = a.cmp_kv != nullptr && a.Tc > 0;
    const int32_t W = a.window;
    const float scale = a.softmax_scale;
    const float c2 = scale * kLog2eBwd;  // P = 2^(c2 s - lse log2 e)

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

    const uint32_t s_q = tc::smem_u32(smem + kOffQ), s_g = tc::smem_u32(smem + kOffG);
    const uint32_t s_k = tc::smem_u32(smem + kOffK), s_p = tc::smem_u32(smem + kOffP);
    const uint32_t s_ds = tc::smem_u32(smem + kOffDS);
    // operand descriptors: K-major (rows of 128 B), MN-major (64-element blocks 8 KB apart)
    const uint64_t d_k_km = tc::smem_desc(s_k, 16, 1024);
    const uint64_t d_q_km = tc::smem_desc(s_q, 16, 1024);
    const uint64_t d_g_km = tc::smem_desc(s_g, 16, 1024);
    const uint64_t d_k_mn = tc::smem_desc(s_k, 8192, 1024);
    const uint64_t d_q_mn = tc::smem_desc(s_q, 8192, 1024);
    const uint64_t d_g_mn = tc::smem_desc(s_g, 8192, 1024);
    const uint64_t d_ds_km = tc::smem_desc(s_ds, 16, 1024);
    const uint64_t d_p_km = tc::smem_desc(s_p, 16, 1024);
    const uint64_t d_ds_mn = tc::smem_desc(s_ds, 8192, 1024);
    constexpr uint32_t id_s = tc::idesc_bf16(64, 64, false, false);
    constexpr uint32_t id_dq = tc::idesc_bf16(128, 64, true, true);
    constexpr uint32_t id_dk = tc::idesc_bf16(64, 128, false, true);

    uint32_t n_commit = 0;
    bool ok = true;
    // every thread waits for the MMAs committed so far
    auto sync_mma = [&]() -> bool {
        if (tid == 0) tc::mma_commit(&ms->bar);
        const bool w = tc::mbar_wait(&ms->bar, n_commit & 1);
        ++n_commit;
        if (!w) {
            ms->abort = 1;
            report_error(a.err, kErrTimeout, kKerMlaBwd, 10);
        }
        __syncthreads();
        tc::tc_fence_after();
        return ms->abort == 0;
    };

    for (int32_t t = blockIdx.x; t < a.T && ok; t += gridDim.x) {
        const int32_t b = find_segment(a.cu_q, a.batch, t);
        if (b < 0) {  // not covered by any sequence: report, zero d_q
            if (tid == 0) report_error(a.err, kErrCheck, kKerMlaBwd, 1);
            for (int i = tid; i < a.H * 512; i += kTcThreads) a.d_q[(int64_t)t * a.H * 512 + i] = 0.0f;
            continue;
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
        if (use_cmp && a.cmp_idx) {
            if (warp == 0) {
                int32_t n = 0;
                const int32_t *row = a.cmp_idx + (int64_t)t * a.topk;
                for (int32_t e0 = 0; e0 < a.topk; e0 += 32) {
                    const int32_t e = e0 + lane;
                    const int32_t j = e < a.topk ? __ldg(row + e) : -1;
                    const bool in = j >= cbase && j < cbase + vis;
                    const uint32_t m = __ballot_sync(0xffffffffu, in);
                    if (in) {
                        const int32_t at = n + __popc(m & ((1u << lane) - 1u));
                        ms->rows[at] = j;
                        ms->slots[at] = e;
                    }
                    n += __popc(m);
                }
                if (lane == 0) ms->n_cmp = n;
            }
        } else if (tid == 0) {
            ms->n_cmp = vis;
        }
        for (int i = tid; i < kTcMaxWin + kTcMaxList; i += kTcThreads) ms->l1[i] = 0.0f;
        // q and dout rows of the token (zero past H), swizzled K-major, by
        // cp.async: every thread's 32 copies are in flight at once
        for (int i = tid; i < 64 * 64; i += kTcThreads) {  // (head, 16-byte unit of 64)
            const int h = i >> 6, c = (i >> 3) & 7, u = i & 7;
            const int64_t o = ((int64_t)t * a.H + min(h, a.H - 1)) * 512 + 64 * c + 8 * u;
            const uint32_t bytes = h < a.H ? 16u : 0u;
            tc::cp_async16_zfill(smem + kOffQ + c * 8192 + sw_off(h, u), a.q + o, bytes);
            tc::cp_async16_zfill(smem + kOffG + c * 8192 + sw_off(h, u), a.dout + o, bytes);
        }
        // Dv = dout . out per head while they land (8 heads per warp, two at a
        // time, 16 dims per lane in 16-byte loads); lse; the sink's gradient
        for (int j0 = 0; j0 < 8; j0 += 2) {
            uint4 gv[2][2], ov[2][2];
#pragma unroll
            for (int jj = 0; jj < 2; ++jj) {
                const int h = warp + 8 * (j0 + jj);
                const int64_t o = ((int64_t)t * a.H + min(h, a.H - 1)) * 512 + 16 * lane;
                gv[jj][0] = __ldg(reinterpret_cast<const uint4 *>(a.dout + o));
                gv[jj][1] = __ldg(reinterpret_cast<const uint4 *>(a.dout + o + 8));
                ov[jj][0] = __ldg(reinterpret_cast<const uint4 *>(a.out + o));
                ov[jj][1] = __ldg(reinterpret_cast<const uint4 *>(a.out + o + 8));
            }
#pragma unroll
            for (int jj = 0; jj < 2; ++jj) {
                const int h = warp + 8 * (j0 + jj);
                float s = 0.0f;
#pragma unroll
                for (int k = 0; k < 2; ++k) {
                    const __nv_bfloat162 *g2 = reinterpret_cast<const __nv_bfloat162 *>(&gv[jj][k]);
                    const __nv_bfloat162 *o2 = reinterpret_cast<const __nv_bfloat162 *>(&ov[jj][k]);
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float2 gf = __bfloat1622float2(g2[e]), of = __bfloat1622float2(o2[e]);
                        s = fmaf(gf.x, of.x, s);
                        s = fmaf(gf.y, of.y, s);
                    }
                }
                s = h < a.H ? warp_sum(s) : 0.0f;
                if (lane == 0) {
                    const float lse = h < a.H ? a.lse[(int64_t)t * a.H + h] : 0.0f;
                    ms->dv[h] = s;
                    ms->lse2[h] = lse * kLog2eBwd;
                    if (h < a.H && a.sinks && a.d_sinks) {
                        const float sk = __ldg(a.sinks + h);
                        if (sk != -INFINITY) atomicAdd(a.d_sinks + h, -expf(sk - lse) * s);
                    }
                }
            }
        }
        tc::cp_async_commit_wait_all();
        __syncthreads();
        const int32_t n_cmp = ms->n_cmp;
        const int32_t n_keys = n_win + n_cmp;
        auto key_row = [&](int32_t key) -> int64_t {  // packed row of key (window or compressed)
            if (key < n_win) return start + key;
            return a.cmp_idx ? ms->rows[key - n_win] : cbase + key - n_win;
        };

        // the key tile from key k0, swizzled K-major, by cp.async (every
        // thread's 16 copies in flight at once); rows past the last key are zero
        auto load_tile = [&](int32_t k0) {
            const int nk = min(kTcKeys, n_keys - k0);
            for (int i = tid; i < kTcKeys * 64; i += kTcThreads) {
                const int r = i >> 6, c = (i >> 3) & 7, u = i & 7;
                const __nv_bfloat16 *src = a.ori_kv;
                uint32_t bytes = 0;
                if (r < nk) {
                    const int32_t key = k0 + r;
                    src = (key < n_win ? a.ori_kv : a.cmp_kv) + key_row(key) * 512 + 64 * c + 8 * u;
                    bytes = 16;
                }
                tc::cp_async16_zfill(smem + kOffK + c * 8192 + sw_off(r, u), src, bytes);
            }
        };
        if (n_keys > 0) load_tile(0);
        for (int32_t k0 = 0; k0 < n_keys && ok; k0 += kTcKeys) {
            const int nk = min(kTcKeys, n_keys - k0);
            // this tile's copies (issued here for the first tile, under the
            // previous tile's row gradients for the others)
            tc::cp_async_commit_wait_all();
            tc::fence_proxy_async_smem();
            __syncthreads();
            if (tid == 0) {
                tc::tc_fence_after();
#pragma unroll
                for (int c = 0; c < 8; ++c)
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint32_t off_k = c * 8192 + kk * 32;
                        tc::mma_bf16(tmem + kColS, tc::desc_add(d_k_km, off_k), tc::desc_add(d_q_km, off_k),
                                     id_s, (c | kk) != 0);
                        tc::mma_bf16(tmem + kColDP, tc::desc_add(d_k_km, off_k), tc::desc_add(d_g_km, off_k),
                                     id_s, (c | kk) != 0);
                    }
            }
            if (!(ok = sync_mma())) break;
            // P and scale*dS for the key rows this warp's lane quarter holds
            // (lanes 0-15: rows 16 q4 + lane), heads 32 hf .. 32 hf + 31
            {
                float sv[32], pv[32];
                tc::tmem_ld32(lane_base + kColS + 32 * hf, sv);
                tc::tmem_ld32(lane_base + kColDP + 32 * hf, pv);
                tc::tmem_wait_ld();
                if (lane < 16) {
                    const int r = 16 * q4 + lane;
                    const bool key_ok = r < nk;
                    float psum = 0.0f;
                    uint32_t pw[16], dw[16];
#pragma unroll
                    for (int i = 0; i < 32; i += 2) {
                        const int h = 32 * hf + i;
                        float p0 = 0.0f, p1 = 0.0f, d0 = 0.0f, d1 = 0.0f;
                        if (key_ok && h < a.H) {
                            p0 = tc::ex2_approx(fmaf(c2, sv[i], -ms->lse2[h]));
                            d0 = scale * p0 * (pv[i] - ms->dv[h]);
                        }
                        if (key_ok && h + 1 < a.H) {
                            p1 = tc::ex2_approx(fmaf(c2, sv[i + 1], -ms->lse2[h + 1]));
                            d1 = scale * p1 * (pv[i + 1] - ms->dv[h + 1]);
                        }
                        psum += p0 + p1;
                        __nv_bfloat162 pb = __floats2bfloat162_rn(p0, p1);
                        __nv_bfloat162 db = __floats2bfloat162_rn(d0, d1);
                        pw[i >> 1] = *reinterpret_cast<uint32_t *>(&pb);
                        dw[i >> 1] = *reinterpret_cast<uint32_t *>(&db);
                    }
#pragma unroll
                    for (int cq = 0; cq < 4; ++cq) {  // 16-byte units 4 hf .. 4 hf + 3 of row r
                        const uint32_t off = sw_off(r, 4 * hf + cq);
                        *reinterpret_cast<uint4 *>(smem + kOffP + off) =
                            make_uint4(pw[4 * cq], pw[4 * cq + 1], pw[4 * cq + 2], pw[4 * cq + 3]);
                        *reinterpret_cast<uint4 *>(smem + kOffDS + off) =
                            make_uint4(dw[4 * cq], dw[4 * cq + 1], dw[4 * cq + 2], dw[4 * cq + 3]);
                    }
                    const int32_t key = k0 + r;
                    if (key_ok && (key < n_win || a.cmp_idx)) atomicAdd(&ms->l1[key], psum);
                }
            }
            tc::tc_fence_before();
            tc::fence_proxy_async_smem();
            __syncthreads();
            // dq^T over this tile's keys, then the rows' gradient a quarter at a time
            for (int qd = 0; qd < 4 && ok; ++qd) {
                if (tid == 0) {
                    tc::tc_fence_after();
                    if (qd == 0) {
#pragma unroll
                        for (int s = 0; s < 4; ++s)
#pragma unroll
                            for (int kk = 0; kk < 4; ++kk)
                                tc::mma_bf16(tmem + kColDQ + 64 * s,
                                             tc::desc_add(d_k_mn, 2 * s * 8192 + kk * 2048),
                                             tc::desc_add(d_ds_mn, kk * 2048), id_dq, (k0 > 0 || kk > 0));
                    }
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        tc::mma_bf16(tmem + kColDK, tc::desc_add(d_ds_km, kk * 32),
                                     tc::desc_add(d_q_mn, 2 * qd * 8192 + kk * 2048), id_dk, kk > 0);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        tc::mma_bf16(tmem + kColDK, tc::desc_add(d_p_km, kk * 32),
                                     tc::desc_add(d_g_mn, 2 * qd * 8192 + kk * 2048), id_dk, 1);
                }
                if (!(ok = sync_mma())) break;
                // the key tile is no longer read (the dq^T MMAs are done): the
                // next tile's copies go in flight under the row gradients
                if (qd == 0 && k0 + kTcKeys < n_keys) load_tile(k0 + kTcKeys);
                // rows 16 q4 + lane (lane < 16), dims 128 qd + 64 hf .. + 63
                float v0[32], v1[32];
                tc::tmem_ld32(lane_base + kColDK + 64 * hf, v0);
                tc::tmem_ld32(lane_base + kColDK + 64 * hf + 32, v1);
                tc::tmem_wait_ld();
                tc::tc_fence_before();
                __syncthreads();  // the quarter's TMEM columns are rewritten next
                // added to the row's fp32 gradient from registers, while the
                // next quarter's MMAs run
                const int r = 16 * q4 + lane;
                if (lane < 16 && r < nk) {
                    const int32_t key = k0 + r;
                    float *dst = (key < n_win ? a.d_ori_kv : a.d_cmp_kv) + key_row(key) * 512 +
                                 128 * qd + 64 * hf;
#pragma unroll
                    for (int i = 0; i < 32; i += 4) {
                        atomicAdd(reinterpret_cast<float4 *>(dst + i),
                                  make_float4(v0[i], v0[i + 1], v0[i + 2], v0[i + 3]));
                        atomicAdd(reinterpret_cast<float4 *>(dst + 32 + i),
                                  make_float4(v1[i], v1[i + 1], v1[i + 2], v1[i + 3]));
                    }
                }
            }
        }
        if (!ok) break;
        // d_q: dims 128 s + 32 q4 + lane, heads 32 hf .. 32 hf + 31
        for (int s = 0; s < 4; ++s) {
            float v[32];
            tc::tmem_ld32(lane_base + kColDQ + 64 * s + 32 * hf, v);
            tc::tmem_wait_ld();
            const int d = 128 * s + 32 * q4 + lane;
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                const int h = 32 * hf + i;
                if (h < a.H) a.d_q[((int64_t)t * a.H + h) * 512 + d] = v[i];
            }
        }
        // head-averaged distributions, in the index lists' shapes
        const float inv_h = 1.0f / (float)a.H;
        if (a.ori_l1)
            for (int i = tid; i < W; i += kTcThreads)
                a.ori_l1[(int64_t)t * W + i] = i < n_win ? ms->l1[i] * inv_h : 0.0f;
        if (a.cmp_l1 && use_cmp && a.cmp_idx)
            for (int i = tid; i < n_cmp; i += kTcThreads)
                a.cmp_l1[(int64_t)t * a.topk + ms->slots[i]] = ms->l1[n_win + i] * inv_h;
        tc::tc_fence_before();
        __syncthreads();  // TMEM and the lists are rewritten by the next token
        tc::tc_fence_after();
    }
    // teardown: every MMA issued has completed before tensor memory is freed
    if (tid == 0) {
        tc::mma_commit(&ms->bar);
        if (!tc::mbar_wait(&ms->bar, n_commit & 1)) report_error(a.err, kErrTimeout, kKerMlaBwd, 11);
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    if (warp == 0) tc::tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

cudaError_t launch_sparse_mla_bwd_tc(const MlaBwdArgs &a, cudaStream_t stream) {
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(sparse_mla_bwd_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kTcSmemBytes);
    if (e != cudaSuccess) return e;
    const int ctas = a.T < sms ? a.T : sms;
    sparse_mla_bwd_tc_kernel<<<ctas, kTcThreads, kTcSmemBytes, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace csa
