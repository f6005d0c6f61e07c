// Shared-KV MLA sparse attention forward with attention sinks (sm_103a,
// tcgen05 tensor cores, TMA).
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
//
// Design (one token per CTA iteration, persistent grid, 1 CTA per SM):
//   * All H (<= 64, padded to 64) heads of a token share its key rows, so the
//     contraction is done transposed, with the keys on the MMA's M side:
//         S^T[key, h]  = K[key, :] . Q[h, :]        M=128 keys, N=64, K=512
//         O^T[d, h]   += V[key, d]^T P[key, h]      M=128 d (x4), N=64, K=128
//     K and V are the same gathered rows: one 128-key x 512 tile in shared
//     memory (SW128, K-major) serves S^T as the A operand and, read MN-major,
//     O^T as the A operand. Accumulators live in tensor memory: S^T in 64
//     columns, O^T in 4 x 64 columns.
//   * Key rows are gathered by TMA gather4 (4 rows x 128 bytes per copy) from
//     two tensor maps (ori_kv, cmp_kv). A token's key list is: its window rows,
//     padded to a multiple of 4 (padding masked), then its valid compressed
//     rows (compacted from cmp_sparse_indices, or the visible range).
//   * Warp roles: warp 0 builds key lists and issues TMA, warp 1 owns tensor
//     memory and issues tcgen05.mma (one thread), warps 2-5 run the softmax
//     (one thread per key = one TMEM lane, 64 head scores each) and the
//     epilogue (one thread per d row of O^T).
//   * Online softmax in base 2 with a lazily moved running max: a head's max
//     only moves when a tile exceeds it by more than 8 (a factor 256), so O^T
//     in tensor memory is rescaled rarely. Row sums accumulate per thread in
//     fp32 and are reduced once per token.
//   * Every mbarrier wait is bounded; a timeout records CSA_ERR_TIMEOUT, the
//     CTA drains its copies and MMAs, frees tensor memory and exits.
#include "common.cuh"
#include "internal.h"
#include "tc_ptx.cuh"
#include "tmap.h"

namespace csa {

namespace {

constexpr int kThreads = 192;  // 6 warps
constexpr int kTileKeys = 128;
constexpr int kMaxList = 2048;  // compressed indices per token (topk bound)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kLazyMax = 8.0f;  // base-2 units

// shared memory map (offsets from a 1024-byte aligned base)
constexpr uint32_t kOffKV = 0;            // 8 chunks x [128 keys x 128 B]
constexpr uint32_t kOffQ = 131072;        // 8 chunks x [64 heads x 128 B]
constexpr uint32_t kOffP = 196608;        // [128 keys x 64 heads] bf16, MN-major
constexpr uint32_t kOffList = 212992;     // kMaxList int32
constexpr uint32_t kOffMisc = kOffList + kMaxList * 4;

// tensor memory columns
constexpr uint32_t kColS = 0;
constexpr uint32_t kColO = 256;
constexpr uint32_t kTmemCols = 512;

struct TokenInfo {
    int32_t t, n_win, n_win4, n_keys, n_tiles, valid;
};

struct Misc {
    uint64_t q_full, q_empty;
    uint64_t kv_full[4], kv_empty[4];
    uint64_t s_full, p_full, o_full, drain;
    uint64_t info_full[2], info_empty[2];
    uint32_t tmem_base;
    int32_t abort;
    int32_t rescale[2];
    TokenInfo info[2];
    float red[4][64];
    float m_run[64];
    float alpha[64];
    float inv_l[64];
};

constexpr size_t kSmemBytes = kOffMisc + sizeof(Misc) + 1024;

__device__ __forceinline__ bool bar_red_and(bool v) {
    uint32_t out;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.and.pred q, 1, 128, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(out)
        : "r"((uint32_t)v)
        : "memory");
    return out != 0;
}

struct Ctx {
    Misc *m;
    int32_t *err;
    __device__ __forceinline__ bool aborted() const {
        return *reinterpret_cast<volatile int32_t *>(&m->abort) != 0;
    }
    __device__ __forceinline__ void fail(int site) const {
        *reinterpret_cast<volatile int32_t *>(&m->abort) = 1;
        report_error(err, kErrTimeout, kKerMla, site);
    }
    // bounded wait; false (and abort) on timeout or when already aborted
    __device__ __forceinline__ bool wait(uint64_t *bar, uint32_t parity, int site) const {
        if (aborted()) return false;
        if (tc::mbar_wait(bar, parity)) return true;
        fail(site);
        return false;
    }
};

// 64 values per thread -> lane L holds the warp-wide reduction of heads 2L, 2L+1.
template <bool kMax>
__device__ __forceinline__ void reduce_scatter64(const float (&x)[64], float &o0, float &o1,
                                                 int lane) {
    auto op = [](float a, float b) { return kMax ? fmaxf(a, b) : a + b; };
    float a[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        const bool hi = lane & 16;
        const float send = hi ? x[i] : x[32 + i];
        const float keep = hi ? x[32 + i] : x[i];
        a[i] = op(keep, __shfl_xor_sync(0xffffffffu, send, 16));
    }
    float b[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const bool hi = lane & 8;
        const float send = hi ? a[i] : a[16 + i];
        const float keep = hi ? a[16 + i] : a[i];
        b[i] = op(keep, __shfl_xor_sync(0xffffffffu, send, 8));
    }
    float c[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const bool hi = lane & 4;
        const float send = hi ? b[i] : b[8 + i];
        const float keep = hi ? b[8 + i] : b[i];
        c[i] = op(keep, __shfl_xor_sync(0xffffffffu, send, 4));
    }
    float d[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const bool hi = lane & 2;
        const float send = hi ? c[i] : c[4 + i];
        const float keep = hi ? c[4 + i] : c[i];
        d[i] = op(keep, __shfl_xor_sync(0xffffffffu, send, 2));
    }
    {
        const bool hi = lane & 1;
        const float s0 = hi ? d[0] : d[2], k0 = hi ? d[2] : d[0];
        const float s1 = hi ? d[1] : d[3], k1 = hi ? d[3] : d[1];
        o0 = op(k0, __shfl_xor_sync(0xffffffffu, s0, 1));
        o1 = op(k1, __shfl_xor_sync(0xffffffffu, s1, 1));
    }
}

struct Params {
    MlaArgs a;
    int32_t window;
};

__global__ void __launch_bounds__(kThreads, 1)
sparse_mla_tc_kernel(const __grid_constant__ CUtensorMap q_map,
                     const __grid_constant__ CUtensorMap ori_map,
                     const __grid_constant__ CUtensorMap cmp_map,
                     const __grid_constant__ Params P) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem =
        reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                          ~uintptr_t(1023));
    Misc *ms = reinterpret_cast<Misc *>(smem + kOffMisc);
    int32_t *list = reinterpret_cast<int32_t *>(smem + kOffList);
    const MlaArgs &a = P.a;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    Ctx cx{ms, a.err};

    // ---------------------------------------------------------------- set-up
    if (tid == 0) {
        tc::mbar_init(&ms->q_full, 1);
        tc::mbar_init(&ms->q_empty, 1);
        for (int s = 0; s < 4; ++s) {
            tc::mbar_init(&ms->kv_full[s], 1);
            tc::mbar_init(&ms->kv_empty[s], 1);
        }
        tc::mbar_init(&ms->s_full, 1);
        tc::mbar_init(&ms->p_full, 128);
        tc::mbar_init(&ms->o_full, 1);
        tc::mbar_init(&ms->drain, 1);
        for (int i = 0; i < 2; ++i) {
            tc::mbar_init(&ms->info_full[i], 1);
            tc::mbar_init(&ms->info_empty[i], 5);
        }
        ms->abort = 0;
        ms->rescale[0] = ms->rescale[1] = 0;
        tc::fence_mbar_init();
    }
    // Rows never written by a copy must hold finite values: zero Q and KV once.
    for (uint32_t i = tid; i < (kOffP - kOffKV) / 16; i += kThreads)
        reinterpret_cast<uint4 *>(smem + kOffKV)[i] = make_uint4(0, 0, 0, 0);
    tc::fence_proxy_async_smem();
    if (warp == 1) {
        tc::tmem_alloc(&ms->tmem_base, kTmemCols);
        tc::tmem_relinquish();
    }
    if (warp == 0 && lane == 0) {
        tc::tma_prefetch_desc(&q_map);
        tc::tma_prefetch_desc(&ori_map);
        tc::tma_prefetch_desc(&cmp_map);
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = ms->tmem_base;
    const bool use_cmp = a.cmp_kv != nullptr && a.Tc > 0;

    if (warp == 0) {
        // ===================================================== producer warp
        uint32_t it = 0, q_n = 0, kv_n = 0;
        for (int32_t t = blockIdx.x; t < a.T; t += gridDim.x, ++it) {
            // ---- key list of token t
            TokenInfo ti{t, 0, 0, 0, 0, 0};
            int32_t win_start = 0, cbase = 0;
            const int32_t b = find_segment(a.cu_q, a.batch, t);
            if (b < 0) {
                if (lane == 0) report_error(a.err, kErrCheck, kKerMla, 1);
            } else {
                const int32_t seg0 = max(__ldg(a.cu_q + b), 0);
                const int32_t pos = t - seg0;
                win_start = max(t - P.window + 1, seg0);
                ti.n_win = t - win_start + 1;
                ti.n_win4 = (ti.n_win + 3) & ~3;
                int32_t n_cmp = 0;
                if (use_cmp) {
                    cbase = __ldg(a.cu_c + b);
                    const int32_t seg_blocks = __ldg(a.cu_c + b + 1) - cbase;
                    int32_t vis = min((pos + 1) / a.cmp_ratio, seg_blocks);
                    if (cbase < 0 || vis < 0 || (int64_t)cbase + vis > a.Tc) {
                        if (lane == 0) report_error(a.err, kErrCheck, kKerMla, 2);
                        vis = 0;
                    }
                    if (a.cmp_idx) {
                        const int32_t *row = a.cmp_idx + (int64_t)t * a.topk;
                        for (int32_t e0 = 0; e0 < a.topk; e0 += 32) {
                            const int32_t e = e0 + lane;
                            const int32_t j = e < a.topk ? __ldg(row + e) : -1;
                            const bool ok = j >= cbase && j < cbase + vis;
                            const uint32_t m = __ballot_sync(0xffffffffu, ok);
                            if (ok) list[n_cmp + __popc(m & ((1u << lane) - 1u))] = j;
                            n_cmp += __popc(m);
                        }
                    } else {
                        n_cmp = vis;
                    }
                }
                ti.n_keys = ti.n_win4 + n_cmp;
                ti.n_tiles = (ti.n_keys + kTileKeys - 1) / kTileKeys;
                ti.valid = 1;
            }
            __syncwarp();
            // ---- publish the token
            const uint32_t slot = it & 1;
            bool ok = cx.wait(&ms->info_empty[slot], ((it >> 1) & 1) ^ 1, 10);
            if (!__all_sync(0xffffffffu, ok)) break;
            if (lane == 0) {
                ms->info[slot] = ti;
                tc::mbar_arrive(&ms->info_full[slot]);
            }
            if (!ti.valid) continue;
            // ---- Q rows of token t (H rows of 512; rows >= H stay zero)
            ok = cx.wait(&ms->q_empty, (q_n & 1) ^ 1, 11);
            if (!__all_sync(0xffffffffu, ok)) break;
            if (lane == 0) {
                tc::mbar_expect_tx(&ms->q_full, 8u * a.H * 128u);
                for (int c = 0; c < 8; ++c)
                    tc::tma_load_3d(smem + kOffQ + c * 8192, &q_map, &ms->q_full, 64 * c, 0, t);
            }
            ++q_n;
            // ---- key tiles: lane g gathers slots 4g..4g+3 of each tile
            bool broke = false;
            for (int32_t j = 0; j < ti.n_tiles; ++j, ++kv_n) {
                const int32_t s0 = j * kTileKeys + 4 * lane;
                const bool group_on = s0 < ti.n_keys;
                const int32_t left = ti.n_keys - j * kTileKeys;
                const int32_t n_groups = min(32, (left + 3) >> 2);
                // Groups never straddle the window/compressed boundary
                // (n_win4 is a multiple of 4); slots past n_keys repeat the
                // group's last real row and are masked like the padding.
                int32_t r[4] = {t, t, t, t};
                bool from_cmp = false;
                if (group_on) {
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int32_t s = min(s0 + e, ti.n_keys - 1);
                        if (s < ti.n_win) {
                            r[e] = win_start + s;
                        } else if (s < ti.n_win4) {
                            r[e] = t;  // window padding (masked)
                        } else {
                            from_cmp = true;
                            const int32_t ci = s - ti.n_win4;
                            r[e] = a.cmp_idx ? list[ci] : cbase + ci;
                        }
                    }
                }
                const CUtensorMap *map = from_cmp ? &cmp_map : &ori_map;
                for (int s = 0; s < 4; ++s) {
                    ok = cx.wait(&ms->kv_empty[s], (kv_n & 1) ^ 1, 12);
                    if (!__all_sync(0xffffffffu, ok)) {
                        broke = true;
                        break;
                    }
                    if (lane == 0) tc::mbar_expect_tx(&ms->kv_full[s], (uint32_t)n_groups * 1024u);
                    __syncwarp();
                    if (group_on) {
#pragma unroll
                        for (int cc = 0; cc < 2; ++cc) {
                            const int c = 2 * s + cc;
                            tc::tma_gather4(smem + kOffKV + c * 16384 + lane * 512, map,
                                            &ms->kv_full[s], 64 * c, r[0], r[1], r[2], r[3]);
                        }
                    }
                }
                if (broke) break;
            }
            if (broke) break;
        }
        // ---- drain: every copy issued has landed before the CTA exits
        if (lane == 0) {
            if (q_n > 0 && !tc::mbar_wait(&ms->q_full, (q_n - 1) & 1)) cx.fail(13);
            if (kv_n > 0)
                for (int s = 0; s < 4; ++s)
                    if (!tc::mbar_wait(&ms->kv_full[s], (kv_n - 1) & 1)) cx.fail(14);
        }
    } else if (warp == 1) {
        // ========================================================= MMA warp
        if (lane == 0) {
            const uint32_t id_s = tc::idesc_bf16(128, 64, false, false);
            const uint32_t id_o = tc::idesc_bf16(128, 64, true, true);
            const uint32_t kv_a = tc::smem_u32(smem + kOffKV);
            const uint32_t q_a = tc::smem_u32(smem + kOffQ);
            const uint32_t p_a = tc::smem_u32(smem + kOffP);
            uint32_t it = 0, q_n = 0, kv_n = 0, p_n = 0;
            bool issued = false;
            for (int32_t t = blockIdx.x; t < a.T; t += gridDim.x, ++it) {
                const uint32_t slot = it & 1;
                if (!cx.wait(&ms->info_full[slot], (it >> 1) & 1, 20)) break;
                const TokenInfo ti = ms->info[slot];
                tc::mbar_arrive(&ms->info_empty[slot]);
                if (!ti.valid) continue;
                if (!cx.wait(&ms->q_full, q_n & 1, 21)) break;
                ++q_n;
                bool stop = false;
                for (int32_t j = 0; j < ti.n_tiles && !stop; ++j, ++kv_n) {
                    for (int s = 0; s < 4; ++s) {
                        if (!cx.wait(&ms->kv_full[s], kv_n & 1, 22)) {
                            stop = true;
                            break;
                        }
                        tc::tc_fence_after();
#pragma unroll
                        for (int cc = 0; cc < 2; ++cc) {
                            const int c = 2 * s + cc;
#pragma unroll
                            for (int kk = 0; kk < 4; ++kk)
                                tc::mma_bf16(tmem + kColS,
                                             tc::smem_desc(kv_a + c * 16384 + kk * 32, 16, 1024),
                                             tc::smem_desc(q_a + c * 8192 + kk * 32, 16, 1024),
                                             id_s, (c | kk) != 0);
                        }
                        issued = true;
                    }
                    if (stop) break;
                    if (j == ti.n_tiles - 1) tc::mma_commit(&ms->q_empty);
                    tc::mma_commit(&ms->s_full);
                    if (!cx.wait(&ms->p_full, p_n & 1, 23)) {
                        stop = true;
                        break;
                    }
                    ++p_n;
                    tc::tc_fence_after();
                    for (int s = 0; s < 4; ++s) {
#pragma unroll
                        for (int kk = 0; kk < 8; ++kk)
                            tc::mma_bf16(tmem + kColO + 64 * s,
                                         tc::smem_desc(kv_a + 2 * s * 16384 + kk * 2048, 16384, 1024),
                                         tc::smem_desc(p_a + kk * 2048, 16384, 1024), id_o,
                                         (j > 0 || kk > 0));
                        tc::mma_commit(&ms->kv_empty[s]);
                    }
                }
                if (stop) break;
                tc::mma_commit(&ms->o_full);
            }
            if (issued) {
                // every MMA issued has completed before tensor memory is freed
                tc::mma_commit(&ms->drain);
                if (!tc::mbar_wait(&ms->drain, 0)) cx.fail(24);
            }
        }
        __syncwarp();
    } else {
        // ================================================ softmax + epilogue
        const int q4 = warp & 3;          // TMEM lane quarter of this warp
        const int row = 32 * q4 + lane;   // key slot (softmax) / d row (epilogue)
        const int ltid = tid - 64;        // 0..127
        const uint32_t lane_addr = tmem + ((uint32_t)(32 * q4) << 16);
        unsigned char *pbuf = smem + kOffP;
        const float c = a.softmax_scale * kLog2e;
        uint32_t it = 0, s_n = 0, o_n = 0, tile_ctr = 0;
        for (int32_t t = blockIdx.x; t < a.T; t += gridDim.x, ++it) {
            const uint32_t slot = it & 1;
            bool ok = cx.wait(&ms->info_full[slot], (it >> 1) & 1, 30);
            if (!bar_red_and(ok)) break;
            const TokenInfo ti = ms->info[slot];
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&ms->info_empty[slot]);
            if (!ti.valid) continue;
            if (ltid < 64) {
                const float sink = (a.sinks && ltid < a.H) ? __ldg(a.sinks + ltid) : -INFINITY;
                ms->m_run[ltid] = sink * kLog2e;
            }
            float lp[64];
#pragma unroll
            for (int h = 0; h < 64; ++h) lp[h] = 0.0f;
            bool stop = false;
            for (int32_t j = 0; j < ti.n_tiles; ++j, ++tile_ctr) {
                ok = cx.wait(&ms->s_full, s_n & 1, 31);
                if (!bar_red_and(ok)) {
                    stop = true;
                    break;
                }
                ++s_n;
                tc::tc_fence_after();
                float v[64];
                {
                    float x[32];
                    tc::tmem_ld32(lane_addr + kColS, x);
                    tc::tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; ++i) v[i] = x[i];
                    tc::tmem_ld32(lane_addr + kColS + 32, x);
                    tc::tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; ++i) v[32 + i] = x[i];
                }
                const int32_t sg = j * kTileKeys + row;
                const bool key_ok = sg < ti.n_win || (sg >= ti.n_win4 && sg < ti.n_keys);
#pragma unroll
                for (int h = 0; h < 64; ++h) v[h] = key_ok ? v[h] * c : -INFINITY;
                // tile max per head -> lazily moved running max
                float m0, m1;
                reduce_scatter64<true>(v, m0, m1, lane);
                ms->red[q4][2 * lane] = m0;
                ms->red[q4][2 * lane + 1] = m1;
                const uint32_t rs = tile_ctr & 1;
                if (ltid == 0) ms->rescale[rs ^ 1] = 0;
                tc::named_bar_sync(1, 128);
                if (ltid < 64) {
                    const float mt = fmaxf(fmaxf(ms->red[0][ltid], ms->red[1][ltid]),
                                           fmaxf(ms->red[2][ltid], ms->red[3][ltid]));
                    const float mo = ms->m_run[ltid];
                    float al = 1.0f;
                    if (mt > mo + kLazyMax) {
                        al = (mo == -INFINITY) ? 0.0f : exp2f(mo - mt);
                        ms->m_run[ltid] = mt;
                        ms->rescale[rs] = 1;
                    }
                    ms->alpha[ltid] = al;
                }
                tc::named_bar_sync(1, 128);
                if (ms->rescale[rs]) {
#pragma unroll
                    for (int h = 0; h < 64; ++h) lp[h] *= ms->alpha[h];
                    if (j > 0) {
                        // O^T of the earlier tiles is complete (the commit that
                        // signalled this S^T covers it); scale its columns.
#pragma unroll 1
                        for (int s = 0; s < 4; ++s) {
#pragma unroll 1
                            for (int half = 0; half < 2; ++half) {
                                float x[32];
                                const uint32_t addr = lane_addr + kColO + 64 * s + 32 * half;
                                tc::tmem_ld32(addr, x);
                                tc::tmem_wait_ld();
#pragma unroll
                                for (int i = 0; i < 32; ++i) x[i] *= ms->alpha[32 * half + i];
                                tc::tmem_st32(addr, x);
                            }
                        }
                        tc::tmem_wait_st();
                    }
                }
                // probabilities; P^T row `row` (64 heads = 128 B, MN-major SW128)
                uint4 packed[8];
#pragma unroll
                for (int ch = 0; ch < 8; ++ch) {
                    uint32_t w4[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int h = 8 * ch + 2 * e;
                        const float mu0 = ms->m_run[h], mu1 = ms->m_run[h + 1];
                        const float p0 = (mu0 == -INFINITY) ? 0.0f : exp2f(v[h] - mu0);
                        const float p1 = (mu1 == -INFINITY) ? 0.0f : exp2f(v[h + 1] - mu1);
                        lp[h] += p0;
                        lp[h + 1] += p1;
                        __nv_bfloat162 pb = __floats2bfloat162_rn(p0, p1);
                        w4[e] = *reinterpret_cast<uint32_t *>(&pb);
                    }
                    packed[ch] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
                }
#pragma unroll
                for (int ch = 0; ch < 8; ++ch)
                    *reinterpret_cast<uint4 *>(pbuf + row * 128 + ((ch ^ (row & 7)) * 16)) =
                        packed[ch];
                tc::fence_proxy_async_smem();
                tc::tc_fence_before();
                tc::mbar_arrive(&ms->p_full);
            }
            if (stop) break;
            // ---- epilogue: row sums, LSE, then O^T / l -> out[t, h, d]
            {
                float s0, s1;
                reduce_scatter64<false>(lp, s0, s1, lane);
                ms->red[q4][2 * lane] = s0;
                ms->red[q4][2 * lane + 1] = s1;
                tc::named_bar_sync(1, 128);
                if (ltid < 64) {
                    float l = (ms->red[0][ltid] + ms->red[1][ltid]) +
                              (ms->red[2][ltid] + ms->red[3][ltid]);
                    const float mu = ms->m_run[ltid];
                    if (a.sinks && ltid < a.H) {
                        const float sk = __ldg(a.sinks + ltid) * kLog2e;
                        if (sk != -INFINITY) l += exp2f(sk - mu);
                    }
                    ms->inv_l[ltid] = l > 0.0f ? 1.0f / l : 0.0f;
                    if (a.lse && ltid < a.H) a.lse[(int64_t)t * a.H + ltid] = (mu + log2f(l)) * kLn2;
                }
                tc::named_bar_sync(1, 128);
            }
            ok = cx.wait(&ms->o_full, o_n & 1, 32);
            if (!bar_red_and(ok)) break;
            ++o_n;
            tc::tc_fence_after();
            __nv_bfloat16 *outp = a.out + (int64_t)t * a.H * 512;
#pragma unroll 1
            for (int s = 0; s < 4; ++s) {
                const int d = 128 * s + row;
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    float x[32];
                    tc::tmem_ld32(lane_addr + kColO + 64 * s + 32 * half, x);
                    tc::tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const int h = 32 * half + i;
                        if (h < a.H)
                            outp[(int64_t)h * 512 + d] = __float2bfloat16_rn(x[i] * ms->inv_l[h]);
                    }
                }
            }
            tc::tc_fence_before();
        }
    }
    // ------------------------------------------------------------- teardown
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    if (warp == 1) tc::tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

cudaError_t launch_sparse_mla_fwd(const MlaArgs &a, cudaStream_t stream) {
    if (a.T == 0) return cudaSuccess;
    if (a.cmp_idx && a.topk > kMaxList) return cudaErrorInvalidValue;
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    CUtensorMap q_map, ori_map, cmp_map;
    if (!encode_bf16_3d(&q_map, a.q, 512, a.H, a.T, 64, a.H, 1)) return cudaErrorInvalidValue;
    if (!encode_bf16_2d(&ori_map, a.ori_kv, a.T, 512, 64, 1)) return cudaErrorInvalidValue;
    if (a.cmp_kv && a.Tc > 0) {
        if (!encode_bf16_2d(&cmp_map, a.cmp_kv, a.Tc, 512, 64, 1)) return cudaErrorInvalidValue;
    } else {
        cmp_map = ori_map;  // never read
    }
    e = cudaFuncSetAttribute(sparse_mla_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    Params p{a, a.window};
    const int ctas = a.T < sms ? a.T : sms;
    sparse_mla_tc_kernel<<<ctas, kThreads, kSmemBytes, stream>>>(q_map, ori_map, cmp_map, p);
    return cudaGetLastError();
}

int32_t sparse_mla_max_topk() { return kMaxList; }

}  // namespace csa
