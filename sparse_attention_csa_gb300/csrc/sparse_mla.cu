// Shared-KV MLA sparse attention forward with attention sinks (sm_103a,
// tcgen05 tensor cores, TMA and cp.async).
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
//     K and V are the same rows: one 128-key x 512 tile in shared memory
//     (SW128, K-major) serves S^T as the A operand and, read MN-major, O^T as
//     the A operand. Accumulators live in tensor memory: S^T in 64 columns,
//     O^T in 4 x 64 columns.
//   * Key tiles. A token with at most 128 keys gets one tile: its window rows
//     then its compressed rows, gathered with 16-byte cp.async. Otherwise its
//     window rows (one contiguous run) fill tiles of their own, loaded by 2-D
//     TMA boxes of 128 rows, and its compressed rows follow in their own
//     tiles: by TMA boxes too when they form one ascending run (always in the
//     compressor-only mode, and in the indexer mode whenever top-k covers
//     every visible block) and at least half a tile long, else gathered by
//     cp.async. Rows of a box past the tile's valid count are masked. (TMA
//     gather4 moves single 128-byte rows an order of magnitude slower than
//     these paths.) Q arrives by 3-D TMA, after an L2 prefetch issued one token ahead.
//   * Warp roles: 0 scheduler (key lists, Q), 1-2 loaders (K/V tiles;
//     gathered slabs are released by cp.async-tracking mbarrier arrivals),
//     3 tensor memory + tcgen05.mma issue (one thread), 4-11 softmax and
//     epilogue in two warpgroups of 32 heads each (softmax: one thread per key
//     = one TMEM lane, 32 head scores; epilogue: one thread per d row of O^T,
//     so a warp's lanes hold 32 consecutive d of each head: 64-byte stores
//     with no data exchanged between lanes. Lane shuffles and cp.async traffic
//     both slow the tensor core's concurrent shared-memory reads, so the
//     kernel keeps them off the common path).
//   * Online softmax in base 2 with a lazily moved running max: a head's max
//     only moves when a tile exceeds it by more than 8 (a factor 256), so O^T
//     in tensor memory is rescaled rarely, and the cross-lane reduction of the
//     tile maxima runs only for tiles where some score exceeds a max by that
//     much (a warpgroup-wide vote decides). Row sums accumulate per thread in
//     fp32 and are reduced once per token.
//   * Every mbarrier wait is bounded; a timeout records CSA_ERR_TIMEOUT, the
//     CTA drains its copies and MMAs, frees tensor memory and exits.
#include "common.cuh"
#include "internal.h"
#include "tc_ptx.cuh"
#include "tmap.h"

namespace csa {

namespace {

constexpr int kThreads = 384;  // 12 warps
constexpr int kTileKeys = 128;
constexpr int kMaxList = 1024;  // compressed indices per token (topk bound)
constexpr int kLoaders = 64;    // threads of the two loader warps
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kLazyMax = 8.0f;  // base-2 units
constexpr int kMinBoxRows = 64;   // shorter compressed runs are gathered, not boxed
#ifndef CSA_MLA_CHUNK
#define CSA_MLA_CHUNK 1
#endif
constexpr int kChunk = CSA_MLA_CHUNK;  // consecutive tokens per CTA visit

// shared memory map (offsets from a 1024-byte aligned base)
constexpr uint32_t kOffKV = 0;            // 8 chunks x [128 keys x 128 B]
constexpr uint32_t kOffQ = 131072;        // 8 chunks x [64 heads x 128 B]
constexpr uint32_t kOffP = 196608;        // [128 keys x 64 heads] bf16, MN-major
constexpr uint32_t kOffList = 212992;     // 2 x kMaxList int32 (one per token slot)
constexpr uint32_t kOffMisc = kOffList + 2 * kMaxList * 4;

// tensor memory columns
constexpr uint32_t kColS = 0;
constexpr uint32_t kColO = 256;
constexpr uint32_t kTmemCols = 512;

enum : int32_t { kTileOri = 0, kTileCmp = 1, kTileGather = 2 };
enum : int32_t { kFlagMixed = 1, kFlagCmpRun = 2 };

struct TokenInfo {
    int32_t t, n_win, n_cmp, n_tiles;
    int32_t valid, win_start, cmp_first, flags;
};

struct TileDesc {
    int32_t kind;     // kTileOri / kTileCmp (TMA box of 128 rows from row0) or kTileGather
    int32_t row0;     // first row of the box
    int32_t n_valid;  // slots [0, n_valid) hold keys
    int32_t key0;     // key index (window rows first, then compressed) of slot 0
};

__device__ __forceinline__ TileDesc tile_desc(const TokenInfo &ti, int32_t j) {
    if (ti.flags & kFlagMixed) return {kTileGather, 0, ti.n_win + ti.n_cmp, 0};
    const int32_t nwt = (ti.n_win + kTileKeys - 1) / kTileKeys;
    if (j < nwt)
        return {kTileOri, ti.win_start + j * kTileKeys, min(kTileKeys, ti.n_win - j * kTileKeys),
                j * kTileKeys};
    const int32_t jc = j - nwt;
    const int32_t n = min(kTileKeys, ti.n_cmp - jc * kTileKeys);
    if ((ti.flags & kFlagCmpRun) && n >= kMinBoxRows)
        return {kTileCmp, ti.cmp_first + jc * kTileKeys, n, ti.n_win + jc * kTileKeys};
    return {kTileGather, 0, n, ti.n_win + jc * kTileKeys};
}

// The it-th token of this CTA: runs of kChunk consecutive tokens, run r of
// the grid going to CTA r mod gridDim.x. Increasing in `it`.
__device__ __forceinline__ int32_t token_at(uint32_t it) {
    const int64_t run = (int64_t)(it / kChunk) * gridDim.x + blockIdx.x;
    const int64_t t = run * kChunk + it % kChunk;
    return t < INT32_MAX ? (int32_t)t : INT32_MAX;
}

struct Misc {
    uint64_t q_full[4], q_empty[4];   // per pair of 64-wide chunks of Q
    uint64_t kv_full[4], kv_empty[4]; // per slab (pair of chunks) of the K/V tile
    uint64_t s_full, p_full, o_full, drain;
    uint64_t info_full[2], info_empty[2];
    uint32_t tmem_base;
    int32_t abort;
    TokenInfo info[2];
    __align__(16) float red[2][4][64];   // [tile parity][lane quarter][head]
    __align__(16) float sink2[64];       // sink * log2(e), -inf when absent
};

constexpr size_t kSmemBytes = kOffMisc + sizeof(Misc) + 1024;
static_assert(kSmemBytes <= 232448, "shared memory budget");

// AND of v over the 128 threads of named barrier `id`.
__device__ __forceinline__ bool bar_red_and(uint32_t id, bool v) {
    uint32_t out;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.and.pred q, %2, 128, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(out)
        : "r"((uint32_t)v), "r"(id)
        : "memory");
    return out != 0;
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
// The mbarrier counts one arrival (already included in its expected count)
// once every cp.async this thread issued so far has landed.
__device__ __forceinline__ void cp_async_arrive(uint64_t *bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(tc::smem_u32(bar))
                 : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.wait_all;" ::: "memory");
}

// OR of v over the 128 threads of named barrier `id`.
__device__ __forceinline__ bool bar_red_or(uint32_t id, bool v) {
    uint32_t out;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, %2, 128, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(out)
        : "r"((uint32_t)v), "r"(id)
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

// 32 values per thread -> lane L holds the warp-wide reduction of value L.
template <bool kMax>
__device__ __forceinline__ float reduce_scatter32(const float (&x)[32], int lane) {
    auto op = [](float a, float b) { return kMax ? fmaxf(a, b) : a + b; };
    float b[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const bool hi = lane & 16;
        const float send = hi ? x[i] : x[16 + i];
        const float keep = hi ? x[16 + i] : x[i];
        b[i] = op(keep, __shfl_xor_sync(0xffffffffu, send, 16));
    }
    float c[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const bool hi = lane & 8;
        const float send = hi ? b[i] : b[8 + i];
        const float keep = hi ? b[8 + i] : b[i];
        c[i] = op(keep, __shfl_xor_sync(0xffffffffu, send, 8));
    }
    float d[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const bool hi = lane & 4;
        const float send = hi ? c[i] : c[4 + i];
        const float keep = hi ? c[4 + i] : c[i];
        d[i] = op(keep, __shfl_xor_sync(0xffffffffu, send, 4));
    }
    float e[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const bool hi = lane & 2;
        const float send = hi ? d[i] : d[2 + i];
        const float keep = hi ? d[2 + i] : d[i];
        e[i] = op(keep, __shfl_xor_sync(0xffffffffu, send, 2));
    }
    const bool hi = lane & 1;
    return op(hi ? e[1] : e[0], __shfl_xor_sync(0xffffffffu, hi ? e[0] : e[1], 1));
}

__global__ void __launch_bounds__(kThreads, 1)
sparse_mla_tc_kernel(const __grid_constant__ CUtensorMap q_map,
                     const __grid_constant__ CUtensorMap ori_map,
                     const __grid_constant__ CUtensorMap cmp_map,
                     const __grid_constant__ MlaArgs a) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem =
        reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                          ~uintptr_t(1023));
    Misc *ms = reinterpret_cast<Misc *>(smem + kOffMisc);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    Ctx cx{ms, a.err};

    // ---------------------------------------------------------------- set-up
    if (tid == 0) {
        for (int s = 0; s < 4; ++s) {
            tc::mbar_init(&ms->q_full[s], 1);
            tc::mbar_init(&ms->q_empty[s], 1);
            tc::mbar_init(&ms->kv_full[s], kLoaders);
            tc::mbar_init(&ms->kv_empty[s], 1);
        }
        tc::mbar_init(&ms->s_full, 1);
        tc::mbar_init(&ms->p_full, 256);
        tc::mbar_init(&ms->o_full, 1);
        tc::mbar_init(&ms->drain, 1);
        for (int i = 0; i < 2; ++i) {
            tc::mbar_init(&ms->info_full[i], 1);
            tc::mbar_init(&ms->info_empty[i], 11);  // MMA + 8 softmax + 2 loader warps
        }
        ms->abort = 0;
        tc::fence_mbar_init();
    }
    if (tid < 64)
        ms->sink2[tid] = (a.sinks && tid < a.H) ? __ldg(a.sinks + tid) * kLog2e : -INFINITY;
    // Rows never written by a copy must hold finite values: zero Q and KV once.
    for (uint32_t i = tid; i < (kOffP - kOffKV) / 16; i += kThreads)
        reinterpret_cast<uint4 *>(smem + kOffKV)[i] = make_uint4(0, 0, 0, 0);
    tc::fence_proxy_async_smem();
    if (warp == 3) {
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
        // ================================================== scheduler warp
        uint32_t it = 0, q_n = 0;
        int32_t seg_lo = 0, seg_hi = 0, seg_b = -1;  // last sequence found: [lo, hi)
        for (int32_t t = token_at(it); t < a.T; t = token_at(++it)) {
            const uint32_t slot = it & 1;
            // the slot's key list is rewritten only once every consumer is done
            bool ok = cx.wait(&ms->info_empty[slot], ((it >> 1) & 1) ^ 1, 10);
            if (!__all_sync(0xffffffffu, ok)) break;
            int32_t *list = reinterpret_cast<int32_t *>(smem + kOffList) + slot * kMaxList;
            TokenInfo ti{t, 0, 0, 0, 0, 0, 0, 0};
            // tokens of a CTA increase, so the last sequence usually still holds t
            if (seg_b < 0 || t < seg_lo || t >= seg_hi) {
                seg_b = find_segment(a.cu_q, a.batch, t);
                if (seg_b >= 0) {
                    seg_lo = __ldg(a.cu_q + seg_b);
                    seg_hi = __ldg(a.cu_q + seg_b + 1);
                }
            }
            const int32_t b = seg_b;
            if (b < 0) {
                if (lane == 0) report_error(a.err, kErrCheck, kKerMla, 1);
            } else {
                const int32_t seg0 = max(seg_lo, 0);
                const int32_t pos = t - seg0;
                ti.win_start = max(t - a.window + 1, seg0);
                ti.n_win = t - ti.win_start + 1;
                int32_t n_cmp = 0;
                bool run = true;
                if (use_cmp) {
                    const int32_t cbase = __ldg(a.cu_c + b);
                    const int32_t seg_blocks = __ldg(a.cu_c + b + 1) - cbase;
                    int32_t vis = min((pos + 1) / a.cmp_ratio, seg_blocks);
                    if (cbase < 0 || vis < 0 || (int64_t)cbase + vis > a.Tc) {
                        if (lane == 0) report_error(a.err, kErrCheck, kKerMla, 2);
                        vis = 0;
                    }
                    if (a.cmp_idx) {
                        // Compact the valid entries, in entry order. Each round
                        // issues all 16 loads of 512 entries before using any.
                        const int32_t *row = a.cmp_idx + (int64_t)t * a.topk;
                        for (int32_t e0 = 0; e0 < a.topk; e0 += 512) {
                            int32_t jv[16];
#pragma unroll
                            for (int r = 0; r < 16; ++r) {
                                const int32_t e = e0 + 32 * r + lane;
                                jv[r] = e < a.topk ? __ldg(row + e) : -1;
                            }
#pragma unroll
                            for (int r = 0; r < 16; ++r) {
                                const bool v = jv[r] >= cbase && jv[r] < cbase + vis;
                                const uint32_t m = __ballot_sync(0xffffffffu, v);
                                if (v) list[n_cmp + __popc(m & ((1u << lane) - 1u))] = jv[r];
                                n_cmp += __popc(m);
                            }
                        }
                        __syncwarp();
                        // one ascending run of consecutive rows?
                        if (n_cmp > 0) {
                            const int32_t first = list[0];
                            bool mine = true;
                            for (int32_t e = lane; e < n_cmp; e += 32) mine &= list[e] == first + e;
                            run = __all_sync(0xffffffffu, mine);
                            ti.cmp_first = first;
                        }
                    } else {
                        n_cmp = vis;
                        ti.cmp_first = cbase;
                    }
                }
                ti.n_cmp = n_cmp;
                const int32_t n_keys = ti.n_win + n_cmp;
                if (n_keys <= kTileKeys) {
                    ti.flags = kFlagMixed;
                    ti.n_tiles = 1;
                } else {
                    ti.flags = run ? kFlagCmpRun : 0;
                    ti.n_tiles = (ti.n_win + kTileKeys - 1) / kTileKeys +
                                 (n_cmp + kTileKeys - 1) / kTileKeys;
                }
                ti.valid = 1;
            }
            __syncwarp();  // list writes before the release below
            if (lane == 0) {
                ms->info[slot] = ti;
                tc::mbar_arrive(&ms->info_full[slot]);
                // Q of this CTA's next token streams from HBM into L2 while
                // this token runs; its TMA load then hits L2.
                const int32_t tn = token_at(it + 1);
                if (tn < a.T) tc::prefetch_l2_bulk(a.q + (int64_t)tn * a.H * 512, (uint32_t)a.H * 1024u);
            }
            if (!ti.valid) continue;
            // Q rows of token t (H rows of 512; rows >= H stay zero), one pair
            // of 64-wide chunks at a time as the previous token frees them
            bool qbroke = false;
            for (int pr = 0; pr < 4; ++pr) {
                ok = cx.wait(&ms->q_empty[pr], (q_n & 1) ^ 1, 11);
                if (!__all_sync(0xffffffffu, ok)) {
                    qbroke = true;
                    break;
                }
                if (lane == 0) {
                    tc::mbar_expect_tx(&ms->q_full[pr], 2u * a.H * 128u);
                    for (int cc = 0; cc < 2; ++cc) {
                        const int c = 2 * pr + cc;
                        tc::tma_load_3d(smem + kOffQ + c * 8192, &q_map, &ms->q_full[pr], 64 * c, 0,
                                        t);
                    }
                }
            }
            if (qbroke) break;
            ++q_n;
        }
        if (lane == 0 && q_n > 0)  // drain: every Q copy issued has landed
            for (int pr = 0; pr < 4; ++pr)
                if (!tc::mbar_wait(&ms->q_full[pr], (q_n - 1) & 1)) cx.fail(13);
    } else if (warp == 1 || warp == 2) {
        // ==================================================== loader warps
        // Gathered tiles: thread i covers, for slab s, the 16-byte column
        // 16 s + (i & 15) of the slots k = (i >> 4) + 4 m (m < 32): one
        // 256-byte row piece per quarter-warp, so every global access is a
        // coalesced run. Row addresses are computed once per tile.
        const int li = tid - 32;  // 0..63
        const int col = li & 15, sgrp = li >> 4;
        uint32_t it = 0, kv_n = 0;
        const uint32_t kv_base = tc::smem_u32(smem + kOffKV);
        bool stop = false;
        for (int32_t t = token_at(it); t < a.T && !stop; t = token_at(++it)) {
            const uint32_t slot = it & 1;
            if (!cx.wait(&ms->info_full[slot], (it >> 1) & 1, 40)) break;
            const TokenInfo ti = ms->info[slot];
            const int32_t *list = reinterpret_cast<const int32_t *>(smem + kOffList) + slot * kMaxList;
            for (int32_t j = 0; j < ti.n_tiles && !stop; ++j, ++kv_n) {
                const TileDesc td = tile_desc(ti, j);
                if (td.kind != kTileGather) {
                    const CUtensorMap *map = td.kind == kTileOri ? &ori_map : &cmp_map;
                    for (int s = 0; s < 4; ++s) {
                        if (!cx.wait(&ms->kv_empty[s], (kv_n & 1) ^ 1, 41)) {
                            stop = true;
                            break;
                        }
                        if (li == 0) {
                            tc::mbar_expect_tx(&ms->kv_full[s], 32768u);
                            for (int cc = 0; cc < 2; ++cc) {
                                const int c = 2 * s + cc;
                                tc::tma_load_2d(smem + kOffKV + c * 16384, map, &ms->kv_full[s],
                                                64 * c, td.row0);
                            }
                        } else {
                            tc::mbar_arrive(&ms->kv_full[s]);
                        }
                    }
                    continue;
                }
                // gathered tile: this thread's 32 slots
                const __nv_bfloat16 *src[32];
#pragma unroll
                for (int m = 0; m < 32; ++m) {
                    const int k = sgrp + 4 * m;
                    const int32_t e = td.key0 + k;
                    const __nv_bfloat16 *p = nullptr;
                    if (k < td.n_valid) {
                        if (e < ti.n_win) {
                            p = a.ori_kv + (int64_t)(ti.win_start + e) * 512;
                        } else {
                            const int32_t ce = e - ti.n_win;
                            p = a.cmp_kv + (int64_t)(a.cmp_idx ? list[ce] : ti.cmp_first + ce) * 512;
                        }
                    }
                    src[m] = p;
                }
                // Each slab is released to the tensor core by the mbarrier
                // itself once this thread's copies land; the thread goes on to
                // the next slab without waiting.
                for (int s = 0; s < 4; ++s) {
                    if (!cx.wait(&ms->kv_empty[s], (kv_n & 1) ^ 1, 42)) {
                        stop = true;
                        break;
                    }
                    const int c16 = 16 * s + col;             // 16-byte column in the row
                    const int chunk = c16 >> 3, w = c16 & 7;  // 128-byte chunk, piece
#pragma unroll
                    for (int m = 0; m < 32; ++m) {
                        const int k = sgrp + 4 * m;
                        if (src[m])
                            cp_async16(kv_base + chunk * 16384 + k * 128 + ((w ^ (k & 7)) << 4),
                                       src[m] + c16 * 8);
                    }
                    cp_async_arrive(&ms->kv_full[s]);
                }
            }
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&ms->info_empty[slot]);
        }
        cp_async_wait_all();  // drain: no copy outlives the CTA
        if (li == 0 && kv_n > 0)  // and no TMA copy either (last tile's phases)
            for (int s = 0; s < 4; ++s)
                if (!tc::mbar_wait(&ms->kv_full[s], (kv_n - 1) & 1)) cx.fail(43);
    } else if (warp == 3) {
        // ========================================================= MMA warp
        if (lane == 0) {
            const uint32_t id_s = tc::idesc_bf16(128, 64, false, false);
            const uint32_t id_o = tc::idesc_bf16(128, 64, true, true);
            // Descriptors of the four operand bases, built once; each MMA adds
            // a constant byte offset (k-step, chunk, slab) to the address field.
            const uint64_t ds_a = tc::smem_desc(tc::smem_u32(smem + kOffKV), 16, 1024);
            const uint64_t ds_b = tc::smem_desc(tc::smem_u32(smem + kOffQ), 16, 1024);
            const uint64_t do_a = tc::smem_desc(tc::smem_u32(smem + kOffKV), 16384, 1024);
            const uint64_t do_b = tc::smem_desc(tc::smem_u32(smem + kOffP), 16384, 1024);
            uint32_t it = 0, q_n = 0, kv_n = 0, p_n = 0;
            bool issued = false;
            for (int32_t t = token_at(it); t < a.T; t = token_at(++it)) {
                const uint32_t slot = it & 1;
                if (!cx.wait(&ms->info_full[slot], (it >> 1) & 1, 20)) break;
                const TokenInfo ti = ms->info[slot];
                tc::mbar_arrive(&ms->info_empty[slot]);
                if (!ti.valid) continue;
                bool stop = false;
                for (int32_t j = 0; j < ti.n_tiles && !stop; ++j, ++kv_n) {
                    for (int s = 0; s < 4; ++s) {
                        if ((j == 0 && !cx.wait(&ms->q_full[s], q_n & 1, 21)) ||
                            !cx.wait(&ms->kv_full[s], kv_n & 1, 22)) {
                            stop = true;
                            break;
                        }
                        // slabs gathered by cp.async were written through the
                        // generic proxy: order them before the tensor core's reads
                        tc::fence_proxy_async_smem();
                        tc::tc_fence_after();
#pragma unroll
                        for (int cc = 0; cc < 2; ++cc) {
                            const int c = 2 * s + cc;
#pragma unroll
                            for (int kk = 0; kk < 4; ++kk)
                                tc::mma_bf16(tmem + kColS, tc::desc_add(ds_a, c * 16384 + kk * 32),
                                             tc::desc_add(ds_b, c * 8192 + kk * 32), id_s,
                                             (c | kk) != 0);
                        }
                        issued = true;
                        // the last tile's S^T frees this pair of Q chunks
                        if (j == ti.n_tiles - 1) tc::mma_commit(&ms->q_empty[s]);
                    }
                    if (stop) break;
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
                                         tc::desc_add(do_a, 2 * s * 16384 + kk * 2048),
                                         tc::desc_add(do_b, kk * 2048), id_o, (j > 0 || kk > 0));
                        tc::mma_commit(&ms->kv_empty[s]);
                    }
                }
                if (stop) break;
                ++q_n;
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
        // Two warpgroups: wg 0 owns heads 0-31, wg 1 heads 32-63. Warp
        // (4 + 4 wg + q) reads TMEM lane quarter q: one key slot per thread in
        // the softmax, one d row of O^T per thread in the epilogue.
        const int wg = (warp - 4) >> 2;
        const int q4 = warp & 3;
        const int row = 32 * q4 + lane;
        const uint32_t bar_id = 1 + wg;
        const int h0 = 32 * wg;                 // first head of this warpgroup
        const uint32_t lane_addr = tmem + ((uint32_t)(32 * q4) << 16);
        unsigned char *pbuf = smem + kOffP;
        const float c = a.softmax_scale * kLog2e;
        uint32_t it = 0, s_n = 0, o_n = 0, tile_ctr = 0;
        for (int32_t t = token_at(it); t < a.T; t = token_at(++it)) {
            const uint32_t slot = it & 1;
            bool ok = cx.wait(&ms->info_full[slot], (it >> 1) & 1, 30);
            if (!bar_red_and(bar_id, ok)) break;
            const TokenInfo ti = ms->info[slot];
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&ms->info_empty[slot]);
            if (!ti.valid) continue;
            // Per-head scalars live one head per lane (head h0 + lane):
            // m_lane the running max (base 2); m_cur[] is every thread's copy
            // of all 32, refreshed by shuffles only when some max moves.
            float m_lane = ms->sink2[h0 + lane];
            float lp[32], m_cur[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) lp[i] = 0.0f;
#pragma unroll
            for (int i = 0; i < 32; ++i) m_cur[i] = __shfl_sync(0xffffffffu, m_lane, i);
            bool stop = false;
            for (int32_t j = 0; j < ti.n_tiles; ++j, ++tile_ctr) {
                ok = cx.wait(&ms->s_full, s_n & 1, 31);
                if (!bar_red_and(bar_id, ok)) {
                    stop = true;
                    break;
                }
                ++s_n;
                tc::tc_fence_after();
                float v[32];
                tc::tmem_ld32(lane_addr + kColS + h0, v);
                tc::tmem_wait_ld();
                const bool key_ok = row < tile_desc(ti, j).n_valid;
#pragma unroll
                for (int i = 0; i < 32; ++i) v[i] = key_ok ? v[i] * c : -INFINITY;
                // A head's max moves only when some score of this tile exceeds
                // it by more than kLazyMax; the warpgroup first checks whether
                // any does, and only then reduces the tile maxima.
                bool exceeds = false;
#pragma unroll
                for (int i = 0; i < 32; ++i) exceeds |= v[i] > m_cur[i] + kLazyMax;
                if (bar_red_or(bar_id, exceeds)) {
                    // tile max per head: warp maxima (one head per lane) across the
                    // four lane quarters; every warp derives the same lazy update
                    const uint32_t rs = tile_ctr & 1;
                    ms->red[rs][q4][h0 + lane] = reduce_scatter32<true>(v, lane);
                    tc::named_bar_sync(bar_id, 128);
                    const float mt =
                        fmaxf(fmaxf(ms->red[rs][0][h0 + lane], ms->red[rs][1][h0 + lane]),
                              fmaxf(ms->red[rs][2][h0 + lane], ms->red[rs][3][h0 + lane]));
                    const bool up = mt > m_lane + kLazyMax;
                    const float al_lane =
                        up ? (m_lane == -INFINITY ? 0.0f : tc::ex2_approx(m_lane - mt)) : 1.0f;
                    if (up) m_lane = mt;
                    if (__any_sync(0xffffffffu, up)) {  // uniform across the warpgroup
#pragma unroll
                        for (int i = 0; i < 32; ++i) {
                            m_cur[i] = __shfl_sync(0xffffffffu, m_lane, i);
                            lp[i] *= __shfl_sync(0xffffffffu, al_lane, i);
                        }
                        if (j > 0) {
                            // O^T of the earlier tiles is complete (the commit that
                            // signalled this S^T covers it); scale this half's columns.
#pragma unroll 1
                            for (int sl = 0; sl < 4; ++sl) {
                                float x[32];
                                const uint32_t addr = lane_addr + kColO + 64 * sl + h0;
                                tc::tmem_ld32(addr, x);
                                tc::tmem_wait_ld();
#pragma unroll
                                for (int i = 0; i < 32; ++i)
                                    x[i] *= __shfl_sync(0xffffffffu, al_lane, i);
                                tc::tmem_st32(addr, x);
                            }
                            tc::tmem_wait_st();
                        }
                    }
                }
                // Probabilities -> P^T row `row`, heads h0..h0+31 (64 B of the
                // 128-byte MN-major SW128 row: 16-byte chunks 4 wg .. 4 wg + 3).
                // m_cur is finite here: every tile holds a valid key, so the
                // first tile always lifts an absent (-inf) sink.
#pragma unroll
                for (int cq = 0; cq < 4; ++cq) {
                    uint32_t w4[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int i = 8 * cq + 2 * e;
                        const float p0 = tc::ex2_approx(v[i] - m_cur[i]);
                        const float p1 = tc::ex2_approx(v[i + 1] - m_cur[i + 1]);
                        lp[i] += p0;
                        lp[i + 1] += p1;
                        __nv_bfloat162 pb = __floats2bfloat162_rn(p0, p1);
                        w4[e] = *reinterpret_cast<uint32_t *>(&pb);
                    }
                    const int ch = 4 * wg + cq;
                    *reinterpret_cast<uint4 *>(pbuf + row * 128 + ((ch ^ (row & 7)) * 16)) =
                        make_uint4(w4[0], w4[1], w4[2], w4[3]);
                }
                tc::fence_proxy_async_smem();
                tc::tc_fence_before();
                tc::mbar_arrive(&ms->p_full);
            }
            if (stop) break;
            // ---- epilogue: row sums and LSE (one head per lane), then O^T / l
            const uint32_t rs = tile_ctr & 1;  // a parity no softmax step of this token still reads
            ms->red[rs][q4][h0 + lane] = reduce_scatter32<false>(lp, lane);
            tc::named_bar_sync(bar_id, 128);
            float l_lane = (ms->red[rs][0][h0 + lane] + ms->red[rs][1][h0 + lane]) +
                           (ms->red[rs][2][h0 + lane] + ms->red[rs][3][h0 + lane]);
            const float sk = ms->sink2[h0 + lane];
            if (sk != -INFINITY) l_lane += tc::ex2_approx(sk - m_lane);
            const float il_lane = l_lane > 0.0f ? tc::rcp_approx(l_lane) : 0.0f;
            if (q4 == 0 && a.lse && h0 + lane < a.H)
                a.lse[(int64_t)t * a.H + h0 + lane] = (m_lane + tc::lg2_approx(l_lane)) * kLn2;
            float il[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) il[i] = __shfl_sync(0xffffffffu, il_lane, i);
            ok = cx.wait(&ms->o_full, o_n & 1, 32);
            if (!bar_red_and(bar_id, ok)) break;
            ++o_n;
            tc::tc_fence_after();
            // O^T slab sl: this thread holds d = 128 sl + row for the 32 heads
            // of its half, and the warp's 32 lanes hold 32 consecutive d: for
            // each head the warp writes one contiguous 64-byte piece of the
            // head's output row. No data moves between lanes.
            const int n_h = min(32, a.H - h0);  // heads of this half that exist
            __nv_bfloat16 *outp = a.out + (int64_t)t * a.H * 512 + (int64_t)h0 * 512 + row;
#pragma unroll 1
            for (int sl = 0; sl < 4 && n_h > 0; ++sl) {
                float x[32];
                tc::tmem_ld32(lane_addr + kColO + 64 * sl + h0, x);
                tc::tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    if (i < n_h) outp[(int64_t)i * 512 + 128 * sl] = __float2bfloat16_rn(x[i] * il[i]);
            }
            tc::tc_fence_before();
        }
    }
    // ------------------------------------------------------------- teardown
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    if (warp == 3) tc::tmem_dealloc(tmem, kTmemCols);
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
    if (!encode_bf16_2d(&ori_map, a.ori_kv, a.T, 512, 64, kTileKeys)) return cudaErrorInvalidValue;
    if (a.cmp_kv && a.Tc > 0) {
        if (!encode_bf16_2d(&cmp_map, a.cmp_kv, a.Tc, 512, 64, kTileKeys))
            return cudaErrorInvalidValue;
    } else {
        cmp_map = ori_map;  // never read: no compressed tile exists
    }
    e = cudaFuncSetAttribute(sparse_mla_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    const int64_t runs = ((int64_t)a.T + kChunk - 1) / kChunk;
    const int ctas = runs < sms ? (int)runs : sms;
    sparse_mla_tc_kernel<<<ctas, kThreads, kSmemBytes, stream>>>(q_map, ori_map, cmp_map, a);
    return cudaGetLastError();
}

int32_t sparse_mla_max_topk() { return kMaxList; }

}  // namespace csa
