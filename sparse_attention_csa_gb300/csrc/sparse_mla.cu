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
// Design (persistent grid, 1 CTA per SM, one token at a time per CTA):
//   * All H (<= 64, padded to 64) heads of a token share its key rows, so the
//     contraction is done transposed, with the keys on the MMA's M side:
//         S^T[key, h]  = K[key, :] . Q[h, :]        M=128 keys, N=64, K=512
//         O^T[d, h]   += V[key, d]^T P[key, h]      M=128 d (x4), N=64, K=128
//     K and V are the same rows: one 128-key x 512 tile in shared memory
//     (SW128, K-major) serves S^T as the A operand and, read MN-major, O^T as
//     the A operand. Accumulators live in tensor memory: S^T in 64 columns,
//     O^T in 4 x 64 columns.
//   * Work split. CTAs claim runs of consecutive tokens from a per-launch
//     counter (guided self-scheduling: each run is a quarter of an even share
//     of the tokens left, 2 to 256), so consecutive tokens of a sequence
//     mostly follow each other in one CTA, and every CTA finishes at about the
//     same time whatever the per-token cost or the speed of its SM.
//   * Key tiles (kinds below) have slot layouts fixed by the token alone, and
//     a token at an even position runs its tiles in the natural order (window
//     first), one at an odd position in reverse. The last tile of a token is
//     then the first tile of the next one, which takes it over with at most
//     its own row and a newly visible block loaded (cp.async): the window as
//     a ring of 128 slots, compressed runs as 128-row boxes that already hold
//     the later blocks. Whole tiles come by 2-D TMA boxes (window rings,
//     contiguous compressed runs) or 16-byte cp.async gathers (top-k lists,
//     short mixed key sets); rows of a box past the token's keys are masked.
//     Results do not depend on the split: every layout and order is a
//     function of the token. Q arrives by 3-D TMA after an L2 prefetch issued
//     one token ahead.
//   * Warp roles: 0 scheduler (key lists, tile plans, Q), 1-2 loaders (K/V
//     tiles; gathered rows are released by cp.async-tracking mbarrier
//     arrivals), 3 tensor memory + tcgen05.mma issue (one thread; it waits on
//     one barrier per tile and issues the 32 S^T MMAs back to back), 4-11
//     softmax and epilogue in two warpgroups of 32 heads each (softmax: one
//     thread per key = one TMEM lane, 32 head scores; epilogue: one thread per
//     d row of O^T, so a warp's lanes hold 32 consecutive d of each head:
//     64-byte stores with no data exchanged between lanes).
//   * Online softmax in base 2. The max starts as the exact maximum of the
//     sink and the first tile (so the largest probability is exactly 1 in
//     bf16, which keeps short key sets within the output bound); after that
//     it moves lazily: only when a tile exceeds it by more than 8 (a factor
//     256), so O^T in tensor memory is rescaled rarely, and the cross-lane
//     reduction of the tile maxima runs only for tiles where some score
//     exceeds a max by that much (a warpgroup-wide vote decides). Row sums
//     accumulate per thread in fp32 and are reduced once per token.
//   * Every mbarrier wait is bounded; a timeout records CSA_ERR_TIMEOUT, the
//     CTA drains its copies and MMAs, frees tensor memory and exits.
#include "common.cuh"
#include "internal.h"
#include "tc_ptx.cuh"
#include "tmap.h"

#include <atomic>
#include <cstdint>

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

// Tile kinds. Every kind has a fixed slot layout that depends only on the
// token (never on which CTA runs it or what it ran before), so a tile left in
// shared memory by one token can be taken over by the next token of the same
// sequence with at most a row or two loaded, and results stay bit-identical
// however the tokens are split between CTAs.
//   kRing   window rows of ori_kv in a ring: row r in slot (r - b0) mod 128,
//           b0 a base fixed by the token's position; optionally the first
//           n_top compressed rows of the sequence in the top slots
//           (compressed row j in slot 127 - j) when they fit beside the window.
//           Loaded as one 128-row TMA box from b0 (rows past the token are
//           future window rows, masked), or gathered when top rows are present.
//   kWinBox window rows win_start + 128 j + slot (windows wider than 128).
//   kCmpBox compressed rows c0 + slot of one ascending run (TMA box).
//   kGather compressed entries e0 + slot of the token's index list (cp.async).
//   kGMix   window rows then compressed entries, gathered (short key sets
//           whose window already slides, or whose compressed set is a top-k).
enum : int32_t { kRing = 0, kWinBox = 1, kCmpBox = 2, kGather = 3, kGMix = 4 };
enum : int32_t { kFlagRun = 1, kFlagAllVis = 2 };

struct TokenInfo {
    int32_t t, valid, pos, seg;          // token, position in its sequence, sequence
    int32_t win_start, n_win, cbase, n_cmp;  // window; first compressed row of the
                                             // sequence; valid compressed keys
    int32_t cmp_first, flags, b0, n_top;     // first compressed row (runs); ring base
    int32_t n_wt, n_ct, n_tiles, single;     // window / compressed / all tiles; single-tile kind or -1
    int32_t reuse, n_delta;                  // first tile taken over from the previous token
    int32_t end;                             // no token: the CTA's stream ends here
    int32_t d_row[2], d_slot[2], d_cmp[2];   // rows loaded into it (d_cmp: from cmp_kv)
};

struct TileDesc {
    int32_t kind;
    int32_t row0;     // kRing: b0; kWinBox / kCmpBox: first row of the box
    int32_t n_valid;  // kRing: n_top; others: slots [0, n_valid) hold keys
    int32_t e0;       // kGather: first list entry
};

// Natural tile order: window tile(s), then compressed tiles. Tokens at even
// positions run it forwards and tokens at odd positions backwards, so the
// last tile of one token is the first tile of the next one.
__device__ __forceinline__ int32_t tile_nat(const TokenInfo &ti, int32_t j) {
    return (ti.pos & 1) ? ti.n_tiles - 1 - j : j;
}

__device__ __forceinline__ TileDesc tile_at(const TokenInfo &ti, int32_t nat) {
    if (ti.single == kRing) return {kRing, ti.b0, ti.n_top, 0};
    if (ti.single == kGMix) return {kGMix, 0, ti.n_win + ti.n_cmp, 0};
    if (nat < ti.n_wt) {
        if (ti.n_wt == 1 && ti.b0 >= 0) return {kRing, ti.b0, 0, 0};
        return {kWinBox, ti.win_start + nat * kTileKeys,
                min(kTileKeys, ti.n_win - nat * kTileKeys), 0};
    }
    const int32_t k = nat - ti.n_wt;
    const int32_t n = min(kTileKeys, ti.n_cmp - k * kTileKeys);
    if ((ti.flags & kFlagRun) && ((ti.flags & kFlagAllVis) || n >= kMinBoxRows))
        return {kCmpBox, ti.cmp_first + k * kTileKeys, n, 0};
    return {kGather, 0, n, k * kTileKeys};
}

// A ring tile is loaded whole as one TMA box from its base when it has no
// compressed rows on top and the token's own row falls inside the box (a
// token at an even position whose window already slides needs one row past
// it, so its ring is gathered instead).
__device__ __forceinline__ bool ring_box(const TokenInfo &ti, const TileDesc &td) {
    return td.kind == kRing && td.n_valid == 0 && ti.t <= td.row0 + kTileKeys - 1;
}

// Does slot `s` of tile `td` hold one of token ti's keys?
__device__ __forceinline__ bool slot_valid(const TokenInfo &ti, const TileDesc &td, int32_t s) {
    if (td.kind != kRing) return s < td.n_valid;
    if (s >= kTileKeys - td.n_valid) return true;  // compressed rows on top
    const int32_t r = ti.t - ((ti.t - td.row0 - s) & (kTileKeys - 1));
    return r >= ti.win_start;
}

// ------------------------------------------------------------ token claims
// CTAs take runs of consecutive tokens from the claim word of the launch's
// slot (dynamic, guided self-scheduling: a run is a share of what is left, so
// runs shrink towards the end of the launch and every CTA finishes at about
// the same time whatever the per-token cost). The high half of a word holds
// the epoch of the launch using it and the low half the tokens claimed so far.
// The last CTA to finish resets the word, so a launch replayed with the same
// epoch (a captured graph) starts afresh; a word left behind by a launch that
// gave up is recognised by its older epoch. Launches in flight at the same
// time take different slots (one per launch, cycling through kClaimSlots); a
// claim that finds another launch's epoch in the word reports it.
constexpr int kClaimSlots = 1024;
__device__ unsigned long long g_claim[kClaimSlots];
__device__ unsigned int g_claim_done[kClaimSlots];

// First token of a run of n claimed by this launch (>= T once all are taken;
// INT64_MAX when the word belongs to another launch).
__device__ int64_t claim_run(unsigned long long *w, uint32_t epoch, uint32_t n) {
    const unsigned long long mine = ((unsigned long long)epoch << 32) | n;
    unsigned long long v = atomicAdd(w, (unsigned long long)n);
    if ((uint32_t)(v >> 32) == epoch) return (int64_t)(uint32_t)v;
    // The word is not this launch's yet: install this launch's epoch with this
    // run as its first claim, unless another CTA of the launch already did.
    unsigned long long cur = v + n;
    for (int tries = 0; tries < 4096; ++tries) {
        const unsigned long long prev = atomicCAS(w, cur, mine);
        if (prev == cur) return 0;
        if ((uint32_t)(prev >> 32) == epoch) {
            v = atomicAdd(w, (unsigned long long)n);
            if ((uint32_t)(v >> 32) != epoch) break;
            return (int64_t)(uint32_t)v;
        }
        cur = prev;
    }
    return INT64_MAX;
}

struct Misc {
    uint64_t q_full, q_empty;         // Q of the token
    uint64_t kv_full, kv_empty[4];    // K/V tile landed; released per slab (pair of chunks)
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
    uint64_t limit;  // pipeline waits give up after this long
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
        if (tc::mbar_wait(bar, parity, limit)) return true;
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
    Ctx cx{ms, a.err, a.wait_ns};

    // ---------------------------------------------------------------- set-up
    if (tid == 0) {
        tc::mbar_init(&ms->q_full, 1);
        tc::mbar_init(&ms->q_empty, 1);
        tc::mbar_init(&ms->kv_full, kLoaders);
        for (int s = 0; s < 4; ++s) tc::mbar_init(&ms->kv_empty[s], 1);
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
    // Rows never written by a copy must hold finite values: zero Q and KV once.
    for (uint32_t i = tid; i < (kOffP - kOffKV) / 16; i += kThreads)
        reinterpret_cast<uint4 *>(smem + kOffKV)[i] = make_uint4(0, 0, 0, 0);
    tc::fence_proxy_async_smem();
    if (warp == 3) {
        tc::tmem_alloc(&ms->tmem_base, kTmemCols);
        tc::tmem_relinquish();
    }
    const bool use_cmp = a.cmp_kv != nullptr && a.Tc > 0;
    if (warp == 0 && lane == 0) {
        tc::tma_prefetch_desc(&q_map);
        tc::tma_prefetch_desc(&ori_map);
        tc::tma_prefetch_desc(&cmp_map);
    }
    // everything above is local: wait for the kernels before this one
    grid_dependency_wait();
    launch_dependents();
    if (tid < 64)
        ms->sink2[tid] = (a.sinks && tid < a.H) ? __ldg(a.sinks + tid) * kLog2e : -INFINITY;
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = ms->tmem_base;

    if (warp == 0) {
        // ================================================== scheduler warp
        uint32_t it = 0, q_n = 0;
        int32_t seg_lo = 0, seg_hi = 0, seg_b = -1;  // last sequence found: [lo, hi)
        // What the K/V tile holds after the previous token's last tile: kind,
        // sequence, token, ring base or box row, highest window row present
        // (ring), compressed rows on top (ring).
        int32_t bs_kind = -1, bs_seg = -1, bs_t = -1, bs_row0 = 0, bs_hi = 0, bs_top = 0;
        // The first 512 index entries of the next token, loaded one token
        // ahead so that their latency hides behind the wait for a free slot.
        int32_t jn[16];
        auto load_first_round = [&](int32_t tt) {
#pragma unroll
            for (int r = 0; r < 16; ++r) {
                const int32_t e = 32 * r + lane;
                jn[r] = (a.cmp_idx && tt < a.T && e < a.topk) ? __ldg(a.cmp_idx + (int64_t)tt * a.topk + e)
                                                               : -1;
            }
        };
        // Runs of tokens claimed from the launch's claim word: a quarter of an
        // even share of what is left, 2 to 256 tokens.
        unsigned long long *claim_word = &g_claim[a.claim_slot];
        int32_t run_end = 0;
        auto claim = [&]() -> int32_t {
            int64_t start = 0;
            uint32_t n = 0;
            if (lane == 0) {
                const int64_t left = max((int64_t)a.T - (int64_t)run_end, (int64_t)0);
                n = (uint32_t)min(max(left / (4 * (int64_t)gridDim.x), (int64_t)2), (int64_t)256);
                start = claim_run(claim_word, a.epoch, n);
                if (start == INT64_MAX) report_error(a.err, kErrCheck, kKerMla, 4);
            }
            start = __shfl_sync(0xffffffffu, start, 0);
            n = __shfl_sync(0xffffffffu, n, 0);
            if (start >= a.T) return a.T;
            run_end = (int32_t)min(start + (int64_t)n, (int64_t)a.T);
            return (int32_t)start;
        };
        int32_t t = claim();
        load_first_round(t);
        for (; t < a.T; ++it) {
            const uint32_t slot = it & 1;
            // the slot's key list is rewritten only once every consumer is done
            bool ok = cx.wait(&ms->info_empty[slot], ((it >> 1) & 1) ^ 1, 10);
            if (!__all_sync(0xffffffffu, ok)) break;
            int32_t *list = reinterpret_cast<int32_t *>(smem + kOffList) + slot * kMaxList;
            TokenInfo ti = {};
            ti.t = t;
            ti.single = -1;
            ti.b0 = -1;
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
                bs_kind = -1;
            } else {
                const int32_t seg0 = max(seg_lo, 0);
                const int32_t pos = t - seg0;
                ti.pos = pos;
                ti.seg = b;
                ti.win_start = max(t - a.window + 1, seg0);
                ti.n_win = t - ti.win_start + 1;
                int32_t n_cmp = 0, cbase = 0, vis = 0;
                bool run = true;
                if (use_cmp) {
                    cbase = __ldg(a.cu_c + b);
                    const int32_t seg_blocks = __ldg(a.cu_c + b + 1) - cbase;
                    vis = min((pos + 1) / a.cmp_ratio, seg_blocks);
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
                                jv[r] = e0 == 0 ? jn[r] : (e < a.topk ? __ldg(row + e) : -1);
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
                // every visible block, in order (the top-k kept them all)?
                const bool allvis = run && n_cmp == vis && (n_cmp == 0 || ti.cmp_first == cbase);
                ti.cbase = cbase;
                ti.n_cmp = n_cmp;
                ti.flags = (run ? kFlagRun : 0) | (allvis ? kFlagAllVis : 0);
                // Ring base, fixed by the position: a token at an odd position
                // starts the ring at its own window start; one at an even
                // position keeps the base of the position before it (its own
                // window is then that one plus its row).
                const bool ring_ok = a.window <= kTileKeys;
                if (ring_ok) ti.b0 = (pos & 1) ? ti.win_start : max(t - a.window, seg0);
                if (ti.n_win + n_cmp <= kTileKeys) {
                    ti.n_tiles = 1;
                    if (ring_ok && (n_cmp == 0 || (allvis && ti.win_start == seg0))) {
                        ti.single = kRing;  // window in slots [0, pos], blocks on top
                        ti.n_top = n_cmp;
                    } else {
                        ti.single = kGMix;
                    }
                } else {
                    ti.n_wt = ring_ok ? 1 : (ti.n_win + kTileKeys - 1) / kTileKeys;
                    ti.n_ct = (n_cmp + kTileKeys - 1) / kTileKeys;
                    ti.n_tiles = ti.n_wt + ti.n_ct;
                }
                ti.valid = 1;
                // Take over the previous token's last tile when it is this
                // token's first one, loading only what it lacks.
                const int32_t first_nat = tile_nat(ti, 0);
                const TileDesc f = tile_at(ti, first_nat);
                if (bs_t == t - 1 && bs_seg == b && bs_kind == f.kind && bs_row0 == f.row0) {
                    if (f.kind == kRing && bs_hi >= t - 1 && f.n_valid <= bs_top + 1) {
                        int32_t nd = 0;
                        if (t > bs_hi) {  // this token's own row
                            ti.d_row[nd] = t;
                            ti.d_slot[nd] = (t - f.row0) & (kTileKeys - 1);
                            ti.d_cmp[nd] = 0;
                            ++nd;
                        }
                        if (f.n_valid > bs_top) {  // a block that just became visible
                            ti.d_row[nd] = ti.cmp_first + bs_top;
                            ti.d_slot[nd] = kTileKeys - 1 - bs_top;
                            ti.d_cmp[nd] = 1;
                            ++nd;
                        }
                        ti.reuse = 1;
                        ti.n_delta = nd;
                    } else if (f.kind == kCmpBox) {
                        ti.reuse = 1;  // the box already holds the later blocks
                    }
                }
                // state after this token: its last tile
                const int32_t last_nat = tile_nat(ti, ti.n_tiles - 1);
                const TileDesc l = tile_at(ti, last_nat);
                if (l.kind == kRing) {
                    int32_t hi;
                    if (last_nat == first_nat && ti.reuse) hi = max(bs_hi, t);
                    else hi = ring_box(ti, l) ? l.row0 + kTileKeys - 1 : t;  // box / gather
                    if (l.n_valid > 0) hi = min(hi, t);  // later slots may hold blocks
                    bs_kind = kRing;
                    bs_hi = hi;
                    bs_top = l.n_valid;
                } else {
                    bs_kind = l.kind == kCmpBox ? kCmpBox : -1;
                    bs_hi = 0;
                    bs_top = 0;
                }
                bs_seg = b;
                bs_t = t;
                bs_row0 = l.row0;
            }
            // the token after this one: the next of the run, or a new run's first
            const int32_t next = t + 1 < run_end ? t + 1 : claim();
            __syncwarp();  // list writes before the release below
            if (lane == 0) {
                ms->info[slot] = ti;
                tc::mbar_arrive(&ms->info_full[slot]);
                // Q of the next token streams from HBM into L2 while this token
                // runs; its TMA load then hits L2.
                if (next < a.T)
                    tc::prefetch_l2_bulk(a.q + (int64_t)next * a.H * 512, (uint32_t)a.H * 1024u);
            }
            if (ti.valid) {
                // Q rows of token t (H rows of 512; rows >= H stay zero), once
                // the previous token's last S^T has read its Q
                ok = cx.wait(&ms->q_empty, (q_n & 1) ^ 1, 11);
                if (!__all_sync(0xffffffffu, ok)) break;
                if (lane == 0) {
                    tc::mbar_expect_tx(&ms->q_full, 8u * a.H * 128u);
                    for (int c = 0; c < 8; ++c)
                        tc::tma_load_3d(smem + kOffQ + c * 8192, &q_map, &ms->q_full, 64 * c, 0, t);
                }
                ++q_n;
            }
            load_first_round(next);
            t = next;
        }
        if (t >= a.T) {  // the end marker, once the slot is free
            const uint32_t slot = it & 1;
            const bool ok = cx.wait(&ms->info_empty[slot], ((it >> 1) & 1) ^ 1, 12);
            if (__all_sync(0xffffffffu, ok) && lane == 0) {
                TokenInfo ti = {};
                ti.end = 1;
                ms->info[slot] = ti;
                tc::mbar_arrive(&ms->info_full[slot]);
            }
        }
        if (lane == 0 && q_n > 0)  // drain: every Q copy issued has landed
            if (!tc::mbar_wait(&ms->q_full, (q_n - 1) & 1)) cx.fail(13);
    } else if (warp == 1 || warp == 2) {
        // ==================================================== loader warps
        // Gathered tiles: thread i covers, for slab s, the 16-byte column
        // 16 s + (i & 15) of the slots k = (i >> 4) + 4 m (m < 32): one
        // 256-byte row piece per quarter-warp, so every global access is a
        // coalesced run. Row addresses are computed once per tile.
        const int li = tid - 32;  // 0..63
        const int col = li & 15, sgrp = li >> 4;
        // kf_n counts the tiles loaded into. Both K/V barriers advance once
        // per loaded tile: kv_full when it has landed, kv_empty when the
        // tensor core has finished with the tile before it. A tile taken over
        // whole from the previous token loads nothing and touches neither, so
        // the parity waits below never fall more than one phase behind.
        uint32_t it = 0, kf_n = 0;
        const uint32_t kv_base = tc::smem_u32(smem + kOffKV);
        bool stop = false;
        for (; !stop; ++it) {
            const uint32_t slot = it & 1;
            // every lane of a loader warp takes the same decision on each wait
            if (!__all_sync(0xffffffffu, cx.wait(&ms->info_full[slot], (it >> 1) & 1, 40))) break;
            const TokenInfo &ti = ms->info[slot];  // released after this token's loads
            if (ti.end) break;
            const int32_t *list = reinterpret_cast<const int32_t *>(smem + kOffList) + slot * kMaxList;
            const int32_t n_tiles = ti.valid ? ti.n_tiles : 0;
            for (int32_t j = 0; j < n_tiles && !stop; ++j) {
                if (j == 0 && ti.reuse) {
                    if (ti.n_delta == 0) continue;
                    // the missing rows: 16 threads per row, 256 B per slab
                    const int dr = li >> 4;
                    for (int s = 0; s < 4; ++s) {
                        if (!__all_sync(0xffffffffu, cx.wait(&ms->kv_empty[s], (kf_n & 1) ^ 1, 44))) {
                            stop = true;
                            break;
                        }
                        if (dr < ti.n_delta) {
                            const int c16 = 16 * s + col;
                            const int chunk = c16 >> 3, w = c16 & 7;
                            const int k = ti.d_slot[dr];
                            const __nv_bfloat16 *src =
                                (ti.d_cmp[dr] ? a.cmp_kv : a.ori_kv) + (int64_t)ti.d_row[dr] * 512;
                            cp_async16(kv_base + chunk * 16384 + k * 128 + ((w ^ (k & 7)) << 4),
                                       src + c16 * 8);
                        }
                    }
                    if (!stop) cp_async_arrive(&ms->kv_full);
                    ++kf_n;
                    continue;
                }
                const TileDesc td = tile_at(ti, tile_nat(ti, j));
                if (td.kind == kWinBox || td.kind == kCmpBox || ring_box(ti, td)) {
                    const CUtensorMap *map = td.kind == kCmpBox ? &cmp_map : &ori_map;
                    for (int s = 0; s < 4; ++s) {
                        if (!__all_sync(0xffffffffu, cx.wait(&ms->kv_empty[s], (kf_n & 1) ^ 1, 41))) {
                            stop = true;
                            break;
                        }
                        if (li == 0) {
                            if (s == 0) tc::mbar_expect_tx(&ms->kv_full, 131072u);
                            for (int cc = 0; cc < 2; ++cc) {
                                const int c = 2 * s + cc;
                                tc::tma_load_2d(smem + kOffKV + c * 16384, map, &ms->kv_full,
                                                64 * c, td.row0);
                            }
                        }
                    }
                    if (!stop && li != 0) tc::mbar_arrive(&ms->kv_full);
                    ++kf_n;
                    continue;
                }
                // gathered tile: this thread's 32 slots
                const __nv_bfloat16 *src[32];
#pragma unroll
                for (int m = 0; m < 32; ++m) {
                    const int k = sgrp + 4 * m;
                    const __nv_bfloat16 *p = nullptr;
                    if (td.kind == kRing) {
                        if (k >= kTileKeys - td.n_valid) {
                            p = a.cmp_kv + (int64_t)(ti.cmp_first + (kTileKeys - 1 - k)) * 512;
                        } else {
                            const int32_t r = ti.t - ((ti.t - td.row0 - k) & (kTileKeys - 1));
                            if (r >= ti.win_start) p = a.ori_kv + (int64_t)r * 512;
                        }
                    } else if (td.kind == kGather) {
                        if (k < td.n_valid) {
                            const int32_t e = td.e0 + k;
                            const int32_t row = (ti.flags & kFlagRun) ? ti.cmp_first + e : list[e];
                            p = a.cmp_kv + (int64_t)row * 512;
                        }
                    } else {  // kGMix: window rows, then compressed entries
                        if (k < ti.n_win) {
                            p = a.ori_kv + (int64_t)(ti.win_start + k) * 512;
                        } else if (k < ti.n_win + ti.n_cmp) {
                            const int32_t e = k - ti.n_win;
                            const int32_t row = (ti.flags & kFlagRun) ? ti.cmp_first + e : list[e];
                            p = a.cmp_kv + (int64_t)row * 512;
                        }
                    }
                    src[m] = p;
                }
                // Each slab is released to the tensor core by the mbarrier
                // itself once this thread's copies land; the thread goes on to
                // the next slab without waiting.
                for (int s = 0; s < 4; ++s) {
                    if (!__all_sync(0xffffffffu, cx.wait(&ms->kv_empty[s], (kf_n & 1) ^ 1, 42))) {
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
                }
                if (!stop) cp_async_arrive(&ms->kv_full);
                ++kf_n;
            }
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&ms->info_empty[slot]);
        }
        cp_async_wait_all();  // drain: no copy outlives the CTA
        if (li == 0 && kf_n > 0)  // and no TMA copy either (last loaded tile's phase)
            if (!tc::mbar_wait(&ms->kv_full, (kf_n - 1) & 1)) cx.fail(43);
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
            uint32_t it = 0, q_n = 0, kf_n = 0, p_n = 0;
            bool issued = false;
            for (;; ++it) {
                const uint32_t slot = it & 1;
                if (!cx.wait(&ms->info_full[slot], (it >> 1) & 1, 20)) break;
                if (ms->info[slot].end) break;
                const int32_t n_tiles = ms->info[slot].valid ? ms->info[slot].n_tiles : 0;
                // a first tile taken over whole needs no load
                const bool first_loaded = !(ms->info[slot].reuse && ms->info[slot].n_delta == 0);
                tc::mbar_arrive(&ms->info_empty[slot]);
                if (n_tiles == 0) continue;
                bool stop = false;
                for (int32_t j = 0; j < n_tiles && !stop; ++j) {
                    const bool loaded = j > 0 || first_loaded;
                    // Q (first tile) and the whole tile, then all 32 S^T MMAs
                    // back to back: issuing slab by slab, between barrier
                    // checks, runs the tensor core at about half speed.
                    if ((j == 0 && !cx.wait(&ms->q_full, q_n & 1, 21)) ||
                        (loaded && !cx.wait(&ms->kv_full, kf_n & 1, 22))) {
                        stop = true;
                        break;
                    }
                    // slabs gathered by cp.async were written through the
                    // generic proxy: order them before the tensor core's reads
                    tc::fence_proxy_async_smem();
                    tc::tc_fence_after();
#pragma unroll
                    for (int c = 0; c < 8; ++c)
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            tc::mma_bf16(tmem + kColS, tc::desc_add(ds_a, c * 16384 + kk * 32),
                                         tc::desc_add(ds_b, c * 8192 + kk * 32), id_s, (c | kk) != 0);
                    issued = true;
                    // the last tile's S^T frees Q
                    if (j == n_tiles - 1) tc::mma_commit(&ms->q_empty);
                    if (loaded) ++kf_n;
                    tc::mma_commit(&ms->s_full);
                    if (!cx.wait(&ms->p_full, p_n & 1, 23)) {
                        stop = true;
                        break;
                    }
                    ++p_n;
                    // The K/V tile is handed back to the loaders only when the
                    // next tile loads into it: the next token's info decides
                    // for this token's last tile.
                    bool release = true;
                    if (j == n_tiles - 1) {
                        const uint32_t ns = (it + 1) & 1;
                        if (!cx.wait(&ms->info_full[ns], ((it + 1) >> 1) & 1, 25)) {
                            stop = true;
                            break;
                        }
                        const TokenInfo &nx = ms->info[ns];
                        release = !(!nx.end && nx.valid && nx.reuse && nx.n_delta == 0);
                    }
                    tc::tc_fence_after();
                    for (int s = 0; s < 4; ++s) {
#pragma unroll
                        for (int kk = 0; kk < 8; ++kk)
                            tc::mma_bf16(tmem + kColO + 64 * s,
                                         tc::desc_add(do_a, 2 * s * 16384 + kk * 2048),
                                         tc::desc_add(do_b, kk * 2048), id_o, (j > 0 || kk > 0));
                        if (release) tc::mma_commit(&ms->kv_empty[s]);
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
        for (;; ++it) {
            const uint32_t slot = it & 1;
            bool ok = cx.wait(&ms->info_full[slot], (it >> 1) & 1, 30);
            if (!bar_red_and(bar_id, ok)) break;
            const TokenInfo ti = ms->info[slot];  // a register copy; the slot is released at the end
            if (ti.end) break;
            const int32_t t = ti.t;
            if (!ti.valid) {
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(&ms->info_empty[slot]);
                continue;
            }
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
                // whether this thread's slot holds a key: known before the scores
                const bool key_ok = slot_valid(ti, tile_at(ti, tile_nat(ti, j)), row);
                ok = cx.wait(&ms->s_full, s_n & 1, 31);
                // A token's first tile agrees on the wait here; later tiles fold
                // it into the max vote below (one barrier per tile).
                if (j == 0 && !bar_red_and(bar_id, ok)) {
                    stop = true;
                    break;
                }
                ++s_n;
                tc::tc_fence_after();
                float v[32];
                tc::tmem_ld32(lane_addr + kColS + h0, v);
                tc::tmem_wait_ld();
                if (j == 0) {
                    // A token's first tile sets the max exactly: the max of the
                    // sink and the tile's scores, so the largest probability is
                    // exactly 1 in bf16 (a single dominant key then carries no
                    // rounding into P V). Row sums are still zero: nothing to scale.
#pragma unroll
                    for (int i = 0; i < 32; ++i) v[i] = key_ok ? v[i] * c : -INFINITY;
                    const uint32_t rs = tile_ctr & 1;
                    ms->red[rs][q4][h0 + lane] = reduce_scatter32<true>(v, lane);
                    tc::named_bar_sync(bar_id, 128);
                    const float mt =
                        fmaxf(fmaxf(ms->red[rs][0][h0 + lane], ms->red[rs][1][h0 + lane]),
                              fmaxf(ms->red[rs][2][h0 + lane], ms->red[rs][3][h0 + lane]));
                    m_lane = fmaxf(m_lane, mt);
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        m_cur[i] = __shfl_sync(0xffffffffu, m_lane, i);
                        v[i] -= m_cur[i];
                    }
                } else {
                    // v = scaled score - running max (base 2), -inf off the keys
#pragma unroll
                    for (int i = 0; i < 32; ++i) v[i] = key_ok ? fmaf(v[i], c, -m_cur[i]) : -INFINITY;
                    // After the first tile a head's max moves only when some score
                    // of a tile exceeds it by more than kLazyMax: the warpgroup
                    // first checks whether any does, and only then reduces the
                    // tile maxima.
                    bool exceeds = !ok;
#pragma unroll
                    for (int i = 0; i < 32; ++i) exceeds |= v[i] > kLazyMax;
                    if (bar_red_or(bar_id, exceeds)) {
                        // rare: some head's max moves, or some wait gave up
                        if (!bar_red_and(bar_id, ok)) {
                            stop = true;
                            break;
                        }
                        // the scaled scores again (S^T is still in tensor memory)
                        tc::tmem_ld32(lane_addr + kColS + h0, v);
                        tc::tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 32; ++i) v[i] = key_ok ? v[i] * c : -INFINITY;
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
#pragma unroll
                        for (int i = 0; i < 32; ++i) v[i] -= m_cur[i];
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
                        const float p0 = tc::ex2_approx(v[i]);
                        const float p1 = tc::ex2_approx(v[i + 1]);
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
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&ms->info_empty[slot]);
            tc::tc_fence_before();
        }
    }
    // ------------------------------------------------------------- teardown
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    if (warp == 3) tc::tmem_dealloc(tmem, kTmemCols);
    if (tid == 0) {  // the last CTA out resets the launch's claim word
        __threadfence();
        if (atomicAdd(&g_claim_done[a.claim_slot], 1u) == gridDim.x - 1) {
            atomicExch(&g_claim[a.claim_slot], 0ull);
            atomicExch(&g_claim_done[a.claim_slot], 0u);
        }
    }
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
    // Each launch takes a fresh epoch and the claim slot it selects.
    static std::atomic<uint32_t> epochs{0};
    MlaArgs la = a;
    la.epoch = epochs.fetch_add(1, std::memory_order_relaxed) + 1;
    la.claim_slot = (int32_t)(la.epoch % kClaimSlots);
    la.wait_ns = pipeline_wait_limit_ns();
    const int ctas = a.T < sms ? a.T : sms;
    return launch_early(sparse_mla_tc_kernel, dim3(ctas), dim3(kThreads), kSmemBytes, stream, q_map,
                        ori_map, cmp_map, la);
}

int32_t sparse_mla_max_topk() { return kMaxList; }

}  // namespace csa
