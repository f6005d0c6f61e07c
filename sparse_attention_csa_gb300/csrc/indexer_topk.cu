// Lightning-indexer score + per-sequence causal top-k over compressed KV
// (sm_103a, tcgen05 tensor cores, TMA).
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
// Design (persistent grid, 1 CTA per SM):
//   * Two consecutive tokens form a group. The contraction is done with the
//     compressed rows on the MMA's M side and the group's (token, head) pairs
//     on N:   S^T[j, (g,h)] = k[j, :] . q[t0+g, h, :]
//     (M = 128 rows, N = 2 x Hpad <= 128, K = Di), accumulated in fp32 in
//     tensor memory, four accumulators of 128 columns, so the epilogue of one
//     tile overlaps the MMAs of the next ones; k tiles come in three stages.
//     With one TMEM lane per row j, the head reduction sum_h w*relu(.) runs
//     inside each thread.
//   * A group whose tokens span several sequences is processed as one pass per
//     sequence (each with its own row range); visibility masks per token.
//   * The scores of a group go to one of two buffers in shared memory (global
//     scratch when a sequence offers more than kScoreCap rows). Four
//     selection warps select the top-k of one group while the eight epilogue
//     warps score the next into the other buffer: each token's selection is
//     done by two warps (pair_topk), a radix select on order-preserving keys
//     with 8-bit digits below the bits all of the token's keys share,
//     stopping once the threshold bucket is taken whole, and an emission in
//     row order.
//   * A token that sees at most topk blocks selects all of them whatever
//     their scores, so unless the caller asks for the values it is not scored
//     at all: a first pass marks the CTA's groups that hold a token to score,
//     only those go through the pipeline, and the epilogue warps write every
//     other row (16-byte stores) while the pipeline's loads and first MMAs
//     run.
//   * Warp roles: 0 producer (TMA), 1 tensor memory + MMA issue, 2-9 epilogue
//     (TMEM lane quarter x token), 10-13 selection. Every mbarrier wait is
//     bounded.
#include "common.cuh"
#include "internal.h"
#include "tc_ptx.cuh"
#include "tmap.h"

namespace csa {

namespace {

constexpr int kThreads = 448;   // producer, MMA, 8 epilogue warps, 4 selection warps
constexpr int kEpiThreads = 256;
constexpr int kSelThreads = 128;
constexpr int kG = 2;               // tokens per group
constexpr int kStagesA = 3;         // k tile stages
constexpr int kAccBufs = 4;         // tensor-memory accumulators (128 columns each)
constexpr int kInfoSlots = 4;       // group descriptors in flight
constexpr int kTileRows = 128;      // compressed rows per MMA tile
constexpr int kScoreCap = 5120;     // rows per token kept in shared memory
constexpr int kMaxCtas = 1024;      // persistent grid bound (sizes the scratch)
constexpr int kCuCap = 250;         // sequences whose offsets are staged in shared memory
constexpr int kGrpBits = 4096;      // groups per CTA tracked by the scored-group bitmap

// shared memory map (1024-aligned base)
constexpr uint32_t kOffB = 0;                 // q group: 2 chunks x [128 rows x 128 B]
constexpr uint32_t kOffA = 32768;             // k tiles: kStagesA stages x 2 chunks x 16 KB
constexpr uint32_t kOffScore = kOffA + kStagesA * 32768;  // 2 buffers x kG x kScoreCap fp32
constexpr uint32_t kOffMisc = kOffScore + 2 * kG * kScoreCap * 4;

struct Pass {
    int32_t mask, cbase, n_tiles, pad;
};

struct GroupInfo {
    int32_t t0, n_pass, spill, valid;
    int32_t nv[kG];       // visible rows per token (0: none / out of range)
    int32_t cb[kG];       // row base of each token's sequence
    Pass pass[kG];
};

struct Misc {
    uint64_t b_full, b_empty;
    uint64_t a_full[kStagesA], a_empty[kStagesA];
    uint64_t acc_full[kAccBufs], acc_empty[kAccBufs];
    uint64_t info_full[kInfoSlots], info_empty[kInfoSlots];
    uint64_t sc_full[2], sc_empty[2];  // score buffers: epilogue -> selection -> epilogue
    uint64_t drain;
    uint32_t tmem_base;
    int32_t abort;
    GroupInfo info[kInfoSlots];
    alignas(16) float w[kG * 64];
    int32_t hist[kG][2][256];  // per token: two rounds of packed counts (two warps)
    uint32_t keyrange[2][kG][2];  // per score buffer and token: smallest and largest key
    int32_t cu_q[kCuCap + 1], cu_c[kCuCap + 1];  // sequence offsets, when batch <= kCuCap
    uint32_t gscored[kGrpBits / 32];             // this CTA's groups with a token to score
};

constexpr size_t kSmemBytes = kOffMisc + sizeof(Misc) + 1024;
static_assert(kSmemBytes <= 232448, "shared memory budget");

// AND of v over the `n` threads of named barrier `id` (whole warps).
__device__ __forceinline__ bool bar_red_and(uint32_t id, uint32_t n, bool v) {
    uint32_t out;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.and.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(out)
        : "r"((uint32_t)v), "r"(id), "r"(n)
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
        report_error(err, kErrTimeout, kKerIndexer, site);
    }
    __device__ __forceinline__ bool wait(uint64_t *bar, uint32_t parity, int site) const {
        if (aborted()) return false;
        if (tc::mbar_wait(bar, parity, limit)) return true;
        fail(site);
        return false;
    }
};

__device__ __forceinline__ int32_t warp_excl_scan(int32_t v, int lane, int32_t *total) {
    int32_t x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int32_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    *total = __shfl_sync(0xffffffffu, x, 31);
    return x - v;
}

// Scores in shared memory are read with shared-space loads (the score row
// pointer is generic: it may point to the global spill buffer instead).
template <bool kShared>
struct ScoreRow {
    const float *p;
    uint32_t s;  // shared-space address of p when kShared
    __device__ __forceinline__ explicit ScoreRow(const float *ptr)
        : p(ptr), s(kShared ? (uint32_t)__cvta_generic_to_shared(ptr) : 0u) {}
    __device__ __forceinline__ float operator[](int32_t i) const {
        if constexpr (kShared) {
            float v;
            asm("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(s + 4u * (uint32_t)i));
            return v;
        } else {
            return p[i];
        }
    }
};

__device__ __forceinline__ void hist_add(uint32_t hist_s, uint32_t bin) {
    asm volatile("red.shared.add.u32 [%0], 1;" ::"r"(hist_s + 4u * bin) : "memory");
}

// One warp selects the top K of sc[0..n) (ties to the lower index) and writes
// them in ascending index order as base + index (values alongside).
// Radix select on order-preserving keys: a first sweep finds the smallest and
// largest key, whose common leading bits every key shares (scores of one
// token often share sign and exponent); the digits below them are then fixed
// 8 bits a sweep from the top. Each sweep counts, in a 256-bin shared
// histogram, the keys that match the digits fixed so far, and fixes the next
// digit as the one holding the K-th largest; the search stops once every key
// of that bucket is taken (its count equals what is left to take), usually
// after two or three sweeps. One more sweep emits, 32 consecutive indices at
// a time, every key above the bucket and the bucket's keys in index order up
// to the count left (so equal keys go to the lower index). Every sweep loads
// kBatch scores per lane before using any, so that the loads overlap.
template <bool kShared>
__device__ void warp_topk(const float *scores, int32_t n, int32_t K, int32_t base,
                          int32_t *__restrict__ idx_row, float *__restrict__ val_row,
                          int32_t *hist, int lane) {
    const ScoreRow<kShared> sc(scores);
    const uint32_t hist_s = (uint32_t)__cvta_generic_to_shared(hist);
    if (n <= K) {
        for (int32_t i = lane; i < K; i += 32) {
            idx_row[i] = i < n ? base + i : -1;
            if (val_row) val_row[i] = i < n ? sc[i] : -INFINITY;
        }
        return;
    }
    constexpr int kBatch = 8;
    uint32_t keys[kBatch];
    auto load_keys = [&](int32_t i0) {  // indices i0 + 32 m + lane
        float v[kBatch];
#pragma unroll
        for (int m = 0; m < kBatch; ++m) v[m] = sc[min(i0 + 32 * m + lane, n - 1)];  // in bounds
#pragma unroll
        for (int m = 0; m < kBatch; ++m) keys[m] = i0 + 32 * m + lane < n ? float_key(v[m]) : 0u;
    };
    uint32_t lo = 0xffffffffu, hi = 0u;
    for (int32_t i0 = 0; i0 < n; i0 += 32 * kBatch) {
        load_keys(i0);
#pragma unroll
        for (int m = 0; m < kBatch; ++m)
            if (i0 + 32 * m + lane < n) {
                lo = min(lo, keys[m]);
                hi = max(hi, keys[m]);
            }
    }
    lo = __reduce_min_sync(0xffffffffu, lo);
    hi = __reduce_max_sync(0xffffffffu, hi);
    // bits below the common leading ones: 0 when every key is equal
    const int free_bits = (lo == hi) ? 0 : 32 - __clz((int)(lo ^ hi));
    uint32_t mask = free_bits == 32 ? 0u : ~((1u << free_bits) - 1u);
    uint32_t prefix = lo & mask;
    int32_t k_rem = K;
#pragma unroll 1
    for (int top = free_bits; top > 0; top -= 8) {
        const int shift = max(top - 8, 0);
        const uint32_t dmask = (1u << (top - shift)) - 1u;
#pragma unroll
        for (int i = 0; i < 8; ++i) hist[lane + 32 * i] = 0;
        __syncwarp();
        for (int32_t i0 = 0; i0 < n; i0 += 32 * kBatch) {
            load_keys(i0);
#pragma unroll
            for (int m = 0; m < kBatch; ++m)
                if (i0 + 32 * m + lane < n && (keys[m] & mask) == prefix)
                    hist_add(hist_s, (keys[m] >> shift) & dmask);
        }
        __syncwarp();
        int32_t c[8], local = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            c[i] = hist[255 - (lane * 8 + i)];
            local += c[i];
        }
        int32_t tot;
        int32_t above = warp_excl_scan(local, lane, &tot);
        int32_t my_digit = -1, my_above = 0, my_count = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            if (above < k_rem && k_rem <= above + c[i]) {
                my_digit = 255 - (lane * 8 + i);
                my_above = above;
                my_count = c[i];
            }
            above += c[i];
        }
        const uint32_t who = __ballot_sync(0xffffffffu, my_digit >= 0);
        const int src = who ? __ffs(who) - 1 : 0;
        const int32_t digit = __shfl_sync(0xffffffffu, my_digit, src);
        k_rem -= __shfl_sync(0xffffffffu, my_above, src);
        const int32_t count = __shfl_sync(0xffffffffu, my_count, src);
        prefix |= (uint32_t)max(digit, 0) << shift;
        mask |= dmask << shift;
        __syncwarp();
        if (count == k_rem) break;  // the whole bucket is taken
    }
    // Emission: all ballots of a batch first (they do not depend on one
    // another), then the running counts as warp-uniform integers, then each
    // lane's stores.
    const uint32_t below = (1u << lane) - 1u;
    int32_t pos = 0, eq_seen = 0;
    for (int32_t i0 = 0; i0 < n; i0 += 32 * kBatch) {
        load_keys(i0);
        uint32_t gts[kBatch], eqs[kBatch];
#pragma unroll
        for (int m = 0; m < kBatch; ++m) {
            const bool in = i0 + 32 * m + lane < n;
            const uint32_t mu = keys[m] & mask;
            gts[m] = __ballot_sync(0xffffffffu, in && mu > prefix);
            eqs[m] = __ballot_sync(0xffffffffu, in && mu == prefix);
        }
        uint32_t takes[kBatch];
        int32_t before[kBatch];
#pragma unroll
        for (int m = 0; m < kBatch; ++m) {
            // the bucket's keys of this round that are still taken: the first
            // `quota` set bits of eqs[m]
            const int32_t ne = __popc(eqs[m]);
            const int32_t quota = k_rem - eq_seen;
            uint32_t eq_take = eqs[m];
            if (quota <= 0) {
                eq_take = 0u;
            } else if (quota < ne) {
                uint32_t x = eqs[m];  // clear its quota - 1 lowest set bits
                for (int32_t j = 1; j < quota; ++j) x &= x - 1u;
                const int last = __ffs(x) - 1;  // the quota-th set bit
                eq_take &= last >= 31 ? 0xffffffffu : ((2u << last) - 1u);
            }
            takes[m] = gts[m] | eq_take;
            before[m] = pos;
            pos += __popc(takes[m]);
            eq_seen += ne;
        }
#pragma unroll
        for (int m = 0; m < kBatch; ++m) {
            if ((takes[m] >> lane) & 1u) {
                const int32_t i = i0 + 32 * m + lane;
                const int32_t p = before[m] + __popc(takes[m] & below);
                idx_row[p] = base + i;
                if (val_row) val_row[p] = sc[min(i, n - 1)];  // i < n: taken
            }
        }
    }
}

// The same selection by two warps (part 0 and part 1, joined by the 64-thread
// named barrier `bar`), each sweeping one contiguous half of the scores; the
// smallest and largest keys come from the epilogue, and each pass's histogram holds both halves' counts packed in one
// word (part 0 in the low 16 bits, part 1 in the high), so that both warps
// fix the same digit and each also learns how many keys of its own half lie
// above the bucket and in it. Part 1's first output slot is then part 0's
// count above the bucket plus the bucket keys part 0 takes, with no further
// exchange. Two rounds of histograms alternate, so one barrier separates a
// pass's reads from the next pass's zeroing. Rows of more than pair_max
// scores (at most kPairMax: 16-bit counts) go to warp_topk on part 0 alone.
constexpr int32_t kPairMax = 130000;

template <bool kShared>
__device__ void pair_topk(const float *scores, int32_t n, int32_t K, int32_t base,
                          int32_t *__restrict__ idx_row, float *__restrict__ val_row,
                          int32_t (*hist)[256], uint32_t lo, uint32_t hi, int part, int lane,
                          uint32_t bar, int32_t pair_max) {
    if (n > pair_max) {
        if (part == 0) warp_topk<kShared>(scores, n, K, base, idx_row, val_row, hist[0], lane);
        return;
    }
    const ScoreRow<kShared> sc(scores);
    if (n <= K) {
        for (int32_t i = lane + 32 * part; i < K; i += 64) {
            idx_row[i] = i < n ? base + i : -1;
            if (val_row) val_row[i] = i < n ? sc[i] : -INFINITY;
        }
        return;
    }
    constexpr int kBatch = 8, kSpan = 32 * kBatch;
    const int32_t nb = (n + kSpan - 1) / kSpan, nbh = (nb + 1) / 2;
    const int32_t split = min(n, nbh * kSpan);  // part 0: [0, split), part 1: [split, n)
    const int32_t r0 = part ? split : 0, r1 = part ? n : split;
    uint32_t keys[kBatch];
    auto load_keys = [&](int32_t i0) {  // indices i0 + 32 m + lane of this half
        float v[kBatch];
#pragma unroll
        for (int m = 0; m < kBatch; ++m) v[m] = sc[min(i0 + 32 * m + lane, n - 1)];  // in bounds
#pragma unroll
        for (int m = 0; m < kBatch; ++m) keys[m] = i0 + 32 * m + lane < r1 ? float_key(v[m]) : 0u;
    };
    // lo, hi: the smallest and largest key of all n scores (the epilogue
    // tracks them while it writes the scores)
    const int free_bits = (lo == hi) ? 0 : 32 - __clz((int)(lo ^ hi));
    uint32_t mask = free_bits == 32 ? 0u : ~((1u << free_bits) - 1u);
    uint32_t prefix = lo & mask;
    int32_t k_rem = K;
    // keys of each half above the bucket and in it (all of them when every
    // key is equal and no pass runs)
    int32_t above0 = 0, above1 = 0, eq0 = split, eq1 = n - split;
    int hb = 0;
#pragma unroll 1
    for (int top = free_bits; top > 0; top -= 8, hb ^= 1) {
        const int shift = max(top - 8, 0);
        const uint32_t dmask = (1u << (top - shift)) - 1u;
        int32_t *H = hist[hb];
        const uint32_t hs = (uint32_t)__cvta_generic_to_shared(H);
        for (int i = lane + 32 * part; i < 256; i += 64) H[i] = 0;
        tc::named_bar_sync(bar, 64);
        const uint32_t one = part ? 65536u : 1u;
        for (int32_t i0 = r0; i0 < r1; i0 += kSpan) {
            load_keys(i0);
#pragma unroll
            for (int m = 0; m < kBatch; ++m)
                if (i0 + 32 * m + lane < r1 && (keys[m] & mask) == prefix)
                    asm volatile("red.shared.add.u32 [%0], %1;" ::"r"(hs + 4u * ((keys[m] >> shift) & dmask)),
                                 "r"(one)
                                 : "memory");
        }
        tc::named_bar_sync(bar, 64);
        uint32_t cw[8];
        int32_t c[8], local = 0, local0 = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            cw[i] = (uint32_t)H[255 - (lane * 8 + i)];
            c[i] = (int32_t)((cw[i] & 0xffffu) + (cw[i] >> 16));
            local += c[i];
            local0 += (int32_t)(cw[i] & 0xffffu);
        }
        int32_t tot;
        int32_t above = warp_excl_scan(local, lane, &tot);
        int32_t a0 = warp_excl_scan(local0, lane, &tot);
        int32_t my_digit = -1, my_above = 0, my_a0 = 0;
        uint32_t my_cw = 0u;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            if (above < k_rem && k_rem <= above + c[i]) {
                my_digit = 255 - (lane * 8 + i);
                my_above = above;
                my_a0 = a0;
                my_cw = cw[i];
            }
            above += c[i];
            a0 += (int32_t)(cw[i] & 0xffffu);
        }
        const uint32_t who = __ballot_sync(0xffffffffu, my_digit >= 0);
        const int src = who ? __ffs(who) - 1 : 0;
        const int32_t digit = __shfl_sync(0xffffffffu, my_digit, src);
        const int32_t A = __shfl_sync(0xffffffffu, my_above, src);
        const int32_t A0 = __shfl_sync(0xffffffffu, my_a0, src);
        const uint32_t bucket = __shfl_sync(0xffffffffu, my_cw, src);
        k_rem -= A;
        above0 += A0;
        above1 += A - A0;
        eq0 = (int32_t)(bucket & 0xffffu);
        eq1 = (int32_t)(bucket >> 16);
        prefix |= (uint32_t)max(digit, 0) << shift;
        mask |= dmask << shift;
        if (eq0 + eq1 == k_rem) break;  // the whole bucket is taken
    }
    (void)above1;
    // emission of this half: part 1 starts after what part 0 takes
    int32_t pos = part ? above0 + min(eq0, k_rem) : 0;
    const int32_t quota = part ? max(0, k_rem - eq0) : k_rem;
    const uint32_t below = (1u << lane) - 1u;
    int32_t eq_seen = 0;
    for (int32_t i0 = r0; i0 < r1; i0 += kSpan) {
        load_keys(i0);
        uint32_t gts[kBatch], eqs[kBatch];
#pragma unroll
        for (int m = 0; m < kBatch; ++m) {
            const bool in = i0 + 32 * m + lane < r1;
            const uint32_t mu = keys[m] & mask;
            gts[m] = __ballot_sync(0xffffffffu, in && mu > prefix);
            eqs[m] = __ballot_sync(0xffffffffu, in && mu == prefix);
        }
        uint32_t takes[kBatch];
        int32_t before[kBatch];
#pragma unroll
        for (int m = 0; m < kBatch; ++m) {
            const int32_t ne = __popc(eqs[m]);
            const int32_t left = quota - eq_seen;
            uint32_t eq_take = eqs[m];
            if (left <= 0) {
                eq_take = 0u;
            } else if (left < ne) {
                uint32_t x = eqs[m];  // clear its left - 1 lowest set bits
                for (int32_t j = 1; j < left; ++j) x &= x - 1u;
                const int last = __ffs(x) - 1;  // the left-th set bit
                eq_take &= last >= 31 ? 0xffffffffu : ((2u << last) - 1u);
            }
            takes[m] = gts[m] | eq_take;
            before[m] = pos;
            pos += __popc(takes[m]);
            eq_seen += ne;
        }
#pragma unroll
        for (int m = 0; m < kBatch; ++m) {
            if ((takes[m] >> lane) & 1u) {
                const int32_t i = i0 + 32 * m + lane;
                const int32_t p = before[m] + __popc(takes[m] & below);
                idx_row[p] = base + i;
                if (val_row) val_row[p] = sc[min(i, n - 1)];  // i < n: taken
            }
        }
    }
}

template <int HPAD, int DI>
__global__ void __launch_bounds__(kThreads, 1)
indexer_tc_kernel(const __grid_constant__ CUtensorMap q_map,
                  const __grid_constant__ CUtensorMap k_map, const __grid_constant__ IndexerArgs a) {
    constexpr int N = kG * HPAD;          // MMA N
    constexpr int NCH = DI / 64;          // 128-byte chunks per row
    constexpr uint32_t kBChunk = N * 128; // bytes per B chunk
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem =
        reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                          ~uintptr_t(1023));
    Misc *ms = reinterpret_cast<Misc *>(smem + kOffMisc);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    Ctx cx{ms, a.err, a.wait_ns};
    const int32_t n_groups = (a.T + kG - 1) / kG;

    if (tid == 0) {
        tc::mbar_init(&ms->b_full, 1);
        tc::mbar_init(&ms->b_empty, 1);
        for (int i = 0; i < kStagesA; ++i) {
            tc::mbar_init(&ms->a_full[i], 1);
            tc::mbar_init(&ms->a_empty[i], 1);
        }
        for (int i = 0; i < kAccBufs; ++i) {
            tc::mbar_init(&ms->acc_full[i], 1);
            tc::mbar_init(&ms->acc_empty[i], kEpiThreads);
        }
        for (int i = 0; i < kInfoSlots; ++i) {
            tc::mbar_init(&ms->info_full[i], 1);
            tc::mbar_init(&ms->info_empty[i], 13);  // the MMA thread, 8 epilogue and 4 selection warps
        }
        for (int i = 0; i < 2; ++i) {
            tc::mbar_init(&ms->sc_full[i], 1);
            tc::mbar_init(&ms->sc_empty[i], 1);
        }
        tc::mbar_init(&ms->drain, 1);
        ms->abort = 0;
        tc::fence_mbar_init();
    }
    if (warp == 1) {
        tc::tmem_alloc(&ms->tmem_base, 512);
        tc::tmem_relinquish();
    }
    if (warp == 0 && lane == 0) {
        tc::tma_prefetch_desc(&q_map);
        tc::tma_prefetch_desc(&k_map);
    }
    // everything above is local: wait for the kernels before this one
    grid_dependency_wait();
    launch_dependents();
    // The producer looks up every token's sequence: keep the offsets on chip.
    const bool cu_smem = a.batch <= kCuCap;
    if (cu_smem)
        for (int i = tid; i <= a.batch; i += kThreads) {
            ms->cu_q[i] = __ldg(a.cu_q + i);
            ms->cu_c[i] = a.Tc > 0 ? __ldg(a.cu_c + i) : 0;
        }
    // This CTA's groups are blockIdx.x + k gridDim.x. Unless values are
    // requested, a first pass marks those holding a token to score; only they
    // go through the pipeline below, and the epilogue warps write the other
    // rows (all visible blocks, then -1) before they start on it.
    const int64_t my_groups =
        blockIdx.x < (uint32_t)n_groups ? (n_groups - 1 - (int64_t)blockIdx.x) / gridDim.x + 1 : 0;
    const bool bulk = a.topk_val == nullptr && my_groups <= kGrpBits;
    const int32_t *cq = cu_smem ? ms->cu_q : a.cu_q;
    const int32_t *cc = cu_smem ? ms->cu_c : a.cu_c;
    // Visible rows of token t (0 when none; -1 when t is outside the pack or
    // the offsets are inconsistent, reported) and their first row.
    auto visible = [&](int32_t t, int32_t *cb) -> int32_t {
        const int32_t seg = cu_smem ? find_segment_smem(cq, a.batch, t) : find_segment(cq, a.batch, t);
        *cb = 0;
        if (seg < 0) return -1;
        if (a.Tc <= 0) return 0;
        const int32_t pos = t - cq[seg];
        *cb = cc[seg];
        const int32_t n = min((pos + 1) / a.cmp_ratio, cc[seg + 1] - *cb);
        return (*cb < 0 || n < 0 || (int64_t)*cb + n > a.Tc) ? -2 : n;
    };
    for (int i = tid; i < kGrpBits / 32; i += kThreads) ms->gscored[i] = 0;
    __syncthreads();
    if (bulk) {
        for (int64_t li = tid; li < my_groups * kG; li += kThreads) {
            const int64_t k = li / kG;
            const int32_t t = (int32_t)(((int64_t)blockIdx.x + k * gridDim.x) * kG + li % kG);
            int32_t cb;
            if (t < a.T && visible(t, &cb) > a.topk) atomicOr(&ms->gscored[k >> 5], 1u << (k & 31));
        }
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = ms->tmem_base;

    // Rows of the groups with nothing to score, written by the twelve epilogue
    // and selection warps first (while the producer and the MMA warp start on
    // the scored groups): 32 tokens found at a time per warp, one row per warp
    // store round (16-byte stores when aligned).
    auto bulk_fill = [&]() {
        if (!bulk) return;
        const bool vec = (a.topk & 3) == 0 && (reinterpret_cast<uintptr_t>(a.topk_idx) & 15) == 0;
        for (int64_t base = 32 * (warp - 2); base < my_groups * kG; base += 384) {
            const int64_t li = base + lane;
            const int64_t k = li / kG;
            int32_t t = -1, n = 0, cb = 0;
            bool write = false;
            if (li < my_groups * kG && !((ms->gscored[k >> 5] >> (k & 31)) & 1u)) {
                t = (int32_t)(((int64_t)blockIdx.x + k * gridDim.x) * kG + li % kG);
                if (t < a.T) {
                    write = true;
                    n = visible(t, &cb);
                    if (n < 0) {
                        report_error(a.err, kErrCheck, kKerIndexer, n == -1 ? 1 : 2);
                        n = 0;
                    }
                }
            }
            for (uint32_t m = __ballot_sync(0xffffffffu, write); m; m &= m - 1) {
                const int src = __ffs(m) - 1;
                const int32_t tw = __shfl_sync(0xffffffffu, t, src);
                const int32_t nw = __shfl_sync(0xffffffffu, n, src);
                const int32_t cw = __shfl_sync(0xffffffffu, cb, src);
                int32_t *idx_row = a.topk_idx + (int64_t)tw * a.topk;
                if (vec) {
                    for (int32_t i = 4 * lane; i < a.topk; i += 128)
                        *reinterpret_cast<int4 *>(idx_row + i) =
                            make_int4(i < nw ? cw + i : -1, i + 1 < nw ? cw + i + 1 : -1,
                                      i + 2 < nw ? cw + i + 2 : -1, i + 3 < nw ? cw + i + 3 : -1);
                } else {
                    for (int32_t i = lane; i < a.topk; i += 32) idx_row[i] = i < nw ? cw + i : -1;
                }
            }
        }
    };

    if (warp == 0) {
        // ===================================================== producer warp
        uint32_t it = 0, b_n = 0, a_n = 0;
        bool quit = false;
        int64_t kg = 0;
        for (int32_t grp = blockIdx.x; grp < n_groups && !quit; grp += gridDim.x, ++kg) {
            // rows already written by the bulk pass and nothing to score
            if (bulk && !((ms->gscored[kg >> 5] >> (kg & 31)) & 1u)) continue;
            GroupInfo gi;
            gi.t0 = grp * kG;
            gi.n_pass = 0;
            gi.spill = 0;
            gi.valid = 1;
            // Lane g < kG works out token t0 + g; the warp then shares the results.
            int32_t my_seg = -1, my_nv = 0, my_cb = 0;
            bool my_scored = false;
            {
                const int32_t t = gi.t0 + lane;
                if (lane < kG && t < a.T) {
                    const int32_t *cq = cu_smem ? ms->cu_q : a.cu_q;
                    const int32_t *cc = cu_smem ? ms->cu_c : a.cu_c;
                    my_seg = cu_smem ? find_segment_smem(cq, a.batch, t) : find_segment(cq, a.batch, t);
                    if (my_seg < 0) {
                        report_error(a.err, kErrCheck, kKerIndexer, 1);
                    } else if (a.Tc > 0) {
                        const int32_t pos = t - cq[my_seg];
                        const int32_t cbase = cc[my_seg];
                        int32_t nv = min((pos + 1) / a.cmp_ratio, cc[my_seg + 1] - cbase);
                        if (cbase < 0 || nv < 0 || (int64_t)cbase + nv > a.Tc) {
                            report_error(a.err, kErrCheck, kKerIndexer, 2);
                            nv = 0;
                        }
                        my_nv = nv;
                        my_cb = cbase;
                        // A token that sees at most topk blocks keeps all of
                        // them, whatever their scores: it is scored only if the
                        // caller asked for the values.
                        my_scored = nv > 0 && (a.topk_val != nullptr || nv > a.topk);
                    }
                }
            }
            int32_t segs[kG];
            bool scored[kG];
#pragma unroll
            for (int g = 0; g < kG; ++g) {
                segs[g] = __shfl_sync(0xffffffffu, my_seg, g);
                gi.nv[g] = __shfl_sync(0xffffffffu, my_nv, g);
                gi.cb[g] = __shfl_sync(0xffffffffu, my_cb, g);
                scored[g] = __shfl_sync(0xffffffffu, my_scored ? 1 : 0, g) != 0;
                gi.pass[g] = Pass{0, 0, 0, 0};
                if (scored[g] && gi.nv[g] > kScoreCap) gi.spill = 1;
            }
            // one pass per run of tokens sharing a sequence
#pragma unroll
            for (int g = 0; g < kG; ++g) {
                if (segs[g] < 0 || !scored[g]) continue;
                const bool joins = g > 0 && gi.n_pass > 0 && segs[g - 1] == segs[g] &&
                                   scored[g - 1];
                if (joins) {
                    Pass &p = gi.pass[gi.n_pass - 1];
                    p.mask |= 1 << g;
                    p.n_tiles = max(p.n_tiles, (gi.nv[g] + kTileRows - 1) / kTileRows);
                } else {
                    Pass &p = gi.pass[gi.n_pass++];
                    p.mask = 1 << g;
                    p.cbase = gi.cb[g];
                    p.n_tiles = (gi.nv[g] + kTileRows - 1) / kTileRows;
                    p.pad = 0;
                }
            }
            if (gi.spill && a.scratch == nullptr) {
                if (lane == 0) report_error(a.err, kErrCheck, kKerIndexer, 3);
                gi.valid = 0;
            }
            if (!gi.valid || gi.n_pass == 0) {
                // Nothing to score: each token keeps all its visible blocks
                // (none when invalid). This warp writes the rows itself and the
                // group never reaches the other roles.
                const bool vec = (a.topk & 3) == 0 && (reinterpret_cast<uintptr_t>(a.topk_idx) & 15) == 0;
                for (int g = 0; g < kG; ++g) {
                    const int32_t t = gi.t0 + g;
                    if (t >= a.T) break;
                    const int32_t n = gi.valid ? gi.nv[g] : 0, cb = gi.cb[g];
                    int32_t *idx_row = a.topk_idx + (int64_t)t * a.topk;
                    if (vec) {  // 16-byte stores: four entries per lane
                        for (int32_t i = 4 * lane; i < a.topk; i += 128)
                            *reinterpret_cast<int4 *>(idx_row + i) =
                                make_int4(i < n ? cb + i : -1, i + 1 < n ? cb + i + 1 : -1,
                                          i + 2 < n ? cb + i + 2 : -1, i + 3 < n ? cb + i + 3 : -1);
                    } else {
                        for (int32_t i = lane; i < a.topk; i += 32) idx_row[i] = i < n ? cb + i : -1;
                    }
                    if (a.topk_val)  // only rows with no visible block get here
                        for (int32_t i = lane; i < a.topk; i += 32)
                            a.topk_val[(int64_t)t * a.topk + i] = -INFINITY;
                }
                continue;
            }
            // Start the group's q rows and its first k tile towards L2 while
            // the buffers they go to are still in use.
            if (lane == 0) {
                const int32_t nt = min(kG, a.T - gi.t0);
                tc::prefetch_l2_bulk(a.q + (int64_t)gi.t0 * a.Hi * DI, (uint32_t)(nt * a.Hi * DI * 2));
                const int32_t rows = min(kTileRows, gi.nv[__ffs(gi.pass[0].mask) - 1]);
                if (rows > 0)
                    tc::prefetch_l2_bulk(a.k + (int64_t)gi.pass[0].cbase * DI, (uint32_t)(rows * DI * 2));
            }
            const uint32_t slot = it % kInfoSlots;
            bool ok = cx.wait(&ms->info_empty[slot], ((it / kInfoSlots) & 1) ^ 1, 10);
            if (!__all_sync(0xffffffffu, ok)) break;
            if (lane == 0) {
                ms->info[slot] = gi;
                tc::mbar_arrive(&ms->info_full[slot]);
            }
            ++it;
            // q rows of the group (kG tokens x HPAD heads; missing rows read as 0)
            ok = cx.wait(&ms->b_empty, (b_n & 1) ^ 1, 11);
            if (!__all_sync(0xffffffffu, ok)) break;
            if (lane == 0) {
                tc::mbar_expect_tx(&ms->b_full, NCH * kBChunk);
                for (int c = 0; c < NCH; ++c)
                    tc::tma_load_3d(smem + kOffB + c * kBChunk, &q_map, &ms->b_full, 64 * c, 0,
                                    gi.t0);
            }
            ++b_n;
            bool broke = false;
            for (int p = 0; p < gi.n_pass && !broke; ++p) {
                for (int32_t j = 0; j < gi.pass[p].n_tiles; ++j, ++a_n) {
                    const uint32_t st = a_n % kStagesA;
                    ok = cx.wait(&ms->a_empty[st], ((a_n / kStagesA) & 1) ^ 1, 12);
                    if (!__all_sync(0xffffffffu, ok)) {
                        broke = true;
                        break;
                    }
                    if (lane == 0) {
                        tc::mbar_expect_tx(&ms->a_full[st], NCH * 16384u);
                        for (int c = 0; c < NCH; ++c)
                            tc::tma_load_2d(smem + kOffA + st * 32768u + c * 16384, &k_map,
                                            &ms->a_full[st], 64 * c,
                                            gi.pass[p].cbase + j * kTileRows);
                    }
                }
            }
            if (broke) quit = true;
        }
        // end of the stream: a group with valid = -1 stops the other roles
        if (!quit) {
            const uint32_t slot = it % kInfoSlots;
            const bool ok = cx.wait(&ms->info_empty[slot], ((it / kInfoSlots) & 1) ^ 1, 15);
            if (__all_sync(0xffffffffu, ok) && lane == 0) {
                ms->info[slot].valid = -1;
                tc::mbar_arrive(&ms->info_full[slot]);
            }
        }
        // drain: every copy issued has landed before the CTA exits
        if (lane == 0) {
            if (b_n > 0 && !tc::mbar_wait(&ms->b_full, (b_n - 1) & 1)) cx.fail(13);
            for (uint32_t k = (a_n > kStagesA ? a_n - kStagesA : 0); k < a_n; ++k)
                if (!tc::mbar_wait(&ms->a_full[k % kStagesA], (k / kStagesA) & 1)) cx.fail(14);
        }
    } else if (warp == 1) {
        // ========================================================= MMA warp
        if (lane == 0) {
            const uint32_t idesc = tc::idesc_bf16(128, N, false, false);
            const uint64_t da = tc::smem_desc(tc::smem_u32(smem + kOffA), 16, 1024);
            const uint64_t db = tc::smem_desc(tc::smem_u32(smem + kOffB), 16, 1024);
            uint32_t it = 0, b_n = 0, a_n = 0, t_n = 0;
            bool issued = false;
            for (;; ++it) {
                const uint32_t slot = it % kInfoSlots;
                if (!cx.wait(&ms->info_full[slot], (it / kInfoSlots) & 1, 20)) break;
                const GroupInfo gi = ms->info[slot];
                tc::mbar_arrive(&ms->info_empty[slot]);
                if (gi.valid < 0) break;
                if (!gi.valid || gi.n_pass == 0) continue;
                if (!cx.wait(&ms->b_full, b_n & 1, 21)) break;
                ++b_n;
                bool stop = false;
                for (int p = 0; p < gi.n_pass && !stop; ++p) {
                    for (int32_t j = 0; j < gi.pass[p].n_tiles; ++j, ++a_n, ++t_n) {
                        const uint32_t st = a_n % kStagesA, buf = t_n % kAccBufs;
                        if (!cx.wait(&ms->acc_empty[buf], ((t_n / kAccBufs) & 1) ^ 1, 22) ||
                            !cx.wait(&ms->a_full[st], (a_n / kStagesA) & 1, 23)) {
                            stop = true;
                            break;
                        }
                        tc::tc_fence_after();
#pragma unroll
                        for (int kk = 0; kk < DI / 16; ++kk) {
                            const int c = kk / 4, ks = kk % 4;
                            tc::mma_bf16(tmem + buf * 128,
                                         tc::desc_add(da, st * 32768 + c * 16384 + ks * 32),
                                         tc::desc_add(db, c * kBChunk + ks * 32), idesc, kk > 0);
                        }
                        issued = true;
                        tc::mma_commit(&ms->a_empty[st]);
                        tc::mma_commit(&ms->acc_full[buf]);
                    }
                }
                if (stop) break;
                tc::mma_commit(&ms->b_empty);
            }
            if (issued) {
                tc::mma_commit(&ms->drain);
                if (!tc::mbar_wait(&ms->drain, 0)) cx.fail(24);
            }
        }
        __syncwarp();
    } else if (warp < 10) {
        // ================================================== epilogue warps
        // Warps 2..9: TMEM lane quarter q4 (the warp's own) and token `half`
        // of the group (its N / 2 columns).
        const int q4 = warp & 3;
        const int row = 32 * q4 + lane;
        const int ltid = tid - 64;
        const int half = (warp - 2) >> 2;
        const uint32_t lane_addr = tmem + ((uint32_t)(32 * q4) << 16);
        float *sc_smem = reinterpret_cast<float *>(smem + kOffScore);
        bulk_fill();
        uint32_t it = 0, t_n = 0, sc_n = 0;
        for (;; ++it) {
            const uint32_t slot = it % kInfoSlots;
            bool ok = cx.wait(&ms->info_full[slot], (it / kInfoSlots) & 1, 30);
            if (!bar_red_and(1, kEpiThreads, ok)) break;
            // read in place; the slot is released at the end of the group
            const GroupInfo &gi = ms->info[slot];
            if (gi.valid < 0) break;
            // the score buffer this group fills, once the selection is done
            // with the group that used it two groups ago
            const uint32_t b = sc_n & 1;
            ok = cx.wait(&ms->sc_empty[b], ((sc_n >> 1) & 1) ^ 1, 33);
            if (!bar_red_and(1, kEpiThreads, ok)) break;
            float *sc;
            int32_t sc_stride;
            if (gi.spill) {
                sc = a.scratch + ((int64_t)blockIdx.x * 2 + b) * kG * a.Tc;
                sc_stride = a.Tc;
            } else {
                sc = sc_smem + b * kG * kScoreCap;
                sc_stride = kScoreCap;
            }
            if (ltid < 2 * kG)  // key range of each token, tracked while scoring
                ms->keyrange[b][ltid >> 1][ltid & 1] = (ltid & 1) ? 0u : 0xffffffffu;
            uint32_t klo = 0xffffffffu, khi = 0u;
            // weights of the group's tokens (0 beyond Hi / T)
            for (int i = ltid; i < kG * 64; i += kEpiThreads) {
                const int g = i >> 6, h = i & 63;
                const int32_t t = gi.t0 + g;
                ms->w[i] = (h < a.Hi && t < a.T) ? __ldg(a.w + (int64_t)t * a.Hi + h) : 0.0f;
            }
            tc::named_bar_sync(1, kEpiThreads);
            bool stop = false;
            for (int p = 0; p < gi.n_pass && !stop; ++p) {
                const Pass &ps = gi.pass[p];
                for (int32_t j = 0; j < ps.n_tiles; ++j, ++t_n) {
                    const uint32_t buf = t_n % kAccBufs;
                    ok = cx.wait(&ms->acc_full[buf], (t_n / kAccBufs) & 1, 31);
                    if (!bar_red_and(1, kEpiThreads, ok)) {
                        stop = true;
                        break;
                    }
                    tc::tc_fence_after();
                    const uint32_t col0 = lane_addr + buf * 128;
                    float acc[kG];
#pragma unroll
                    for (int g = 0; g < kG; ++g) acc[g] = 0.0f;
                    if constexpr (HPAD >= 32) {
                        // this token's HPAD columns: all its 32-column chunks
                        // per tensor-memory wait, weights as float4, two
                        // partial sums
                        constexpr int kChunks = HPAD / 32;
                        float x[kChunks][32];
#pragma unroll
                        for (int cc = 0; cc < kChunks; ++cc)
                            tc::tmem_ld32(col0 + HPAD * half + 32 * cc, x[cc]);
                        tc::tmem_wait_ld();
                        float part0 = 0.0f, part1 = 0.0f;
#pragma unroll
                        for (int cc = 0; cc < kChunks; ++cc) {
                            const float4 *wv = reinterpret_cast<const float4 *>(ms->w + half * 64 + 32 * cc);
#pragma unroll
                            for (int i = 0; i < 8; ++i) {
                                const float4 w4 = wv[i];
                                const float *xi = x[cc] + 4 * i;
                                part0 = fmaf(w4.x, fmaxf(xi[0], 0.0f), part0);
                                part1 = fmaf(w4.y, fmaxf(xi[1], 0.0f), part1);
                                part0 = fmaf(w4.z, fmaxf(xi[2], 0.0f), part0);
                                part1 = fmaf(w4.w, fmaxf(xi[3], 0.0f), part1);
                            }
                        }
                        acc[half] = part0 + part1;
                    } else {
                        // fewer than 32 heads: all N (<= 32) columns from column
                        // 0; this warp keeps its token's
#pragma unroll
                        for (int cc = 0; cc < (N + 31) / 32; ++cc) {
                            float x[32];
                            tc::tmem_ld32(col0 + 32 * cc, x);
                            tc::tmem_wait_ld();
#pragma unroll
                            for (int i = 0; i < 32; ++i) {
                                const int col = 32 * cc + i;
                                if (col < N && col / HPAD == half) {
                                    const int h = col % HPAD;
                                    acc[half] = fmaf(ms->w[half * 64 + h], fmaxf(x[i], 0.0f), acc[half]);
                                }
                            }
                        }
                    }
                    tc::tc_fence_before();
                    tc::mbar_arrive(&ms->acc_empty[buf]);
                    const int32_t jl = j * kTileRows + row;
#pragma unroll
                    for (int g = 0; g < kG; ++g)
                        if (g == half && ((ps.mask >> g) & 1) && jl < gi.nv[g]) {
                            sc[(int64_t)g * sc_stride + jl] = acc[g];
                            const uint32_t u = float_key(acc[g]);
                            klo = min(klo, u);
                            khi = max(khi, u);
                        }
                }
            }
            if (stop) break;
            // scores complete: hand the buffer to the selection warps (the
            // barrier orders every epilogue thread's writes before the arrive)
            klo = __reduce_min_sync(0xffffffffu, klo);
            khi = __reduce_max_sync(0xffffffffu, khi);
            if (lane == 0) {
                atomicMin(&ms->keyrange[b][half][0], klo);
                atomicMax(&ms->keyrange[b][half][1], khi);
            }
            __threadfence_block();
            tc::named_bar_sync(1, kEpiThreads);
            if (ltid == 0) tc::mbar_arrive(&ms->sc_full[b]);
            ++sc_n;
            if (lane == 0) tc::mbar_arrive(&ms->info_empty[slot]);
        }
    } else {
        // ================================================= selection warps
        // Warps 10, 11 select token 0 of each group and 12, 13 token 1, one
        // half of the scores each (pair_topk), while the epilogue scores the
        // next group into the other buffer.
        const int sel_tok = (warp - 10) >> 1;
        const int part = (warp - 10) & 1;
        const int stid = tid - 320;
        float *sc_smem = reinterpret_cast<float *>(smem + kOffScore);
        bulk_fill();
        uint32_t it = 0, sc_n = 0;
        for (;; ++it) {
            const uint32_t slot = it % kInfoSlots;
            bool ok = cx.wait(&ms->info_full[slot], (it / kInfoSlots) & 1, 34);
            if (!bar_red_and(7, kSelThreads, ok)) break;
            const GroupInfo &gi = ms->info[slot];
            if (gi.valid < 0) break;
            const uint32_t b = sc_n & 1;
            ok = cx.wait(&ms->sc_full[b], (sc_n >> 1) & 1, 35);
            if (!bar_red_and(7, kSelThreads, ok)) break;
            const float *sc;
            int32_t sc_stride;
            if (gi.spill) {
                sc = a.scratch + ((int64_t)blockIdx.x * 2 + b) * kG * a.Tc;
                sc_stride = a.Tc;
            } else {
                sc = sc_smem + b * kG * kScoreCap;
                sc_stride = kScoreCap;
            }
            const int g = sel_tok;
            const int32_t t = gi.t0 + g;
            if (t < a.T) {
                int32_t *idx_row = a.topk_idx + (int64_t)t * a.topk;
                float *val_row = a.topk_val ? a.topk_val + (int64_t)t * a.topk : nullptr;
                const int32_t n = gi.valid ? gi.nv[g] : 0;
                const uint32_t lo = ms->keyrange[b][g][0], hi = ms->keyrange[b][g][1];
                if (gi.spill)
                    pair_topk<false>(sc + (int64_t)g * sc_stride, n, a.topk, gi.cb[g], idx_row,
                                     val_row, ms->hist[g], lo, hi, part, lane, 2 + g, a.pair_max);
                else
                    pair_topk<true>(sc + (int64_t)g * sc_stride, n, a.topk, gi.cb[g], idx_row,
                                    val_row, ms->hist[g], lo, hi, part, lane, 2 + g, a.pair_max);
            }
            // the buffer is free for the epilogue's group after next
            tc::named_bar_sync(7, kSelThreads);
            if (stid == 0) tc::mbar_arrive(&ms->sc_empty[b]);
            ++sc_n;
            if (lane == 0) tc::mbar_arrive(&ms->info_empty[slot]);
        }
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    if (warp == 1) tc::tmem_dealloc(tmem, 512);
}

template <int HPAD, int DI>
cudaError_t launch_t(const IndexerArgs &a, const CUtensorMap &qm, const CUtensorMap &km, int ctas,
                     cudaStream_t stream) {
    cudaError_t e = cudaFuncSetAttribute(indexer_tc_kernel<HPAD, DI>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    return launch_early(indexer_tc_kernel<HPAD, DI>, dim3(ctas), dim3(kThreads), kSmemBytes, stream,
                        qm, km, a);
}

template <int DI>
cudaError_t launch_di(const IndexerArgs &a, int hpad, const CUtensorMap &qm, const CUtensorMap &km,
                      int ctas, cudaStream_t stream) {
    switch (hpad) {
        case 4: return launch_t<4, DI>(a, qm, km, ctas, stream);
        case 8: return launch_t<8, DI>(a, qm, km, ctas, stream);
        case 16: return launch_t<16, DI>(a, qm, km, ctas, stream);
        case 32: return launch_t<32, DI>(a, qm, km, ctas, stream);
        default: return launch_t<64, DI>(a, qm, km, ctas, stream);
    }
}

}  // namespace

int32_t indexer_scratch_rows_threshold() { return kScoreCap; }

// two score buffers of kG tokens (one being scored, one being selected)
int64_t indexer_scratch_floats_per_cta(int32_t Tc) { return 2 * (int64_t)kG * Tc; }

size_t indexer_workspace_bytes(int32_t T, int32_t Tc, int32_t, int32_t, int32_t) {
    if (Tc <= kScoreCap || T <= 0) return 0;
    const int64_t groups = ((int64_t)T + kG - 1) / kG;
    const int64_t ctas = groups < kMaxCtas ? groups : kMaxCtas;
    return (size_t)ctas * (size_t)indexer_scratch_floats_per_cta(Tc) * sizeof(float);
}

cudaError_t launch_indexer_topk(const IndexerArgs &args, cudaStream_t stream) {
    if (args.T == 0) return cudaSuccess;
    IndexerArgs a = args;
    a.wait_ns = pipeline_wait_limit_ns();
    a.pair_max = pair_select_max_rows(kPairMax);
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    const int32_t groups = (a.T + kG - 1) / kG;
    int ctas = groups < sms ? groups : sms;
    if (ctas > kMaxCtas) ctas = kMaxCtas;
    if (a.max_ctas > 0 && ctas > a.max_ctas) ctas = a.max_ctas;
    const int hpad = a.Hi <= 4 ? 4 : a.Hi <= 8 ? 8 : a.Hi <= 16 ? 16 : a.Hi <= 32 ? 32 : 64;
    CUtensorMap qm, km;
    // q viewed as [T][Hi][Di]; a box of (64 dims, hpad heads, kG tokens) zero-fills
    // heads >= Hi and tokens >= T.
    if (!encode_bf16_3d(&qm, a.q, a.Di, a.Hi, a.T, 64, hpad, kG)) return cudaErrorInvalidValue;
    if (a.Tc > 0) {
        if (!encode_bf16_2d(&km, a.k, a.Tc, a.Di, 64, kTileRows)) return cudaErrorInvalidValue;
    } else {
        km = qm;  // never read: no token has a visible row
    }
    return a.Di == 64 ? launch_di<64>(a, hpad, qm, km, ctas, stream)
                      : launch_di<128>(a, hpad, qm, km, ctas, stream);
}

}  // namespace csa
