// THD compressor core (sm_103a): grouping, position embedding, overlap
// transform and slot pooling of one DeepSeek-V4 compressor.
//
// The miles PR 2038 report (compressor.py, _forward_thd and
// _overlap_transform_thd) groups the rows of each packed sequence: compressed
// row g = cu_c[b] + j takes rows cu[b] + j r + i (i < r) of the two
// projections kv = x W_kv^T and score = x W_gate^T; with overlap, each group
// becomes 2r slots of head_dim -- the first halves of the previous group's
// rows (missing for a sequence's first group: kv 0, score -inf) and the
// second halves of its own rows. The page omits what follows; the -inf fill
// of the score only means something as a softmax logit, so the reading here
// is the softmax over the slots, per dimension, weighting kv, with the
// position embedding ape[i] added to the score of slot i before the overlap.
//
// Design. The usual case (head_dim a multiple of 4, 16-byte aligned arrays)
// runs compress_thd_vec_kernel: a block covers 128 dimensions of one
// compressed row, each of its 32 lanes 4 consecutive dimensions, and S = 1,
// 2 or 4 thread rows split the group's slots (4 for the few long groups of a
// large ratio: 225 groups of 256 slots on the mixed 32k pack at ratio 128;
// with fewer rows a block covers 4 / S groups).
// Each thread streams its slots' 16-byte pieces into shared memory with
// cp.async, a few slots ahead of the ones it pools into an fp32 online softmax
// (running max, rescaled sum and weighted sum); thread row 0 merges the S
// partial results in a fixed order, so the output does not depend on timing.
// Every input element is read once (a row's first half by the next group,
// its second half by its own group): the kernel is HBM-bound on the grouped
// rows of both projections plus the output. Other shapes run
// compress_thd_kernel, one thread per (compressed row, dimension).
#include "common.cuh"
#include "internal.h"

namespace csa {

namespace {

constexpr int kCmpThreads = 128;

__device__ __forceinline__ void pool_slot(float s, float v, float &m, float &z, float &acc) {
    if (s > m) {
        const float c = expf(m - s);  // 0 while m is still -inf
        z = z * c + 1.0f;
        acc = acc * c + v;
        m = s;
    } else {
        const float p = expf(s - m);
        z += p;
        acc = fmaf(p, v, acc);
    }
}

// Thread (0, 0) of a block finds the sequence of compressed row g and checks
// that the group's rows lie inside it: info = {segment or -1, the sequence's
// first packed row, j = g's index in the sequence}.
__device__ __forceinline__ void group_info(const CompressArgs &a, int32_t g, int32_t *info) {
    const int32_t b = find_segment(a.cu_c, a.batch, g);
    info[0] = b;
    if (b >= 0) {
        info[1] = __ldg(a.cu_q + b);
        info[2] = g - __ldg(a.cu_c + b);
        const int64_t last = (int64_t)info[1] + ((int64_t)info[2] + 1) * a.r - 1;
        if (last >= __ldg(a.cu_q + b + 1) || last >= a.T) info[0] = -1;
    }
    if (info[0] < 0) report_error(a.err, kErrCheck, kKerCompressor, 1);
}

// The same from offsets staged in shared memory (cu_c, then cu_q).
__device__ __forceinline__ void group_info_staged(const CompressArgs &a, const int32_t *cc,
                                                  const int32_t *cq, int32_t g, int32_t *info) {
    const int32_t b = find_segment_smem(cc, a.batch, g);
    info[0] = b;
    if (b >= 0) {
        info[1] = cq[b];
        info[2] = g - cc[b];
        const int64_t last = (int64_t)info[1] + ((int64_t)info[2] + 1) * a.r - 1;
        if (last >= cq[b + 1] || last >= a.T) info[0] = -1;
    }
    if (info[0] < 0) report_error(a.err, kErrCheck, kKerCompressor, 1);
}

__global__ void __launch_bounds__(kCmpThreads) compress_thd_kernel(CompressArgs a) {
    __shared__ int32_t info[3];  // segment, its first packed row, j (group index in it)
    const int32_t g = blockIdx.x;
    if (threadIdx.x == 0) group_info(a, g, info);
    __syncthreads();
    const int32_t e = blockIdx.y * kCmpThreads + threadIdx.x;
    if (e >= a.hd) return;
    float *dst = a.out + (int64_t)g * a.hd + e;
    if (info[0] < 0) {
        *dst = 0.0f;
        return;
    }
    const int64_t wd = a.overlap ? 2 * (int64_t)a.hd : a.hd;
    const int64_t first = (int64_t)info[1] + (int64_t)info[2] * a.r;  // own group's first row
    const bool has_prev = a.overlap && info[2] > 0;
    const int64_t own_col = a.overlap ? a.hd + e : e;
    float m = -INFINITY, z = 0.0f, acc = 0.0f;
    for (int32_t i = 0; i < a.r; ++i) {
        if (has_prev) {
            const int64_t row = first - a.r + i;
            const float s = __ldg(a.score + row * wd + e) + (a.ape ? __ldg(a.ape + i * wd + e) : 0.0f);
            pool_slot(s, __ldg(a.kv + row * wd + e), m, z, acc);
        }
        const int64_t row = first + i;
        const float s = __ldg(a.score + row * wd + own_col) +
                        (a.ape ? __ldg(a.ape + i * wd + own_col) : 0.0f);
        pool_slot(s, __ldg(a.kv + row * wd + own_col), m, z, acc);
    }
    *dst = acc / z;
}

// 2^x (the hardware approximation: relative error about 2^-22; 2^-inf = 0).
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Merge a partial result (m2, z2, a2) into (m, z, acc); maxima in log2 units.
__device__ __forceinline__ void merge_partial(float m2, float z2, float a2, float &m, float &z,
                                              float &acc) {
    if (m2 == -INFINITY) return;  // that thread row held no slot
    const float mn = fmaxf(m, m2);
    const float c = ex2(m - mn), c2 = ex2(m2 - mn);
    z = z * c + z2 * c2;
    acc = acc * c + a2 * c2;
    m = mn;
}

// 16-byte copy global -> shared that bypasses L1 and registers.
__device__ __forceinline__ void cp_async16(void *dst, const float *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(
                     (uint32_t)__cvta_generic_to_shared(dst)),
                 "l"(src)
                 : "memory");
}

__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}

// Wait until at most N of this thread's copy groups are still in flight.
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

constexpr int kVecLanes = 32;  // threads along dimensions: 4 each, 128 per block
constexpr int kStages = 3;     // chunks of slots each thread has in its ring
constexpr int kChunk = 2;      // slots per chunk
// the ring when it also carries the position embedding
constexpr int kStages3 = 2, kChunk3 = 1;
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kStagedCu = 256;  // sequences + 1 staged in shared memory

// Block (32, S, G): 128 dimensions (blockIdx.y) of G consecutive compressed
// rows (z), thread row y taking the slots y, y + S, ... of its row. Each
// thread streams its slots' 16-byte pieces (score and kv, and with J = 3 the
// position embedding; with J = 2 that small table is read through the cache)
// through a ring of NS chunks of NC slots in shared memory with
// cp.async, so that NS - 1 chunks stay in flight while it pools the
// current one; a thread reads only what it copied itself, so the ring needs
// no barrier. Pooling works in base 2 on scores scaled by log2(e) (the same
// weights), one rescale per chunk. Thread row 0 then merges rows 1 .. S-1 in
// order.
template <int S, int G, int J>
__global__ void __launch_bounds__(kVecLanes * S * G) compress_thd_vec_kernel(CompressArgs a) {
    constexpr int X = kVecLanes;
    constexpr int NS = J == 3 ? kStages3 : kStages, NC = J == 3 ? kChunk3 : kChunk;
    __shared__ int32_t info[G][3];
    // ring[k][u][j][z][y][x]: stage k, slot u of the chunk, piece j, thread
    // (x, y, z); after the loop, rows 1 .. S-1 leave (m, z, acc) in its first
    // entries
    __shared__ float4 ring[NS * NC * J * G * S * X];
    // sequence offsets, staged by all threads at once when there are few
    // sequences (one load latency instead of a search's chain of loads)
    __shared__ int32_t cu_s[2][kStagedCu];
    const int x = threadIdx.x, y = threadIdx.y, zz = threadIdx.z;
    const int32_t g = blockIdx.x * G + zz;
    const bool has_row = g < a.Tc;
    const bool staged = a.batch < kStagedCu;
    if (staged) {
        const int tid = (zz * S + y) * X + x;
        for (int i = tid; i <= a.batch; i += X * S * G) {
            cu_s[0][i] = __ldg(a.cu_c + i);
            cu_s[1][i] = __ldg(a.cu_q + i);
        }
        __syncthreads();
    }
    if (x == 0 && y == 0 && has_row) {
        if (staged)
            group_info_staged(a, cu_s[0], cu_s[1], g, info[zz]);
        else
            group_info(a, g, info[zz]);
    }
    __syncthreads();
    const int32_t e = blockIdx.y * 4 * X + 4 * x;  // this thread's first dimension
    const bool live = has_row && e < a.hd;          // head_dim is a multiple of 4
    float4 m4 = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
    float4 z4 = make_float4(0.f, 0.f, 0.f, 0.f), a4 = z4;
    if (live && info[zz][0] >= 0) {
        const int32_t *gi = info[zz];
        const int64_t wd = a.overlap ? 2 * (int64_t)a.hd : a.hd;
        const int64_t first = (int64_t)gi[1] + (int64_t)gi[2] * a.r;  // own first row
        // Slots q of the group: with a previous group, q < r are its rows (first
        // half of each row), then the own rows (second half); else own rows only.
        const int32_t prev = (a.overlap && gi[2] > 0) ? a.r : 0;
        const int32_t n = prev + a.r;
        const int32_t mine = y < n ? (n - y + S - 1) / S : 0;  // slots of this thread row
        const int32_t chunks = (mine + NC - 1) / NC;
        const int32_t own_col = a.overlap ? a.hd + e : e;
        // element offsets of slot index 0 of the previous and of the own rows
        const int64_t off_p = (first - a.r) * wd + e, off_o = first * wd + own_col;
        const float *const ape = a.ape;
        auto piece = [&](int k, int u, int j) -> float4 * {
            return ring + ((((k * NC + u) * J + j) * G + zz) * S + y) * X + x;
        };
        // thread slot i: offset of its row piece and of its embedding entry
        auto where = [&](int32_t i, int64_t &o, int64_t &ao) {
            const int32_t q = y + i * S;
            const bool own = q >= prev;
            const int64_t sw = (int64_t)(own ? q - prev : q) * wd;
            o = (own ? off_o : off_p) + sw;
            ao = sw + (own ? own_col : e);
        };
        auto issue = [&](int32_t c) {  // chunk c into stage c % NS
            const int k = c % NS;
#pragma unroll
            for (int u = 0; u < NC; ++u) {
                const int32_t i = c * NC + u;
                if (i >= mine) break;
                int64_t o, ao;
                where(i, o, ao);
                cp_async16(piece(k, u, 0), a.score + o);
                cp_async16(piece(k, u, 1), a.kv + o);
                if (J == 3) cp_async16(piece(k, u, 2), ape + ao);
            }
        };
#pragma unroll
        for (int c = 0; c < NS - 1; ++c) {
            if (c < chunks) issue(c);
            cp_async_commit();  // empty groups keep the count uniform
        }
        for (int32_t c = 0; c < chunks; ++c) {
            if (c + NS - 1 < chunks) issue(c + NS - 1);
            cp_async_commit();
            cp_async_wait<NS - 1>();  // chunk c has landed
            const int k = c % NS;
            float4 sc[NC], v[NC];
            float4 mn = m4;
#pragma unroll
            for (int u = 0; u < NC; ++u) {
                if (c * NC + u < mine) {
                    sc[u] = *piece(k, u, 0);
                    v[u] = *piece(k, u, 1);
                    if (ape) {
                        float4 p;
                        if (J == 3) {
                            p = *piece(k, u, 2);
                        } else {
                            int64_t o, ao;
                            where(c * NC + u, o, ao);
                            p = __ldg(reinterpret_cast<const float4 *>(ape + ao));
                        }
                        sc[u].x += p.x, sc[u].y += p.y, sc[u].z += p.z, sc[u].w += p.w;
                    }
                    sc[u].x *= kLog2e, sc[u].y *= kLog2e, sc[u].z *= kLog2e, sc[u].w *= kLog2e;
                } else {
                    sc[u] = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
                    v[u] = make_float4(0.f, 0.f, 0.f, 0.f);
                }
                mn.x = fmaxf(mn.x, sc[u].x), mn.y = fmaxf(mn.y, sc[u].y);
                mn.z = fmaxf(mn.z, sc[u].z), mn.w = fmaxf(mn.w, sc[u].w);
            }
            // 0 while the running max is still -inf; the chunk's first slot is real
            const float4 cr = make_float4(ex2(m4.x - mn.x), ex2(m4.y - mn.y),
                                          ex2(m4.z - mn.z), ex2(m4.w - mn.w));
            z4.x *= cr.x, z4.y *= cr.y, z4.z *= cr.z, z4.w *= cr.w;
            a4.x *= cr.x, a4.y *= cr.y, a4.z *= cr.z, a4.w *= cr.w;
#pragma unroll
            for (int u = 0; u < NC; ++u) {
                const float px = ex2(sc[u].x - mn.x), py = ex2(sc[u].y - mn.y);
                const float pz = ex2(sc[u].z - mn.z), pw = ex2(sc[u].w - mn.w);
                z4.x += px, z4.y += py, z4.z += pz, z4.w += pw;
                a4.x = fmaf(px, v[u].x, a4.x), a4.y = fmaf(py, v[u].y, a4.y);
                a4.z = fmaf(pz, v[u].z, a4.z), a4.w = fmaf(pw, v[u].w, a4.w);
            }
            m4 = mn;
        }
        cp_async_wait<0>();
    }
    if (S > 1) {
        __syncthreads();  // every thread's copies are done: the ring is free
        float4 *const part = ring;  // [3][S-1][G][X]
        auto at = [&](int j, int row) { return part + ((j * (S - 1) + row - 1) * G + zz) * X + x; };
        if (y > 0) *at(0, y) = m4, *at(1, y) = z4, *at(2, y) = a4;
        __syncthreads();
        if (y > 0) return;
        for (int k = 1; k < S; ++k) {
            const float4 m2 = *at(0, k), z2 = *at(1, k), a2 = *at(2, k);
            merge_partial(m2.x, z2.x, a2.x, m4.x, z4.x, a4.x);
            merge_partial(m2.y, z2.y, a2.y, m4.y, z4.y, a4.y);
            merge_partial(m2.z, z2.z, a2.z, m4.z, z4.z, a4.z);
            merge_partial(m2.w, z2.w, a2.w, m4.w, z4.w, a4.w);
        }
    }
    if (!live) return;
    float4 *dst = reinterpret_cast<float4 *>(a.out + (int64_t)g * a.hd + e);
    if (info[zz][0] < 0) {
        *dst = make_float4(0.f, 0.f, 0.f, 0.f);
        return;
    }
    *dst = make_float4(a4.x / z4.x, a4.y / z4.y, a4.z / z4.z, a4.w / z4.w);
}

template <int S, int G, int J>
cudaError_t launch_vec(const CompressArgs &a, cudaStream_t stream) {
    const dim3 grid((unsigned)((a.Tc + G - 1) / G),
                    (unsigned)((a.hd + 4 * kVecLanes - 1) / (4 * kVecLanes)));
    compress_thd_vec_kernel<S, G, J><<<grid, dim3(kVecLanes, S, G), 0, stream>>>(a);
    return cudaGetLastError();
}

template <int J>
cudaError_t launch_vec_rows(const CompressArgs &a, int s, cudaStream_t stream) {
    switch (s) {
        case 1: return launch_vec<1, 4, J>(a, stream);
        case 2: return launch_vec<2, 2, J>(a, stream);
        default: return launch_vec<4, 1, J>(a, stream);
    }
}

bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

}  // namespace

cudaError_t launch_compress_thd(const CompressArgs &a, cudaStream_t stream) {
    if (a.Tc == 0) return cudaSuccess;
    if (a.hd % 4 == 0 && aligned16(a.kv) && aligned16(a.score) && aligned16(a.out) &&
        (a.ape == nullptr || aligned16(a.ape))) {
        int dev = 0, sms = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return e;
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        const int64_t cols = (int64_t)a.Tc * ((a.hd + 4 * kVecLanes - 1) / (4 * kVecLanes));
        const int32_t slots = (a.overlap ? 2 : 1) * a.r;  // most slots of a group
        // One thread row per group while the groups alone give the grid half of
        // the threads the SMs keep resident; more rows (up to 4) for few long
        // groups (a large ratio on a short pack), each keeping a chunk or more.
        int s = 1;
        while (s < 4 && 2 * kChunk * s <= slots && cols * kVecLanes * s < (int64_t)sms * 1024)
            s *= 2;
        // The position embedding goes through the ring too once it is too large
        // to stay in the L1 cache beside the rings (r * wd * 4 bytes).
        const int64_t wd = a.overlap ? 2 * (int64_t)a.hd : a.hd;
        const bool ape_ring = a.ape != nullptr && (int64_t)a.r * wd * 4 > (64 << 10);
        return ape_ring ? launch_vec_rows<3>(a, s, stream) : launch_vec_rows<2>(a, s, stream);
    }
    const dim3 grid((unsigned)a.Tc, (unsigned)((a.hd + kCmpThreads - 1) / kCmpThreads));
    compress_thd_kernel<<<grid, kCmpThreads, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace csa
