// Internal helpers shared by the CSA kernels (sm_103a only).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "csa.h"

namespace csa {

// ---------------------------------------------------------------------------
// Device error word. Kernels never trap: an inconsistency in device data, or a
// bounded wait that gave up, is recorded here (first writer wins) and the
// kernel skips the offending work. csa_device_error() reads and clears it.
// Layout: kind << 24 | kernel << 16 | site.
// ---------------------------------------------------------------------------
enum ErrKind : int32_t { kErrCheck = 1, kErrTimeout = 2 };
enum KernelId : int32_t {
    kKerCompress = 1,
    kKerWindow = 2,
    kKerIndexer = 3,
    kKerMla = 4,
    kKerMlaBwd = 5,
    kKerIndexerKl = 6,
    kKerBsnd = 7,
    kKerCompressor = 8,
};

__device__ __forceinline__ void report_error(int32_t *err, int32_t kind, int32_t kernel,
                                             int32_t site) {
    if (err) atomicCAS(err, 0, (kind << 24) | (kernel << 16) | (site & 0xffff));
}

// Sequence owning packed row t: the b in [0, batch) with cu[b] <= t < cu[b+1]
// (empty sequences are skipped). -1 when t is not covered.
__device__ __forceinline__ int32_t find_segment(const int32_t *__restrict__ cu, int32_t batch,
                                                int32_t t) {
    int32_t lo = 0, hi = batch;  // search the last b in [0, batch] with cu[b] <= t
    if (batch <= 0 || t < __ldg(cu)) return -1;
    while (lo < hi) {
        int32_t mid = (lo + hi + 1) >> 1;
        if (__ldg(cu + mid) <= t) lo = mid;
        else hi = mid - 1;
    }
    if (lo >= batch || __ldg(cu + lo + 1) <= t) return -1;
    return lo;
}

// The same lookup over offsets already staged in shared memory.
__device__ __forceinline__ int32_t find_segment_smem(const int32_t *cu, int32_t batch, int32_t t) {
    int32_t lo = 0, hi = batch;
    if (batch <= 0 || t < cu[0]) return -1;
    while (lo < hi) {
        int32_t mid = (lo + hi + 1) >> 1;
        if (cu[mid] <= t) lo = mid;
        else hi = mid - 1;
    }
    if (lo >= batch || cu[lo + 1] <= t) return -1;
    return lo;
}

// Order-preserving map fp32 -> uint32 (larger float -> larger key); -0 maps
// like +0 so that equal scores are equal keys.
__device__ __forceinline__ uint32_t float_key(float s) {
    uint32_t u = __float_as_uint(s + 0.0f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ int32_t warp_sum_i(int32_t v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Exclusive prefix sum of one int per thread over a block of NT threads.
// `scratch` holds at least NT/32 + 1 ints of shared memory; returns the
// block total through *total. Contains __syncthreads().
template <int NT>
__device__ __forceinline__ int32_t block_exclusive_scan(int32_t v, int32_t *scratch,
                                                        int32_t *total) {
    static_assert(NT % 32 == 0 && NT <= 1024, "block size");
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int32_t x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int32_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) scratch[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int32_t w = lane < NT / 32 ? scratch[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int32_t y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        if (lane < NT / 32) scratch[lane] = w;  // inclusive warp totals
        if (lane == NT / 32 - 1) scratch[NT / 32] = w;
    }
    __syncthreads();
    int32_t before = (warp > 0 ? scratch[warp - 1] : 0) + x - v;
    *total = scratch[NT / 32];
    __syncthreads();
    return before;
}

// ---------------------------------------------------------------------------
// Programmatic dependent launch. The forward kernels are launched so that they
// may start while the kernel before them on the stream finishes: each one does
// its purely local set-up (barriers, tensor memory, shared memory), then waits
// here for the grids it depends on to complete with their memory visible,
// before its first global read or write. For a launch that did not start early
// the wait returns at once.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void grid_dependency_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Lets the next kernel on the stream (if launched the same way) be scheduled;
// its CTAs still wait in grid_dependency_wait until this grid has completed.
__device__ __forceinline__ void launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Launch with programmatic stream serialization (see grid_dependency_wait).
template <typename... KArgs, typename... Args>
cudaError_t launch_early(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                         cudaStream_t stream, Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

}  // namespace csa
