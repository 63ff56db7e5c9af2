// M = 1 GEMV on CUDA cores: y[n] = fp16( sum_k x[k] * W[n][k] ), FP32 accumulation
// (and the same with bf16 operands and output).
//
// The shape reads each W element exactly once (117,440,512 of the 117,477,376
// algorithmic bytes at N = 4096, K = 14336), so the bound is HBM bandwidth, not
// arithmetic ("Learning TileLang with GEMV", §02 Bandwidth Bound).  The page's
// rules for a bandwidth-bound kernel (§07 Summary) decide the design:
//   - enough independent work: one warp per output row gives N warps (4096 at
//     the Llama-3-8B down-projection shape, about 27 per SM), all resident at
//     once, so every warp gets the same HBM share and no SM tail remains;
//   - coalesced: at every step the 32 lanes of a warp read 32 adjacent 16-byte
//     chunks of the row, 512 contiguous bytes (§4.3 Coalescing);
//   - wide: every load is 128 bits = 8 fp16 (§4.5 thread_vectorized_split_k).
// What the page leaves implicit, and what sets the achieved bandwidth here, is
// the number of bytes in flight per SM (HBM latency x per-SM bandwidth, about
// 40 KB).  Each lane keeps two groups of GROUP 16-byte loads in flight: the
// loads of group g+1 are issued before group g is consumed (explicit double
// buffering), so a warp always has 4-8 KB outstanding.
// The per-lane FP32 partial sums are combined with warp shuffles (§4.6
// Reduction: thread all-reduce lowered to shuffles) and y[n] is written once
// with cvt.rn.  W is streamed with L1::no_allocate so it does not evict x,
// which every warp re-reads from L1.  No atomics: results are deterministic.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "launch.h"
#include "ptx.cuh"

namespace tmagemm {

namespace {

constexpr int kGvWarps = 8;      // rows per block
constexpr int kGvGroup = 4;      // 16-byte loads per lane per group
#ifndef TMAGEMM_GV_PREFETCH_CHUNKS
#define TMAGEMM_GV_PREFETCH_CHUNKS 256
#endif
// 16-byte chunks at the head of each row warmed in L2 before the wait (4 KB).
constexpr int32_t kGvPrefetchChunks = TMAGEMM_GV_PREFETCH_CHUNKS;

__device__ __forceinline__ uint4 ld_stream_v4(const uint4* p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

// Two packed 16-bit values -> two floats (exact for fp16 and bf16).
template <bool BF16>
__device__ __forceinline__ float2 unpack2(uint32_t v) {
    if constexpr (BF16)
        return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&v));
    else
        return __half22float2(*reinterpret_cast<const __half2*>(&v));
}

template <bool BF16>
__device__ __forceinline__ float dot8(const uint4& w, const uint4& x, float acc) {
    const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
    const uint32_t xv[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 wf = unpack2<BF16>(wv[i]);
        const float2 xf = unpack2<BF16>(xv[i]);
        acc = fmaf(wf.x, xf.x, acc);
        acc = fmaf(wf.y, xf.y, acc);
    }
    return acc;
}

// This lane's chunks idx0 + 32*u, u < GROUP.
__device__ __forceinline__ void load_group(const uint4* wrow, int32_t idx0, uint4 (&w)[kGvGroup]) {
#pragma unroll
    for (int u = 0; u < kGvGroup; ++u) w[u] = ld_stream_v4(wrow + idx0 + 32 * u);
}

template <bool BF16>
__device__ __forceinline__ void consume_group(const uint4* __restrict__ x, int32_t idx0,
                                              const uint4 (&w)[kGvGroup], float (&acc)[kGvGroup]) {
#pragma unroll
    for (int u = 0; u < kGvGroup; ++u) acc[u] = dot8<BF16>(w[u], __ldg(x + idx0 + 32 * u), acc[u]);
}

template <bool BF16>
__global__ void __launch_bounds__(kGvWarps * 32)
gemv_f16_kernel(const uint4* __restrict__ x, const uint4* __restrict__ W, uint16_t* __restrict__ y,
                int32_t N, int32_t K8, uint32_t* __restrict__ err) {
    // Every block of this grid is resident by the time all have issued this,
    // so the next grid may be scheduled; it waits for this one to finish.
    grid_launch_dependents();
    const int lane = threadIdx.x & 31;
    const int32_t n = blockIdx.x * kGvWarps + (threadIdx.x >> 5);
    if (n >= N) return;
    const uint4* wrow = W + static_cast<int64_t>(n) * K8;
    // While the previous grid finishes, pull the head of this row into L2 (a
    // prefetch cannot see stale data: L2 is where global memory is coherent),
    // so the first loads after the wait hit L2 instead of HBM.
    if (kGvPrefetchChunks > 0 && lane == 0)
        prefetch_l2_bytes(wrow, static_cast<uint32_t>(min(K8, kGvPrefetchChunks)) * 16u);
    grid_dependency_wait();   // x and W may come from the grid before this one
    float acc[kGvGroup] = {};
    // Whole groups: group g covers this lane's chunks lane + 32*(g*GROUP + u).
    constexpr int32_t kStep = 32 * kGvGroup;
    const int32_t groups = K8 / kStep;
    uint4 wa[kGvGroup], wb[kGvGroup];
    if (groups > 0) load_group(wrow, lane, wa);
    for (int32_t g = 0; g < groups; g += 2) {
        const int32_t ia = lane + g * kStep;
        const int32_t ib = ia + kStep;
        if (g + 1 < groups) load_group(wrow, ib, wb);
        consume_group<BF16>(x, ia, wa, acc);
        if (g + 2 < groups) load_group(wrow, ib + kStep, wa);
        if (g + 1 < groups) consume_group<BF16>(x, ib, wb, acc);
    }
    // Tail: the remaining (< 32 * GROUP) chunks, one per lane per step.
    for (int32_t idx = groups * kStep + lane; idx < K8; idx += 32)
        acc[0] = dot8<BF16>(ld_stream_v4(wrow + idx), __ldg(x + idx), acc[0]);
    float s = acc[0];
#pragma unroll
    for (int u = 1; u < kGvGroup; ++u) s += acc[u];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    if (lane == 0) {
        if constexpr (BF16)
            y[n] = __bfloat16_as_ushort(__float2bfloat16_rn(s));
        else
            y[n] = __half_as_ushort(__float2half_rn(s));
        check_count_unit(err, n);   // checked build: output rows written
    }
}

}  // namespace

cudaError_t launch_gemv(int64_t N, int64_t K, const void* x, const void* W, void* y, bool bf16,
                        cudaStream_t stream, uint32_t* err, bool pdl) {
    const int32_t K8 = static_cast<int32_t>(K / 8);
    const int64_t blocks = (N + kGvWarps - 1) / kGvWarps;
    auto kernel = bf16 ? gemv_f16_kernel<true> : gemv_f16_kernel<false>;
    return launch_kernel(kernel, dim3(static_cast<unsigned>(blocks)), dim3(kGvWarps * 32), 0,
                         stream, 1u, pdl, static_cast<const uint4*>(x), static_cast<const uint4*>(W),
                         static_cast<uint16_t*>(y), static_cast<int32_t>(N), K8, err);
}

}  // namespace tmagemm
