// M = 1 GEMV on CUDA cores: y[n] = fp16( sum_k x[k] * W[n][k] ), FP32 accumulation.
//
// The shape reads each W element exactly once (117,440,512 of the 117,477,376
// algorithmic bytes at N = 4096, K = 14336), so the bound is HBM bandwidth, not
// arithmetic ("Learning TileLang with GEMV", §02 Bandwidth Bound).  Following
// the page's lessons for bandwidth-bound kernels (§07 Summary):
//   - each output row is owned by one warp, so there are N warps in flight;
//   - at every step the 32 lanes of a warp read 32 adjacent 16-byte chunks of
//     the row: fully coalesced, 512 contiguous bytes (§4.3 Coalescing);
//   - every load is 128 bits = 8 fp16 (§4.5 thread_vectorized_split_k), and
//     UNROLL independent loads per lane are issued before any is consumed, to
//     keep enough bytes in flight per SM to cover HBM latency;
//   - the per-lane partial sums are combined with warp shuffles
//     (§4.6 Reduction: thread all-reduce lowered to shuffles).
// W is streamed with L1::no_allocate so it does not evict x, which every warp
// re-reads from L1.
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "launch.h"

namespace tmagemm {

namespace {

constexpr int kGemvWarps = 4;     // rows per block
constexpr int kGemvUnroll = 8;    // 16-byte loads in flight per lane

__device__ __forceinline__ uint4 ld_stream_v4(const uint4* p) {
    uint4 r;
    asm("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

__device__ __forceinline__ float dot8(const uint4& w, const uint4& x, float acc) {
    const __half2* wh = reinterpret_cast<const __half2*>(&w);
    const __half2* xh = reinterpret_cast<const __half2*>(&x);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 wf = __half22float2(wh[i]);
        const float2 xf = __half22float2(xh[i]);
        acc = fmaf(wf.x, xf.x, acc);
        acc = fmaf(wf.y, xf.y, acc);
    }
    return acc;
}

template <int WARPS, int UNROLL>
__global__ void __launch_bounds__(WARPS * 32)
gemv_f16_kernel(const uint4* __restrict__ x, const uint4* __restrict__ W, __half* __restrict__ y,
                int32_t N, int32_t K8) {
    const int lane = threadIdx.x & 31;
    const int32_t n = blockIdx.x * WARPS + (threadIdx.x >> 5);
    if (n >= N) return;
    const uint4* wrow = W + static_cast<int64_t>(n) * K8;
    float acc = 0.f;
    // Main part: whole groups of 32 * UNROLL chunks, no predicates.
    const int32_t k_main = (K8 / (32 * UNROLL)) * (32 * UNROLL);
    for (int32_t base = lane; base < k_main; base += 32 * UNROLL) {
        uint4 wv[UNROLL], xv[UNROLL];
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) wv[u] = ld_stream_v4(wrow + base + 32 * u);
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) xv[u] = __ldg(x + base + 32 * u);
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) acc = dot8(wv[u], xv[u], acc);
    }
    // Tail: the remaining (< 32 * UNROLL) chunks, one per lane per step.
    for (int32_t idx = k_main + lane; idx < K8; idx += 32)
        acc = dot8(ld_stream_v4(wrow + idx), __ldg(x + idx), acc);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (lane == 0) y[n] = __float2half_rn(acc);
}

}  // namespace

cudaError_t launch_gemv(int64_t N, int64_t K, const void* x, const void* W, void* y,
                        cudaStream_t stream) {
    const int32_t K8 = static_cast<int32_t>(K / 8);
    const int64_t blocks = (N + kGemvWarps - 1) / kGemvWarps;
    gemv_f16_kernel<kGemvWarps, kGemvUnroll><<<static_cast<unsigned>(blocks), kGemvWarps * 32, 0,
                                               stream>>>(
        static_cast<const uint4*>(x), static_cast<const uint4*>(W), static_cast<__half*>(y),
        static_cast<int32_t>(N), K8);
    return cudaGetLastError();
}

}  // namespace tmagemm
