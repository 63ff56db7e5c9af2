// M = 1 GEMV on CUDA cores: y[n] = fp16( sum_k x[k] * W[n][k] ), FP32 accumulation
// (and the same with bf16 operands and output).
//
// The shape reads each W element exactly once (117,440,512 of the 117,477,376
// algorithmic bytes at N = 4096, K = 14336), so the bound is HBM bandwidth, not
// arithmetic ("Learning TileLang with GEMV", §02 Bandwidth Bound).  The page's
// rules for a bandwidth-bound kernel (§07 Summary) decide the design:
//   - enough independent work: N rows of K / 8 independent 16-byte loads
//     (4096 rows of 1792 at the Llama-3-8B down-projection shape), spread over
//     every SM at once;
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
//
// Two kernels share these rules.  gemv_pieces_kernel (the default wherever a
// CTA's rows and a row's pieces fit its shared-memory table): one CTA per SM
// takes N / SMs contiguous rows and cuts them into pieces of 3.5 KB that its
// warps take in turn from a shared-memory counter, each warp issuing the next
// piece's loads before it sums the current one (a row's last, shorter part is
// summed after, by one warp per row).  A warp's share of the SM's
// bandwidth varies from warp to warp, so a static one-row-per-warp split ends
// when its slowest warp does; taking pieces in turn ends all warps of a CTA
// together.  Each piece's sum goes to a fixed slot and a row adds its slots in
// order, so which warp took which piece does not change the result.
// gemv_f16_kernel (one warp per row, all resident at once) covers the rest.
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

// ---- pieces: one CTA per SM, warps take 3.5 KB pieces of the CTA's rows ----
constexpr int kPcWarps = 28;        // warps per CTA
constexpr int kPcLoads = 7;         // 16-byte loads per lane per piece
constexpr int32_t kPcChunks = 32 * kPcLoads;   // 16-byte chunks per piece (3.5 KB)
constexpr int kPcMaxRows = 64;      // rows per CTA the slot table holds
constexpr int kPcMaxPieces = 64;    // pieces per row the slot table holds

template <bool BF16>
__global__ void __launch_bounds__(kPcWarps * 32, 1)
gemv_pieces_kernel(const uint4* __restrict__ x, const uint4* __restrict__ W,
                   uint16_t* __restrict__ y, int32_t N, int32_t K8, uint32_t* __restrict__ err) {
    grid_launch_dependents();
    __shared__ int next_piece;
    __shared__ float slot[kPcMaxRows][kPcMaxPieces];
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int32_t r0 = static_cast<int32_t>(static_cast<int64_t>(blockIdx.x) * N / gridDim.x);
    const int32_t r1 = static_cast<int32_t>(static_cast<int64_t>(blockIdx.x + 1) * N / gridDim.x);
    const int32_t rows = r1 - r0;
    // Whole pieces of a row, taken in turn; the rest of the row (fewer than
    // kPcChunks chunks) is one more slot, summed by one warp per row after.
    const int32_t pieces = K8 / kPcChunks;
    const int32_t tail0 = pieces * kPcChunks;
    const int32_t items = rows * pieces;
    if (threadIdx.x == 0) next_piece = 0;
    // While the previous grid finishes, pull the head of each of this CTA's
    // rows into L2 (a prefetch cannot see stale data).
    if (kGvPrefetchChunks > 0 && threadIdx.x < rows)
        prefetch_l2_bytes(W + static_cast<int64_t>(r0 + threadIdx.x) * K8,
                          static_cast<uint32_t>(min(K8, kGvPrefetchChunks)) * 16u);
    __syncthreads();
    grid_dependency_wait();   // x and W may come from the grid before this one
    auto take = [&]() {
        int v = 0;
        if (lane == 0) v = atomicAdd(&next_piece, 1);
        return __shfl_sync(0xffffffffu, v, 0);
    };
    // Piece `it` = row it / pieces, chunks [pc * kPcChunks, +kPcChunks) of it;
    // lane l holds chunks pc * kPcChunks + l + 32 u.
    auto load = [&](int it, uint4 (&w)[kPcLoads]) {
        const int32_t row = it / pieces, pc = it % pieces;
        const uint4* p = W + static_cast<int64_t>(r0 + row) * K8 + pc * kPcChunks + lane;
#pragma unroll
        for (int u = 0; u < kPcLoads; ++u) w[u] = ld_stream_v4(p + 32 * u);
    };
    uint4 wa[kPcLoads], wb[kPcLoads];
    int cur = take();
    if (cur < items) load(cur, wa);
    while (cur < items) {
        const int nxt = take();
        if (nxt < items) load(nxt, wb);
        const int32_t row = cur / pieces, pc = cur % pieces;
        const int32_t base = pc * kPcChunks + lane;
        float acc = 0.f;
#pragma unroll
        for (int u = 0; u < kPcLoads; ++u) acc = dot8<BF16>(wa[u], __ldg(x + base + 32 * u), acc);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
        if (lane == 0) slot[row][pc] = acc;
#pragma unroll
        for (int u = 0; u < kPcLoads; ++u) wa[u] = wb[u];
        cur = nxt;
    }
    if (tail0 < K8) {
        for (int32_t row = warp; row < rows; row += kPcWarps) {
            const uint4* wrow = W + static_cast<int64_t>(r0 + row) * K8;
            float acc = 0.f;
            for (int32_t c = tail0 + lane; c < K8; c += 32)
                acc = dot8<BF16>(ld_stream_v4(wrow + c), __ldg(x + c), acc);
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
            if (lane == 0) slot[row][pieces] = acc;
        }
    }
    __syncthreads();
    if (threadIdx.x < rows) {
        const int32_t slots = pieces + (tail0 < K8 ? 1 : 0);
        float s = slot[threadIdx.x][0];
        for (int32_t pc = 1; pc < slots; ++pc) s += slot[threadIdx.x][pc];
        const int32_t n = r0 + static_cast<int32_t>(threadIdx.x);
        if constexpr (BF16)
            y[n] = __bfloat16_as_ushort(__float2bfloat16_rn(s));
        else
            y[n] = __half_as_ushort(__float2half_rn(s));
        check_count_unit(err, n);   // checked build: output rows written
    }
}

}  // namespace

cudaError_t launch_gemv(int64_t N, int64_t K, const void* x, const void* W, void* y, bool bf16,
                        int num_sms, cudaStream_t stream, uint32_t* err, bool pdl) {
    const int32_t K8 = static_cast<int32_t>(K / 8);
    const int64_t pieces = K8 / kPcChunks + (K8 % kPcChunks != 0 ? 1 : 0);   // slots per row
    if (num_sms > 0 && N >= num_sms && (N + num_sms - 1) / num_sms <= kPcMaxRows &&
        pieces <= kPcMaxPieces) {
        auto kernel = bf16 ? gemv_pieces_kernel<true> : gemv_pieces_kernel<false>;
        return launch_kernel(kernel, dim3(static_cast<unsigned>(num_sms)), dim3(kPcWarps * 32), 0,
                             stream, 1u, pdl, static_cast<const uint4*>(x),
                             static_cast<const uint4*>(W), static_cast<uint16_t*>(y),
                             static_cast<int32_t>(N), K8, err);
    }
    const int64_t blocks = (N + kGvWarps - 1) / kGvWarps;
    auto kernel = bf16 ? gemv_f16_kernel<true> : gemv_f16_kernel<false>;
    return launch_kernel(kernel, dim3(static_cast<unsigned>(blocks)), dim3(kGvWarps * 32), 0,
                         stream, 1u, pdl, static_cast<const uint4*>(x), static_cast<const uint4*>(W),
                         static_cast<uint16_t*>(y), static_cast<int32_t>(N), K8, err);
}

}  // namespace tmagemm
