// Skinny GEMM for a few tokens, D = fp16(X W^T) with 2 <= M <= 64 (and the same
// with bf16 operands and output), on tcgen05
// with the weights staged in shared memory by the SMs' own loads.
//
// The decode step reads each weight once ("Learning TileLang with GEMV", §01
// GEMV, §02 Bandwidth Bound), so the weight stream sets the time.  On GB300
// per-thread 16-byte loads with enough of them in flight stream HBM faster
// than the TMA-fed swap-AB kernel does (about 4 TB/s).  This
// kernel keeps the tensor-core path (tcgen05.mma from shared-memory
// descriptors, FP32 accumulator in TMEM) and moves only the weight operand
// off TMA.
//
// Work: the swapped problem D^T = W X^T.  A CTA owns 128 weight rows (the MMA
// M) and one K slice; the 8 CTAs of a thread-block cluster own the same rows
// and the 8 slices of K.
//   - Weight producers, two warpgroups taking k-blocks in turn: a k-block of
//     the tile is 128 rows x 128 bytes; each warp instruction loads 4 whole
//     rows (512 contiguous bytes per row group, 16 bytes per lane), eight per
//     thread, with the next k-block's loads in flight.  The threads store the
//     chunks into the 128B-swizzled K-major layout the MMA descriptor reads
//     (chunk j of row r at j ^ (r mod 8)), fence the generic-proxy writes
//     for the async proxy and arrive on the stage's barrier.
//   - X producer (one thread): TMA loads the 64-k slab of the Mp (16/32/64)
//     token rows, rows past M zero-filled.
//   - MMA issuer (one thread): per k-block four tcgen05.mma (K = 16 each)
//     into one 128 x Mp FP32 accumulator.
//   - Epilogue: the first warpgroup reads the accumulator (tcgen05.ld) into a
//     shared-memory partial tile; after a cluster barrier CTA q adds the 8
//     slices' partials of rows 16q .. 16q+15 in slice order through
//     distributed shared memory, rounds once to fp16 and writes D.
// No workspace, one launch, deterministic.  Every mbarrier wait is bounded
// (the CTA-wide abort flag and the device error word, as in the GEMM).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <atomic>
#include <cstdint>

#include "launch.h"
#include "ptx.cuh"

namespace tmagemm {

namespace {

constexpr int kTmRows = 128;          // weight rows per CTA (MMA M)
constexpr int kTmSlices = 8;          // CTAs per cluster = K slices
constexpr int kTmStages = 4;          // k-blocks in flight between producers and MMA
constexpr int kTmProducerWarps = 8;   // two warpgroups
constexpr int kTmMmaWarp = 8;
constexpr int kTmXWarp = 9;
constexpr uint32_t kTmABytes = kTmRows * 128;   // one k-block of the weight tile

static_assert(kTmStages % 2 == 0, "each stage belongs to one producer warpgroup");

__device__ __forceinline__ void st_shared_u4(uint32_t addr, const uint4& v) {
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};"
                 ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w) : "memory");
}

__device__ __forceinline__ uint4 ld_weight_chunk(const uint4* p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

__device__ __forceinline__ float ld_cluster_f32(uint32_t addr) {
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
    return v;
}

// Lane 0 waits; the result is shared by the warp (keeps warp-collective
// tcgen05 instructions convergent).
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          uint32_t* err, uint32_t site, uint64_t limit_ns) {
    bool ok = true;
    if ((threadIdx.x & 31) == 0) ok = wait_or_abort(bar, parity, abort_flag, err, site, limit_ns);
    return __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
}

template <int MP>
struct TmLayout {
    static constexpr uint32_t kXStage = MP * 128;                    // Mp rows x 64 fp16
    static constexpr uint32_t kOffA = 0;
    static constexpr uint32_t kOffX = kOffA + kTmStages * kTmABytes;
    static constexpr uint32_t kPartStride = MP + 1;                  // floats per partial row
    // The partial tile reuses the weight stages once every MMA has finished.
    static constexpr uint32_t kOffPart = kOffA;
    static constexpr uint32_t kOffBar = kOffX + kTmStages * kXStage;
    static constexpr uint32_t kNumBars = 3 * kTmStages + 2;
    static constexpr uint32_t kOffMisc = kOffBar + kNumBars * 8;
    static constexpr uint32_t kSmemBytes = kOffMisc + 16 + 1024;     // + alignment slack
    static constexpr uint32_t kTmemCols = MP <= 32 ? 32 : 64;
    static_assert(kXStage % 1024 == 0, "X stages stay 1024-byte aligned (128B swizzle atoms)");
    static_assert(kTmRows * kPartStride * 4 <= kTmStages * kTmABytes, "partial tile fits");
};

// Two producer warpgroups, the MMA warp and the X warp; two CTAs per SM.
constexpr int kTmThreads = 320;

template <int MP, bool BF16>
__global__ void __launch_bounds__(kTmThreads, 2)
small_m_lsu_kernel(const __grid_constant__ CUtensorMap tmX, const uint4* __restrict__ W,
                   uint16_t* __restrict__ D, int32_t M, int32_t N, int32_t K8, int32_t kb_total,
                    int32_t kb_per_slice, uint64_t limit_ns, uint32_t* __restrict__ err) {
    using L = TmLayout<MP>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;
    uint8_t* smem = smem_raw + (sbase - raw);
    float* part = reinterpret_cast<float*>(smem + L::kOffPart);
    const uint32_t bar0 = sbase + L::kOffBar;
    auto wfull_bar = [&](uint32_t s) { return bar0 + 8u * s; };
    auto xfull_bar = [&](uint32_t s) { return bar0 + 8u * (kTmStages + s); };
    auto empty_bar = [&](uint32_t s) { return bar0 + 8u * (2 * kTmStages + s); };
    const uint32_t acc_bar = bar0 + 8u * (3 * kTmStages);
    const uint32_t done_bar = acc_bar + 8u;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + L::kOffMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kOffMisc + 4);

    grid_launch_dependents();
    const int warp = __shfl_sync(0xffffffffu, static_cast<int>(threadIdx.x) / 32, 0);
    const int lane = static_cast<int>(threadIdx.x) & 31;
    const uint32_t rank = cluster_ctarank();
    const int32_t row0 = static_cast<int32_t>(blockIdx.x / kTmSlices) * kTmRows;
    const int32_t kb_begin = static_cast<int32_t>(rank) * kb_per_slice;
    const int32_t kb_end = min(kb_total, kb_begin + kb_per_slice);
    const int32_t nkb = kb_end > kb_begin ? kb_end - kb_begin : 0;

    if (threadIdx.x == 0) {
        for (uint32_t s = 0; s < static_cast<uint32_t>(kTmStages); ++s) {
            mbar_init(wfull_bar(s), 128);   // every thread of the stage's warpgroup
            mbar_init(xfull_bar(s), 1);   // the X producer's arrival + TMA bytes
            mbar_init(empty_bar(s), 1);   // the MMA commit
        }
        mbar_init(acc_bar, 1);
        mbar_init(done_bar, 1);
        *abort_flag = 0;
        fence_mbarrier_init();
        tma_prefetch_desc(&tmX);
    }
    grid_dependency_wait();   // X, W and D (and the previous grid's TMEM) are touched after this
    if (warp == 0) {
        tmem_alloc(smem_u32(tmem_holder), L::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;
    const uint32_t lane_base = static_cast<uint32_t>(32 * (warp & 3)) << 16;

    if (warp < kTmProducerWarps) {
        // ============ weight producers: warpgroup g takes k-blocks g, g+2, ... ============
        // Thread t of the warpgroup moves chunks q = 128 j + t (j < 8) of the
        // 128-row x 8-chunk k-block: row q / 8 = t / 8 + 16 j, chunk t % 8, so
        // a warp instruction covers 4 whole 128-byte row segments.
        const int g = warp / 4;
        const int t = static_cast<int>(threadIdx.x) & 127;
        // Rows r0 + 16 j (j < 8) at chunk ch; the swizzled chunk position is
        // the same for every j because 16 j is a multiple of the 8-row atom.
        const int r0 = t >> 3, ch = t & 7;
        const uint4* src0 = W + static_cast<int64_t>(row0 + r0) * K8 + ch;
        const int64_t row_step = static_cast<int64_t>(16) * K8;
        uint32_t valid = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) valid |= (row0 + r0 + 16 * j < N ? 1u : 0u) << j;
        const uint32_t dst0 = static_cast<uint32_t>(r0 * 128 + ((ch ^ (r0 & 7)) << 4));
        auto load = [&](int32_t i, uint4 (&v)[8]) {
            const int32_t c0 = (kb_begin + i) * 8;
            const bool ok = c0 + ch < K8;
#pragma unroll
            for (int j = 0; j < 8; ++j)
                v[j] = (ok && ((valid >> j) & 1u)) ? ld_weight_chunk(src0 + j * row_step + c0)
                                                   : make_uint4(0, 0, 0, 0);
        };
        uint4 cur[8], nxt[8];
        int32_t i = g;
        if (i < nkb) load(i, cur);
        for (; i < nkb; i += 2) {
            if (i + 2 < nkb) load(i + 2, nxt);
            const uint32_t s = static_cast<uint32_t>(i) % kTmStages;
            const uint32_t use = static_cast<uint32_t>(i) / kTmStages;
            if (!warp_wait(empty_bar(s), (use & 1u) ^ 1u, abort_flag, err, kSiteProducerEmpty,
                           limit_ns))
                break;
            const uint32_t a_stage = sbase + L::kOffA + s * kTmABytes;
#pragma unroll
            for (int j = 0; j < 8; ++j) st_shared_u4(a_stage + dst0 + 2048u * j, cur[j]);
            fence_proxy_async_smem();   // generic-proxy writes -> the MMA's async proxy
            mbar_arrive(wfull_bar(s));
#pragma unroll
            for (int j = 0; j < 8; ++j) cur[j] = nxt[j];

        }
    } else if (warp == kTmXWarp) {
        // ============ X producer ============
        if (lane == 0) {
            int32_t issued = 0;
            for (int32_t i = 0; i < nkb; ++i) {
                const uint32_t s = static_cast<uint32_t>(i) % kTmStages;
                const uint32_t use = static_cast<uint32_t>(i) / kTmStages;
                if (!wait_or_abort(empty_bar(s), (use & 1u) ^ 1u, abort_flag, err,
                                   kSiteProducerEmpty, limit_ns))
                    break;
                mbar_arrive_expect_tx(xfull_bar(s), L::kXStage);
                tma_load_2d(sbase + L::kOffX + s * L::kXStage, &tmX, (kb_begin + i) * 64, 0,
                            xfull_bar(s));
                issued = i + 1;
            }
            // Every issued copy lands before shared memory is released.
            for (int32_t j = issued > kTmStages ? issued - kTmStages : 0; j < issued; ++j)
                wait_bounded(xfull_bar(static_cast<uint32_t>(j) % kTmStages),
                             (static_cast<uint32_t>(j) / kTmStages) & 1u, err, kSiteDrainFull,
                             limit_ns);
        }
        __syncwarp();
    } else if (warp == kTmMmaWarp) {
        // ============ MMA issuer ============
        if (lane == 0) {
            constexpr uint32_t kIdesc = umma_idesc_16bit_f32(kTmRows, MP, BF16);
            bool ok = true;
            for (int32_t i = 0; i < nkb; ++i) {
                const uint32_t s = static_cast<uint32_t>(i) % kTmStages;
                const uint32_t ph = (static_cast<uint32_t>(i) / kTmStages) & 1u;
                if (!wait_or_abort(wfull_bar(s), ph, abort_flag, err, kSiteMmaFull, limit_ns) ||
                    !wait_or_abort(xfull_bar(s), ph, abort_flag, err, kSiteMmaFull, limit_ns)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t a_addr = sbase + L::kOffA + s * kTmABytes;
                const uint32_t x_addr = sbase + L::kOffX + s * L::kXStage;
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    mma_f16_ss(tmem_base, umma_desc_sw128_kmajor(a_addr + 32u * j),
                               umma_desc_sw128_kmajor(x_addr + 32u * j), kIdesc,
                               (i != 0 || j != 0) ? 1u : 0u);
                mma_commit(empty_bar(s));
            }
            if (ok && nkb > 0) mma_commit(acc_bar);
            // Every issued MMA finishes before TMEM is released.
            mma_commit(done_bar);
            wait_bounded(done_bar, 0, err, kSiteDrainMma, limit_ns);
        }
        __syncwarp();
    }

    // ============ epilogue: accumulator -> this slice's partial tile ============
    if (warp < 4) {
        const int rl = 32 * warp + lane;
        bool ok = nkb > 0;
        if (ok) ok = warp_wait(acc_bar, 0, abort_flag, err, kSiteEpiAccFull, limit_ns);
        tc_fence_after();
        if (ok) {
#pragma unroll
            for (int c0 = 0; c0 < MP; c0 += 16) {
                uint32_t v[16];
                tmem_ld_32x32b_x16(tmem_base + lane_base + c0, v);
                tmem_ld_wait();
#pragma unroll
                for (int c = 0; c < 16; ++c) part[rl * L::kPartStride + c0 + c] = __uint_as_float(v[c]);
            }
        } else {
#pragma unroll
            for (int c = 0; c < MP; ++c) part[rl * L::kPartStride + c] = 0.0f;
        }
    }
    tc_fence_before();
    cluster_sync();   // every slice's partial tile is visible cluster-wide

    // CTA `rank` finishes weight rows [16 rank, 16 rank + 16): each output is
    // the sum of the 8 slices' partials, loaded together, added in slice order.
    constexpr int kRowsPerCta = kTmRows / kTmSlices;
    for (int o = static_cast<int>(threadIdx.x); o < kRowsPerCta * MP; o += kTmThreads) {
        const int rl = static_cast<int>(rank) * kRowsPerCta + o % kRowsPerCta;
        const int m = o / kRowsPerCta;
        const int32_t n = row0 + rl;
        if (m >= M || n >= N) continue;
        const uint32_t local = smem_u32(&part[rl * L::kPartStride + m]);
        float v[kTmSlices];
#pragma unroll
        for (int q = 0; q < kTmSlices; ++q) v[q] = ld_cluster_f32(map_to_rank(local, q));
        float sum = v[0];
#pragma unroll
        for (int q = 1; q < kTmSlices; ++q) sum += v[q];
        if constexpr (BF16)
            D[static_cast<int64_t>(m) * N + n] = __bfloat16_as_ushort(__float2bfloat16_rn(sum));
        else
            D[static_cast<int64_t>(m) * N + n] = __half_as_ushort(__float2half_rn(sum));
    }
    cluster_sync();   // peers' shared memory stays alive until every CTA has read it
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem_base, L::kTmemCols);
    }
    if (threadIdx.x == 0 && !*abort_flag) check_count_unit(err, static_cast<int32_t>(blockIdx.x));
}

template <int MP, bool BF16>
cudaError_t launch_mp(const CUtensorMap& tmX, int64_t M, int64_t N, int64_t K, const void* W,
                      void* D, uint64_t limit_ns, uint32_t* err, cudaStream_t stream, bool pdl) {
    auto kernel = small_m_lsu_kernel<MP, BF16>;
    static ContextMarks attr_done;
    cudaError_t e = smem_opt_in(kernel, static_cast<int>(TmLayout<MP>::kSmemBytes), attr_done,
                                false);
    if (e != cudaSuccess) return e;
    const int32_t kb_total = static_cast<int32_t>((K + 63) / 64);
    const int32_t kb_per_slice = (kb_total + kTmSlices - 1) / kTmSlices;
    const int64_t clusters = (N + kTmRows - 1) / kTmRows;
    return launch_kernel(kernel, dim3(static_cast<unsigned>(clusters * kTmSlices)), dim3(kTmThreads),
                         TmLayout<MP>::kSmemBytes, stream, static_cast<unsigned>(kTmSlices), pdl,
                         tmX,
                         static_cast<const uint4*>(W), static_cast<uint16_t*>(D),
                         static_cast<int32_t>(M), static_cast<int32_t>(N),
                         static_cast<int32_t>(K / 8), kb_total, kb_per_slice, limit_ns, err);
}

}  // namespace

int64_t small_m_lsu_cols(int64_t M) { return M <= 16 ? 16 : M <= 32 ? 32 : 64; }

cudaError_t launch_small_m_lsu(const CUtensorMap& tmX, int64_t M, int64_t N, int64_t K,
                               const void* W, void* D, uint64_t limit_ns, uint32_t* err,
                               cudaStream_t stream, bool bf16, bool pdl) {
    switch (small_m_lsu_cols(M) * (bf16 ? -1 : 1)) {
        case 16: return launch_mp<16, false>(tmX, M, N, K, W, D, limit_ns, err, stream, pdl);
        case 32: return launch_mp<32, false>(tmX, M, N, K, W, D, limit_ns, err, stream, pdl);
        case 64: return launch_mp<64, false>(tmX, M, N, K, W, D, limit_ns, err, stream, pdl);
        case -16: return launch_mp<16, true>(tmX, M, N, K, W, D, limit_ns, err, stream, pdl);
        case -32: return launch_mp<32, true>(tmX, M, N, K, W, D, limit_ns, err, stream, pdl);
        default: return launch_mp<64, true>(tmX, M, N, K, W, D, limit_ns, err, stream, pdl);
    }
}

}  // namespace tmagemm
