// Persistent, warp-specialised FP16 TN GEMM for sm_103a:
//   D[M x N] = fp16( A[M x K] * B[N x K]^T ), FP32 accumulation in TMEM.
//
// Roles (one CTA per SM, 6 warps):
//   warp 0      TMA producer: one elected lane streams A/B k-blocks into a
//               STAGES-deep ring of 128B-swizzled SMEM stages.  Per stage it
//               waits `empty[s]`, registers the stage's bytes with
//               arrive.expect_tx on `full[s]` and issues two TMA tile loads
//               ("使用 TMA 为 GEMM 建立 Pipeline", 第 4 步 发起 TMA Load / 第 5 步
//               Pipeline 机制; the Croqtile producer/consumer pipeline with
//               full/empty events, "示例：流水线矩阵乘法中的 TMA").
//   warp 1      MMA issuer: one elected lane waits `full[s]`, issues
//               BK/16 tcgen05.mma (128 x BN x 16) into one of two TMEM
//               accumulators and releases the stage with tcgen05.commit onto
//               `empty[s]`; after a tile's last k-block it commits onto
//               `acc_full[acc]`.  This warp also owns the TMEM allocation.
//   warps 2..5  epilogue: wait `acc_full[acc]`, tcgen05.ld the accumulator
//               (warp w reads TMEM lanes 32*(w%4)..+31 = tile rows), hand the
//               accumulator back through `acc_empty[acc]`, convert to fp16
//               (round to nearest even), write a 128B-swizzled SMEM box and
//               TMA-store it (commit_group / wait_group.read before reuse)
//               (step 4, 等待 TMA Load 和 Store 完成).
// The two TMEM accumulators let the epilogue of tile t overlap the mainloop
// of tile t+1 — the overlap the pages defer to a warp-specialised step 7.
//
// Ragged M/N/K: TMA zero-fills out-of-range operand elements (the .zfill rule
// of "高级数据搬运…", 零填充) and clamps out-of-range stores, so interior and
// edge tiles run the same code.
//
// Every mbarrier wait is bounded (see ptx.cuh): on a timeout the CTA raises a
// shared abort flag, all roles leave their loops, in-flight TMA loads and
// MMAs are drained, TMEM is freed, and the error word records the site.
#include <cuda.h>
#include <cuda_runtime.h>
#include <atomic>
#include <cstdint>

#include "launch.h"
#include "ptx.cuh"
#include "tile_sched.cuh"

namespace tmagemm {

namespace {

template <int BN_, int EPI_COLS_, int STAGES_>
struct Cfg {
    static constexpr int BM = 128, BN = BN_, BK = 64, STAGES = STAGES_;
    static constexpr int kThreads = 192;            // 6 warps
    static constexpr int kEpiThreads = 128;         // warps 2..5
    static constexpr int kEpiCols = EPI_COLS_;      // columns per TMA store box
    static constexpr uint32_t kEpiRowBytes = kEpiCols * 2;       // = the box's swizzle span
    static constexpr uint32_t kEpiChunks = kEpiRowBytes / 16;    // 16-byte chunks per box row
    static constexpr int kGroupM = 8;               // L2 group height in tiles
    static constexpr uint32_t kABytes = BM * BK * 2;
    static constexpr uint32_t kBBytes = BN * BK * 2;
    static constexpr uint32_t kStageBytes = kABytes + kBBytes;
    static constexpr uint32_t kEpiBufBytes = BM * kEpiRowBytes;
    static constexpr int kEpiBufs = 2;
    static constexpr uint32_t kTmemCols = 512;      // two accumulators, 256 columns apart
    static constexpr uint32_t kAccStride = 256;
    static constexpr uint32_t kOffA = 0;
    static constexpr uint32_t kOffB = kOffA + STAGES * kABytes;
    static constexpr uint32_t kOffD = kOffB + STAGES * kBBytes;
    static constexpr uint32_t kOffBar = kOffD + kEpiBufs * kEpiBufBytes;
    static constexpr uint32_t kNumBars = 2 * STAGES + 5;
    static constexpr uint32_t kOffMisc = kOffBar + kNumBars * 8;
    static constexpr uint32_t kSmemBytes = kOffMisc + 16 + 1024;   // + base alignment slack
    static constexpr uint32_t kIdesc = umma_idesc_f16_f32(BM, BN);

    static_assert(BK * 2 == 128, "a K-major row of one k-block is one 128-byte swizzle atom");
    static_assert(BN % 16 == 0 && BN >= 16 && BN <= 256, "UMMA N for M = 128");
    static_assert(kEpiCols == 32 || kEpiCols == 64, "store boxes are 64 or 128 bytes wide");
    static_assert(BN % kEpiCols == 0, "epilogue boxes tile BN");
    static_assert(kAccStride + BN <= kTmemCols, "two accumulators fit in TMEM");
    static_assert(kABytes % 1024 == 0 && kBBytes % 1024 == 0, "stages stay 1024-B aligned");
    static_assert(kEpiBufBytes % 1024 == 0, "epilogue boxes stay 1024-B aligned");
    static_assert(kSmemBytes <= 232448, "fits the 227 KB opt-in shared memory");
};

// Tile shapes the host plan chooses from (all 128 rows x BN columns x 64 K).
using Cfg256 = Cfg<256, 64, 4>;
using Cfg224 = Cfg<224, 32, 4>;
using Cfg192 = Cfg<192, 64, 4>;

template <class C>
__global__ void __launch_bounds__(C::kThreads, 1)
gemm_tn_f16_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmD, const int32_t N, const int32_t grid_m,
                   const int32_t grid_n, const int32_t num_tiles, const int32_t k_blocks,
                   const uint64_t limit_ns, uint32_t* __restrict__ err) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // Dynamic shared memory is only guaranteed 16-byte aligned: round up.
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;
    uint8_t* smem = smem_raw + (sbase - raw);

    const uint32_t bar0 = sbase + C::kOffBar;
    auto full_bar = [&](uint32_t s) { return bar0 + 8u * s; };
    auto empty_bar = [&](uint32_t s) { return bar0 + 8u * (C::STAGES + s); };
    auto acc_full_bar = [&](uint32_t a) { return bar0 + 8u * (2 * C::STAGES + a); };
    auto acc_empty_bar = [&](uint32_t a) { return bar0 + 8u * (2 * C::STAGES + 2 + a); };
    const uint32_t mma_done_bar = bar0 + 8u * (2 * C::STAGES + 4);
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 4);

    const int warp = __shfl_sync(0xffffffffu, static_cast<int>(threadIdx.x) / 32, 0);
    const int lane = static_cast<int>(threadIdx.x) % 32;

    // ---- one-time setup: barriers (warp 0), TMEM (warp 1) ----
    if (warp == 0) {
        if (elect_one()) {
            for (uint32_t s = 0; s < (uint32_t)C::STAGES; ++s) {
                mbar_init(full_bar(s), 1);
                mbar_init(empty_bar(s), 1);
            }
            for (uint32_t a = 0; a < 2; ++a) {
                mbar_init(acc_full_bar(a), 1);
                mbar_init(acc_empty_bar(a), C::kEpiThreads / 32);
            }
            mbar_init(mma_done_bar, 1);
            *abort_flag = 0;
            fence_mbarrier_init();
            tma_prefetch_desc(&tmA);
            tma_prefetch_desc(&tmB);
            tma_prefetch_desc(&tmD);
        }
        __syncwarp();
    } else if (warp == 1) {
        tmem_alloc(smem_u32(tmem_holder), C::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;

    if (warp == 0) {
        // ================= TMA producer =================
        if (elect_one()) {
            uint32_t it = 0;
            bool ok = true;
            for (int32_t tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x) {
                const TileCoord tc = tile_coord(tile, grid_m, grid_n, C::kGroupM);
                const int32_t m0 = tc.m_blk * C::BM;
                const int32_t n0 = tc.n_blk * C::BN;
                for (int32_t kb = 0; kb < k_blocks; ++kb) {
                    const uint32_t s = ring_stage(it, C::STAGES);
                    const uint32_t ph = ring_phase(it, C::STAGES);
                    if (!wait_or_abort(empty_bar(s), ph ^ 1u, abort_flag, err, kSiteProducerEmpty,
                                       limit_ns)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(full_bar(s), C::kStageBytes);
                    tma_load_2d(sbase + C::kOffA + s * C::kABytes, &tmA, kb * C::BK, m0, full_bar(s));
                    tma_load_2d(sbase + C::kOffB + s * C::kBBytes, &tmB, kb * C::BK, n0, full_bar(s));
                    ++it;
                }
            }
            // Drain: the last (up to) STAGES issued stages must have landed
            // before shared memory is released.
            const uint32_t first = it > (uint32_t)C::STAGES ? it - C::STAGES : 0u;
            for (uint32_t j = first; j < it; ++j)
                wait_bounded(full_bar(ring_stage(j, C::STAGES)), ring_phase(j, C::STAGES), err,
                             kSiteDrainFull, limit_ns);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ================= MMA issuer =================
        if (elect_one()) {
            uint32_t it = 0, tcount = 0;
            bool ok = true;
            for (int32_t tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x, ++tcount) {
                const uint32_t acc = tcount & 1u;
                const uint32_t acc_ph = (tcount >> 1) & 1u;
                if (!wait_or_abort(acc_empty_bar(acc), acc_ph ^ 1u, abort_flag, err,
                                   kSiteMmaAccEmpty, limit_ns))
                    break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * C::kAccStride;
                for (int32_t kb = 0; kb < k_blocks; ++kb) {
                    const uint32_t s = ring_stage(it, C::STAGES);
                    const uint32_t ph = ring_phase(it, C::STAGES);
                    if (!wait_or_abort(full_bar(s), ph, abort_flag, err, kSiteMmaFull, limit_ns)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_addr = sbase + C::kOffA + s * C::kABytes;
                    const uint32_t b_addr = sbase + C::kOffB + s * C::kBBytes;
#pragma unroll
                    for (int j = 0; j < C::BK / 16; ++j) {
                        mma_f16_ss(d_tmem, umma_desc_sw128_kmajor(a_addr + 32u * j),
                                   umma_desc_sw128_kmajor(b_addr + 32u * j), C::kIdesc,
                                   (kb | j) != 0 ? 1u : 0u);
                    }
                    mma_commit(empty_bar(s));   // stage s free once these MMAs finish
                    ++it;
                }
                if (!ok) break;
                mma_commit(acc_full_bar(acc));  // accumulator ready for the epilogue
            }
            // All issued MMAs must finish before TMEM is released.
            mma_commit(mma_done_bar);
            wait_bounded(mma_done_bar, 0, err, kSiteDrainMma, limit_ns);
        }
        __syncwarp();
    } else {
        // ================= epilogue (warps 2..5) =================
        const uint32_t quarter = static_cast<uint32_t>(warp) & 3u;   // TMEM lane quarter
        const uint32_t row = quarter * 32u + static_cast<uint32_t>(lane);  // row in tile
        const bool leader = threadIdx.x == 64;
        uint32_t tcount = 0, box = 0;
        for (int32_t tile = blockIdx.x; tile < num_tiles; tile += gridDim.x, ++tcount) {
            const TileCoord tc = tile_coord(tile, grid_m, grid_n, C::kGroupM);
            const int32_t m0 = tc.m_blk * C::BM;
            const int32_t n0 = tc.n_blk * C::BN;
            const uint32_t acc = tcount & 1u;
            const uint32_t acc_ph = (tcount >> 1) & 1u;
            bool ok = wait_or_abort(acc_full_bar(acc), acc_ph, abort_flag, err, kSiteEpiAccFull,
                                    limit_ns);
            // All 128 epilogue threads take the same decision.
            if (!named_bar_and(1, C::kEpiThreads, ok)) break;
            tc_fence_after();
            const uint32_t t_row = tmem_base + ((quarter * 32u) << 16) + acc * C::kAccStride;
#pragma unroll 1
            for (int c = 0; c < C::BN / C::kEpiCols; ++c, ++box) {
                uint32_t v[C::kEpiCols];
#pragma unroll
                for (int h = 0; h < C::kEpiCols / 32; ++h)
                    tmem_ld_32x32b_x32(t_row + c * C::kEpiCols + 32 * h,
                                       *reinterpret_cast<uint32_t(*)[32]>(&v[32 * h]));
                tmem_ld_wait();
                if (c == C::BN / C::kEpiCols - 1) {
                    // Whole accumulator read: give it back to the MMA warp.
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(acc_empty_bar(acc));
                }
                const uint32_t buf = sbase + C::kOffD + (box & 1u) * C::kEpiBufBytes;
                // The store that last read this buffer (two boxes ago) must be done.
                if (leader) bulk_wait_group_read<1>();
                named_bar_sync(1, C::kEpiThreads);
                // Row `row` of the box holds kEpiChunks 16-byte chunks.  The
                // TMA swizzle whose span equals the row width (64B or 128B)
                // XORs the chunk index with address bits 7.. of the row start:
                // chunk j of row r lands at j ^ ((r * row_bytes / 128) % chunks).
                const uint32_t row_addr = buf + row * C::kEpiRowBytes;
                const uint32_t xr = ((row * C::kEpiRowBytes) >> 7) & (C::kEpiChunks - 1);
#pragma unroll
                for (uint32_t j = 0; j < C::kEpiChunks; ++j) {
                    const uint32_t p0 = pack_half2_rn(v[8 * j + 0], v[8 * j + 1]);
                    const uint32_t p1 = pack_half2_rn(v[8 * j + 2], v[8 * j + 3]);
                    const uint32_t p2 = pack_half2_rn(v[8 * j + 4], v[8 * j + 5]);
                    const uint32_t p3 = pack_half2_rn(v[8 * j + 6], v[8 * j + 7]);
                    st_shared_v4(row_addr + ((j ^ xr) << 4), p0, p1, p2, p3);
                }
                fence_proxy_async_smem();
                named_bar_sync(1, C::kEpiThreads);
                if (leader) {
                    const int32_t x = n0 + c * C::kEpiCols;
                    if (x < N) tma_store_2d(&tmD, buf, x, m0);
                    bulk_commit_group();
                }
            }
        }
        if (leader) bulk_wait_group<0>();
    }

    // ---- teardown ----
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, C::kTmemCols);
    }
}

}  // namespace

namespace {

template <class C>
GemmPlan plan_for(int64_t M, int64_t N, int64_t K, int64_t sms) {
    GemmPlan p{};
    p.bm = C::BM;
    p.bn = C::BN;
    p.bk = C::BK;
    p.stages = C::STAGES;
    p.epi_cols = C::kEpiCols;
    p.grid_m = ceil_div(M, C::BM);
    p.grid_n = ceil_div(N, C::BN);
    p.k_blocks = ceil_div(K, C::BK);
    p.tiles = p.grid_m * p.grid_n;
    p.grid = static_cast<int>(p.tiles < sms ? p.tiles : sms);
    p.threads = C::kThreads;
    p.smem_bytes = static_cast<int>(C::kSmemBytes);
    return p;
}

// Modelled time of a plan: the busiest CTA runs ceil(tiles / grid) tiles, and
// a tile's mainloop costs about BN + 32 units (MMA time grows with BN, the A
// operand traffic per k-block does not).
int64_t plan_cost(const GemmPlan& p) {
    const int64_t rounds = ceil_div(p.tiles, p.grid);
    return rounds * (p.bn + 32);
}

template <class C>
cudaError_t launch_cfg(const GemmPlan& plan, const CUtensorMap& tmA, const CUtensorMap& tmB,
                       const CUtensorMap& tmD, const GemmArgs& args, cudaStream_t stream) {
    auto kernel = gemm_tn_f16_kernel<C>;
    // Per-device opt-in to > 48 KB dynamic shared memory, once per device.
    static std::atomic<bool> attr_done[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64 || !attr_done[dev].load(std::memory_order_acquire)) {
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(C::kSmemBytes));
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) attr_done[dev].store(true, std::memory_order_release);
    }
    kernel<<<plan.grid, C::kThreads, C::kSmemBytes, stream>>>(
        tmA, tmB, tmD, args.N, static_cast<int32_t>(plan.grid_m), static_cast<int32_t>(plan.grid_n),
        static_cast<int32_t>(plan.tiles), static_cast<int32_t>(plan.k_blocks), args.wait_limit_ns,
        args.err_word);
    return cudaGetLastError();
}

}  // namespace

int g_force_tile_n = 0;

GemmPlan plan_gemm(int64_t M, int64_t N, int64_t K, int num_sms) {
    const int64_t sms = num_sms > 0 ? num_sms : 1;
    const GemmPlan cands[3] = {plan_for<Cfg256>(M, N, K, sms), plan_for<Cfg224>(M, N, K, sms),
                               plan_for<Cfg192>(M, N, K, sms)};
    const int forced = __atomic_load_n(&g_force_tile_n, __ATOMIC_ACQUIRE);
    GemmPlan best = cands[0];
    for (const GemmPlan& c : cands) {
        if (forced != 0) {
            if (c.bn == forced) return c;
            continue;
        }
        if (plan_cost(c) < plan_cost(best)) best = c;
    }
    return best;
}

cudaError_t launch_gemm_tn(const GemmPlan& plan, const CUtensorMap& tmA, const CUtensorMap& tmB,
                           const CUtensorMap& tmD, const GemmArgs& args, cudaStream_t stream) {
    switch (plan.bn) {
        case 256: return launch_cfg<Cfg256>(plan, tmA, tmB, tmD, args, stream);
        case 224: return launch_cfg<Cfg224>(plan, tmA, tmB, tmD, args, stream);
        case 192: return launch_cfg<Cfg192>(plan, tmA, tmB, tmD, args, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace tmagemm
