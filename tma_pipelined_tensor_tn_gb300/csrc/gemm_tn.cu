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
// CTA pairs (PAIR): the two CTAs of a pair (cluster ranks 2p, 2p + 1) run one
// 256-row tile with cta_group::2 MMAs issued by the first; each holds its
// 128 rows of A and half of B, so per SM the B traffic halves.  The tile
// order visits groups of GROUP_M tile rows; the plan picks GROUP_M per shape
// (row order when A, B and D fit in L2).
//
// Cluster split (CK): for few-tile shapes the CTAs (or pairs) of a cluster
// compute one tile over separate K ranges and add their FP32 accumulators
// through distributed shared memory before writing D (no workspace).
//
// Ragged M/N/K: TMA zero-fills out-of-range operand elements (the .zfill rule
// of "高级数据搬运…", 零填充) and clamps out-of-range stores, so interior and
// edge tiles run the same code.
//
// Split-K: the same kernel runs work units (tile, k-split).  With FP32 output
// (OUT_F32) each unit stores its partial accumulator to a caller-provided
// workspace [splits][M][N] through a 3-D tensor map, and splitk_reduce sums the
// partials in split order and rounds to fp16 ("Learning TileLang with GEMV",
// §5.2 block_split_k: partial sums across blocks need an FP32 destination and
// one final conversion).  The reduction order is fixed, so results are
// deterministic.
//
// Every mbarrier wait is bounded (see ptx.cuh): on a timeout the CTA raises a
// shared abort flag, all roles leave their loops, in-flight TMA loads and
// MMAs are drained, TMEM is freed, and the error word records the site.
#include <cuda.h>
#include <cuda_runtime.h>
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <vector>

#include "launch.h"
#include "ptx.cuh"
#include "tile_sched.cuh"

namespace tmagemm {

namespace {

#ifndef TMAGEMM_L2_WARMUP
#define TMAGEMM_L2_WARMUP 1
#endif
// Prefetch of each CTA's first k-blocks into L2 before the dependency wait.
constexpr bool kL2WarmUp = TMAGEMM_L2_WARMUP != 0;


template <int BN_, int EPI_COLS_, int STAGES_, bool OUT_F32_, bool BF16_, int TMEM_COLS_ = 512,
          int CTAS_PER_SM_ = 1, bool PAIR_ = false, int CK_ = 0, int A_ROWS_ = 128>
struct Cfg {
    static constexpr int BM = 128, BN = BN_, BK = 64, STAGES = STAGES_;
    // PAIR: a cluster of two CTAs runs one 256 x BN tile with cta_group::2
    // MMAs; each CTA holds its 128 rows of A and BN/2 rows of B.
    static constexpr bool kPair = PAIR_;
    // CK (2, 4 or 8): the CTAs of a CK-CTA cluster own one output tile and one
    // K slice each; they add their FP32 accumulators through distributed
    // shared memory and write D directly (one unit per CTA, no workspace).
    static constexpr int kClusterK = CK_;
    static constexpr int kTileM = PAIR_ ? 256 : 128;       // rows of one work tile
    static constexpr int kBRows = PAIR_ ? BN_ / 2 : BN_;  // rows of B in this CTA
    static constexpr bool kOutF32 = OUT_F32_;
    static constexpr bool kBF16 = BF16_;           // operands (and D) bf16 instead of fp16
    static constexpr int kThreads = 192;            // 6 warps
    static constexpr int kEpiThreads = 128;         // warps 2..5
    // One store box row is one swizzle span: 32 or 64 fp16 columns, or 32 fp32
    // (16 fp32 when the whole tile is only 16 columns wide).
    static constexpr int kEpiCols = OUT_F32_ ? (BN_ < 32 ? BN_ : 32) : EPI_COLS_;
    static constexpr uint32_t kEpiElemBytes = OUT_F32_ ? 4 : 2;
    static constexpr uint32_t kEpiRowBytes = kEpiCols * kEpiElemBytes;
    static constexpr uint32_t kEpiChunks = kEpiRowBytes / 16;    // 16-byte chunks per box row
    static constexpr int kGroupM = 8;   // L2 group height in tiles (grouped GEMM; dense: per plan)
    // A_ROWS < 128 (problems of at most A_ROWS rows): a stage holds only
    // A_ROWS rows of A, so more stages fit.  The 128-row MMA still reads 128
    // rows from the stage's A address; rows past A_ROWS fall on the start of
    // the same stage's B box (landed with it) and reach only accumulator rows
    // >= M, which are never stored.
    static constexpr int kARows = A_ROWS_;
    static constexpr uint32_t kABytes = kARows * BK * 2;
    static constexpr uint32_t kBBytes = kBRows * BK * 2;
    static constexpr uint32_t kStageBytes = kABytes + kBBytes;
    static constexpr uint32_t kEpiBufBytes = BM * kEpiRowBytes;
    static constexpr int kEpiBufs = CK_ ? 0 : 2;   // cluster splits write D without TMA
    // Two accumulators, kAccStride columns apart, in kTmemCols allocated
    // columns (a power of two >= 32; CTAS_PER_SM CTAs must fit in 512).
    static constexpr uint32_t kTmemCols = TMEM_COLS_;
    static constexpr uint32_t kAccStride = TMEM_COLS_ / 2;
    static constexpr int kCtasPerSm = CTAS_PER_SM_;
    // Stage s: its A box at kOffA + s * kStageBytes, its B box right after.
    static constexpr uint32_t kOffA = 0;
    static constexpr uint32_t kOffD = kOffA + STAGES * kStageBytes;
    static constexpr uint32_t kOffBar = kOffD + kEpiBufs * kEpiBufBytes;
    static constexpr uint32_t kNumBars = 2 * STAGES + 5;
    static constexpr uint32_t kOffMisc = kOffBar + kNumBars * 8;
    static constexpr uint32_t kSmemBytes = kOffMisc + 16 + 1024;   // + base alignment slack
    // Cluster split: this CTA's 128 x BN FP32 partial tile, row stride BN + 4
    // floats (conflict-free 16-byte stores), over the stages once the
    // mainloop is done.
    static constexpr uint32_t kPartStride = BN + 4;
    static constexpr uint32_t kIdesc = umma_idesc_16bit_f32(kTileM, BN, BF16_);
    // Tail split: a tile of the last, partly filled round of the schedule may
    // run as two units of kNarrowCols and BN - kNarrowCols columns (whole
    // store boxes; MMA N a multiple of 16), so that round takes about half as
    // long.  A narrow unit's B box has kNarrowBRows rows in this CTA.
    static constexpr int kNarrowStep = kEpiCols > 16 ? kEpiCols : 16;
    static constexpr int kNarrowCols = (BN_ / 2 + kNarrowStep - 1) / kNarrowStep * kNarrowStep;
    static constexpr int kNarrowBRows = PAIR_ ? kNarrowCols / 2 : kNarrowCols;
    static constexpr uint32_t kNarrowBBytes = kNarrowBRows * BK * 2;
    static constexpr bool kTailSplit = !OUT_F32_ && CK_ == 0 && kNarrowCols < BN_ &&
                                       kNarrowBRows % 8 == 0 &&
                                       ((BN_ - kNarrowCols) / (PAIR_ ? 2 : 1)) % 8 == 0;
    // Units narrower than BN (tail-split parts, transposed grouped blocks):
    // their MMA N and store boxes follow the unit.
    static constexpr bool kVarCols = !OUT_F32_ && CK_ == 0;

    static_assert(BK * 2 == 128, "a K-major row of one k-block is one 128-byte swizzle atom");
    static_assert(BN % 16 == 0 && BN >= 16 && BN <= 256, "UMMA N for M = 128");
    static_assert(CK_ != 0 || kEpiRowBytes == 64 || kEpiRowBytes == 128,
                  "store boxes are 64 or 128 bytes wide (cluster splits store without them)");
    static_assert(kEpiCols % 16 == 0 && BN % kEpiCols == 0, "epilogue boxes tile BN");
    static_assert(kAccStride + BN <= kTmemCols, "two accumulators fit in TMEM");
    static_assert(kABytes % 1024 == 0 && kBBytes % 1024 == 0, "stages stay 1024-B aligned");
    static_assert(kARows == BM || (kARows % 16 == 0 && kARows < BM && !PAIR_ &&
                                   uint32_t(BM - kARows) * BK * 2 <= kBBytes),
                  "a short A box: the MMA's rows past it stay inside the stage");
    static_assert(kEpiBufBytes % 1024 == 0, "epilogue boxes stay 1024-B aligned");
    static_assert(kSmemBytes <= 232448, "fits the 227 KB opt-in shared memory");
    static_assert(kTmemCols * CTAS_PER_SM_ <= 512, "resident CTAs share the SM's 512 TMEM columns");
    static_assert(!PAIR_ || (CTAS_PER_SM_ == 1 && !OUT_F32_ && kBRows % 8 == 0),
                  "pairs: one CTA per SM, plain output, whole 8-row swizzle atoms of B");
    static_assert(CTAS_PER_SM_ == 1 || kSmemBytes * CTAS_PER_SM_ <= 232448,
                  "resident CTAs share the SM's shared memory");
    static_assert(CK_ == 0 || ((CK_ == 2 || CK_ == 4 || (CK_ == 8 && !PAIR_)) && !OUT_F32_ &&
                               CTAS_PER_SM_ == 1 && BN % 8 == 0 &&
                               BM * kPartStride * 4 <= STAGES * kStageBytes),
                  "cluster split: fp16/bf16 D, at most 8 CTAs, partial tile within the stages");
};

// Tile shapes the host plan chooses from (all 128 rows x BN columns x 64 K),
// for fp16 (T = false) and bf16 (T = true) operands.
template <bool T> using Cfg256 = Cfg<256, 64, 4, false, T>;
template <bool T> using Cfg224 = Cfg<224, 32, 4, false, T>;
template <bool T> using Cfg192 = Cfg<192, 64, 4, false, T>;
// Split-K partial-tile variants (FP32 output boxes of 32 columns).
template <bool T> using Cfg256F = Cfg<256, 32, 4, true, T>;
template <bool T> using Cfg224F = Cfg<224, 32, 4, true, T>;
template <bool T> using Cfg192F = Cfg<192, 32, 4, true, T>;

// Swap-AB tiles for skinny GEMMs (M = 2..64 rows of activations): the weight
// matrix is the 128-row "A" operand, the activations the narrow "B" operand,
// so the MMA is 128 x Mp x 16 with Mp in {16, 32, 64}.  Stages are small, so
// the ring is deeper to keep more of the weight stream in flight.
// CTA-pair tiles (256 x BN) for the plain fp16/bf16 GEMM.
template <bool T> using CfgP256 = Cfg<256, 64, 6, false, T, 512, 1, true>;
template <bool T> using CfgP224 = Cfg<224, 32, 6, false, T, 512, 1, true>;
template <bool T> using CfgP192 = Cfg<192, 64, 6, false, T, 512, 1, true>;
// Cluster split-K tiles: 128 x 256 single CTAs (CK CTAs per tile), or 256 x 256
// CTA pairs (CK pairs, 2 CK CTAs per cluster; ranks 2p and 2p + 1 form pair p).
template <bool T, int CK> using CfgCK256 = Cfg<256, 64, 4, false, T, 512, 1, false, CK>;
template <bool T, int CK> using CfgPCK256 = Cfg<256, 64, 6, false, T, 512, 1, true, CK>;
// Narrower cluster-split tiles for outputs with only a few tile rows (a few
// tokens against a wide weight matrix): more tiles, so more CTAs stream the
// weights at once within the device's cluster co-residency (GB300 holds 15
// clusters of 8 CTAs at ~200 KB each, 36 of 4, 76 of 2), with deeper rings.
template <bool T, int CK> using CfgCK128 = Cfg<128, 64, 6, false, T, 256, 1, false, CK>;
template <bool T, int CK> using CfgCK192 = Cfg<192, 64, 5, false, T, 512, 1, false, CK>;
// Decode-sized cluster split (at most 64 rows of A, so a stage holds a
// 64-row A box): the 128-wide 4-CTA tiles with a 9-stage ring instead of 6,
// half again as many weight bytes in flight per SM.
template <bool T> using CfgCKD128 = Cfg<128, 64, 9, false, T, 256, 1, false, 4, 64>;

// Two CTAs per SM (each with half the ring and 128 TMEM columns) keep two
// independent weight streams per SM in flight.
using CfgS16 = Cfg<16, 16, 5, true, false, 128, 2>;
using CfgS32 = Cfg<32, 32, 4, true, false, 128, 2>;
using CfgS64 = Cfg<64, 32, 3, true, false, 128, 2>;

// What one work unit needs: operand row coordinates, its k-block range and
// where its output box goes.
struct UnitInfo {
    int32_t a_row, b_row;    // TMA row coordinates of the A and B tiles
    int32_t kb0, kb1;        // k-blocks [kb0, kb1)
    int32_t store_y;         // output row coordinate (in the store map)
    int32_t store_z;         // split index (split-K) or group index (grouped)
    int32_t n_limit;         // columns >= n_limit are outside the output
    int32_t m_limit;         // rows >= m_limit are outside the output (store map rows)
    int32_t cols;            // output columns of this unit (BN, or a tail-split part)
    int32_t narrow;          // 1: a tail-split part (B through the narrow box)
};

// Dense problem: D (or split-K partials) = A * B^T.  Unit u < full_units
// covers output tile u % num_tiles and k-blocks [split * kb_per_unit,
// min(k_blocks, ...)) with split = u / num_tiles (without split-K,
// kb_per_unit = k_blocks); the units after full_units are the column parts
// of the tail-split tiles, over all of K.
struct Work {
    int32_t M, N, grid_m, grid_n, num_tiles, num_units, k_blocks, kb_per_unit;
    int32_t group_m;   // L2 group height in tiles (chosen by the plan)
    int32_t a_box_rows;   // rows of each A box (the A part of a stage's bytes)
    // Tail split: units < full_units are whole tiles; unit full_units + 2 t + p
    // is part p of tile full_units + t, columns [0, narrow_cols) for p = 0 and
    // [narrow_cols, BN) for p = 1.  narrow_cols = 0 (and full_units =
    // num_units): no tail split.
    int32_t full_units, narrow_cols;
    int32_t narrow_b_bytes;   // bytes of one stage's B box for a narrow unit (per CTA)
};

struct DenseProblem {
    static constexpr bool kTransposed = false;   // D tiles stored as computed
    CUtensorMap tmA, tmB, tmD;
    CUtensorMap tmBn;   // B with the narrow box of tail-split parts
    Work w;
    void* d_out;   // D itself (M x N, row-major), for the cluster-split epilogue

    __device__ __forceinline__ int32_t num_units() const { return w.num_units; }
    // Bytes one stage's B box brings for this unit (per CTA); `full` for a whole box.
    __device__ __forceinline__ uint32_t b_box_bytes(const UnitInfo& ui, int,
                                                    uint32_t full) const {
        return ui.narrow ? static_cast<uint32_t>(w.narrow_b_bytes) : full;
    }
    // Bytes one stage's A box brings (the rest of the A stage is not written).
    __device__ __forceinline__ uint32_t a_box_bytes(int BK) const {
        return static_cast<uint32_t>(w.a_box_rows) * static_cast<uint32_t>(BK) * 2u;
    }
    __device__ __forceinline__ void prefetch() const {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
        tma_prefetch_desc(&tmD);
        if (w.narrow_cols > 0) tma_prefetch_desc(&tmBn);
    }
    // L2 warm-up of one k-block of this CTA's A and B rows (row offsets
    // row_a and row_b into the unit's tiles).
    __device__ __forceinline__ void prefetch_l2(int32_t k, const UnitInfo& ui, int32_t row_a,
                                                int32_t row_b) const {
        tma_prefetch_l2_2d(&tmA, k, ui.a_row + row_a);
        tma_prefetch_l2_2d(ui.narrow ? &tmBn : &tmB, k, ui.b_row + row_b);
    }
    __device__ __forceinline__ UnitInfo unit(int32_t u, int BM, int BN, int) const {
        int32_t tile, split = 0, part = -1;
        if (u < w.full_units) {
            tile = u % w.num_tiles;
            split = u / w.num_tiles;
        } else {
            tile = w.full_units + ((u - w.full_units) >> 1);
            part = (u - w.full_units) & 1;
        }
        const TileCoord tc = tile_coord(tile, w.grid_m, w.grid_n, w.group_m);
        UnitInfo ui;
        ui.a_row = tc.m_blk * BM;
        ui.b_row = tc.n_blk * BN + (part == 1 ? w.narrow_cols : 0);
        ui.cols = part < 0 ? BN : (part == 0 ? w.narrow_cols : BN - w.narrow_cols);
        ui.narrow = part >= 0 ? 1 : 0;
        ui.kb0 = split * w.kb_per_unit;
        ui.kb1 = min(w.k_blocks, ui.kb0 + w.kb_per_unit);
        ui.store_y = ui.a_row;
        ui.store_z = split;
        ui.n_limit = w.N;
        ui.m_limit = w.M;
        return ui;
    }
    __device__ __forceinline__ void load_a(uint32_t dst, int32_t k, const UnitInfo& ui,
                                           uint32_t bar) const {
        tma_load_2d(dst, &tmA, k, ui.a_row, bar);
    }
    __device__ __forceinline__ void load_b(uint32_t dst, int32_t k, const UnitInfo& ui,
                                           uint32_t bar) const {
        tma_load_2d(dst, ui.narrow ? &tmBn : &tmB, k, ui.b_row, bar);
    }
    // Pair forms: this CTA's rows (unit row + offset), bytes counted on the
    // leader's barrier (cluster address).
    __device__ __forceinline__ void load_a_pair(uint32_t dst, int32_t k, const UnitInfo& ui,
                                                int32_t row_off, uint32_t bar_cluster) const {
        tma_load_2d_pair(dst, &tmA, k, ui.a_row + row_off, bar_cluster);
    }
    __device__ __forceinline__ void load_b_pair(uint32_t dst, int32_t k, const UnitInfo& ui,
                                                int32_t row_off, uint32_t bar_cluster) const {
        tma_load_2d_pair(dst, ui.narrow ? &tmBn : &tmB, k, ui.b_row + row_off, bar_cluster);
    }
    template <bool kOutF32>
    __device__ __forceinline__ void store(uint32_t buf, int32_t x, int32_t y,
                                          const UnitInfo& ui) const {
        if constexpr (kOutF32)
            tma_store_3d(&tmD, buf, x, y, ui.store_z);
        else
            tma_store_2d(&tmD, buf, x, y);
    }
};

// Grouped problem: G independent GEMMs sharing N and K, with the rows of
// group g at [m_off[g], m_off[g+1]) of one A and one D, and B holding G
// stacked N x K matrices — the "window at a run-time origin" of the Croqtile
// chapter ("任意偏移窗口：view 与 from": the pipeline is unchanged, only the
// origin moves).  A is one 2-D map over all rows (a tile may read rows of the
// next group; they only reach output rows that are not stored), B a 3-D map
// {K, N, G} (clamps N per group), D one 2-D map per group, so a store never
// crosses the group's last row.
constexpr int kMaxGroups = 64;

struct GroupedProblem {
    static constexpr bool kTransposed = false;
    CUtensorMap tmA, tmB;
    CUtensorMap tmD[kMaxGroups];
    int32_t tile_start[kMaxGroups + 1];   // prefix sums of the groups' tile counts
    int32_t m_off[kMaxGroups + 1];        // row offsets; m_off[groups] = all rows
    int32_t groups, grid_n, N, k_blocks;

    __device__ __forceinline__ int32_t num_units() const { return tile_start[groups]; }
    __device__ __forceinline__ uint32_t b_box_bytes(const UnitInfo&, int, uint32_t full) const {
        return full;   // no narrow units
    }
    __device__ __forceinline__ uint32_t a_box_bytes(int BK) const {
        return 128u * static_cast<uint32_t>(BK) * 2u;
    }
    __device__ __forceinline__ void prefetch() const {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
    }
    __device__ __forceinline__ void prefetch_l2(int32_t k, const UnitInfo& ui, int32_t row_a,
                                                int32_t row_b) const {
        tma_prefetch_l2_2d(&tmA, k, ui.a_row + row_a);
        tma_prefetch_l2_3d(&tmB, k, ui.b_row + row_b, ui.store_z);
    }
    __device__ __forceinline__ UnitInfo unit(int32_t u, int BM, int BN, int group_m) const {
        int32_t g = 0;
        while (g + 1 < groups && tile_start[g + 1] <= u) ++g;
        const int32_t local = u - tile_start[g];
        const int32_t rows = m_off[g + 1] - m_off[g];
        const int32_t gm = (rows + BM - 1) / BM;
        const TileCoord tc = tile_coord(local, gm, grid_n, group_m);
        UnitInfo ui;
        ui.a_row = m_off[g] + tc.m_blk * BM;
        ui.b_row = tc.n_blk * BN;
        ui.kb0 = 0;
        ui.kb1 = k_blocks;
        ui.store_y = tc.m_blk * BM;
        ui.store_z = g;
        ui.n_limit = N;
        ui.m_limit = rows;
        ui.cols = BN;
        ui.narrow = 0;
        return ui;
    }
    __device__ __forceinline__ void load_a(uint32_t dst, int32_t k, const UnitInfo& ui,
                                           uint32_t bar) const {
        tma_load_2d(dst, &tmA, k, ui.a_row, bar);
    }
    __device__ __forceinline__ void load_b(uint32_t dst, int32_t k, const UnitInfo& ui,
                                           uint32_t bar) const {
        tma_load_3d(dst, &tmB, k, ui.b_row, ui.store_z, bar);
    }
    __device__ __forceinline__ void load_a_pair(uint32_t dst, int32_t k, const UnitInfo& ui,
                                                int32_t row_off, uint32_t bar_cluster) const {
        tma_load_2d_pair(dst, &tmA, k, ui.a_row + row_off, bar_cluster);
    }
    __device__ __forceinline__ void load_b_pair(uint32_t dst, int32_t k, const UnitInfo& ui,
                                                int32_t row_off, uint32_t bar_cluster) const {
        tma_load_3d_pair(dst, &tmB, k, ui.b_row + row_off, ui.store_z, bar_cluster);
    }
    template <bool kOutF32>
    __device__ __forceinline__ void store(uint32_t buf, int32_t x, int32_t y,
                                          const UnitInfo& ui) const {
        tma_store_2d(&tmD[ui.store_z], buf, x, y);
    }
};

// Grouped problem, transposed: each group is computed as D_g^T = B_g A_g^T,
// so that its run-time row count becomes the MMA's N (whole 16-row steps)
// instead of a tile's 128 or 256 rows.  The weights B_g (N x K) are the
// 128-row (per CTA) operand, the group's rows of A the narrow one; the
// accumulator of a tile holds [weight row n][row t of A] and is stored
// transposed, as rows t, columns n of D: 64 rows at a time through one map
// over all of D where those rows lie inside the group, else 16 rows at a
// time through the group's own map, which clips at the group's last row.  A group's rows are cut into
// tb_count(g) blocks of nearly equal width (multiples of 16, at most maxw16 *
// 16): no block is padded by more than 15 rows.  A block of w rows loads
// only those rows of A (w / CTAs per tile per CTA), through the map for its
// width, so a narrow block moves no more bytes than it uses.  Units run group
// by group,
// and within a group a block of rows against every weight block in turn, so
// a group's weights and rows are reused from L2 while the group runs.
struct GroupedTProblem {
    static constexpr bool kTransposed = true;
    CUtensorMap tmW;                      // B as {K, N, G}, box {64, 128, 1}
    CUtensorMap tmX[16];                  // A as {K, rows}, box {64, 16 (j + 1) / x_ctas}
    CUtensorMap tmD[kMaxGroups];          // D rows of group g as {N, M_g}, box {128, 16}
    CUtensorMap tmD64;                    // all of D as {N, rows}, box {128, 64}
    int32_t tile_start[kMaxGroups + 1];   // prefix sums of the groups' unit counts
    int32_t m_off[kMaxGroups + 1];        // row offsets; m_off[groups] = all rows
    int32_t groups, n_blocks, N, k_blocks, maxw16;
    int32_t x_ctas;                       // CTAs per tile (2 for a pair): A rows per CTA = w / x_ctas
    uint32_t x_used;                      // bit j: tmX[j] (blocks of 16 (j + 1) rows) is encoded

    __device__ __forceinline__ int32_t num_units() const { return tile_start[groups]; }
    // The map of A for this unit's block width (a multiple of 16, at most 256).
    __device__ __forceinline__ const CUtensorMap* x_map(const UnitInfo& ui) const {
        return &tmX[ui.cols / 16 - 1];
    }
    __device__ __forceinline__ uint32_t b_box_bytes(const UnitInfo& ui, int BK, uint32_t) const {
        return static_cast<uint32_t>(ui.cols / x_ctas) * static_cast<uint32_t>(BK) * 2u;
    }
    __device__ __forceinline__ uint32_t a_box_bytes(int BK) const {
        return 128u * static_cast<uint32_t>(BK) * 2u;
    }
    __device__ __forceinline__ void prefetch() const {
        tma_prefetch_desc(&tmW);
        for (uint32_t m = x_used; m != 0; m &= m - 1) tma_prefetch_desc(&tmX[__ffs(m) - 1]);
        tma_prefetch_desc(&tmD64);
    }
    __device__ __forceinline__ void prefetch_l2(int32_t k, const UnitInfo& ui, int32_t row_a,
                                                int32_t row_b) const {
        tma_prefetch_l2_3d(&tmW, k, ui.a_row + row_a, ui.store_z);
        tma_prefetch_l2_2d(x_map(ui), k, ui.b_row + row_b);
    }
    __device__ __forceinline__ UnitInfo unit(int32_t u, int BM, int, int) const {
        int32_t g = 0;
        while (g + 1 < groups && tile_start[g + 1] <= u) ++g;
        const int32_t local = u - tile_start[g];
        const int32_t tb = local / n_blocks, nb = local % n_blocks;
        const int32_t rows = m_off[g + 1] - m_off[g];
        // rows in 16-row steps, cut into tb blocks of q or q + 1 steps
        const int32_t steps = (rows + 15) / 16;
        const int32_t tb_count = (steps + maxw16 - 1) / maxw16;
        const int32_t q = steps / tb_count, extra = steps % tb_count;
        UnitInfo ui;
        ui.a_row = nb * BM;                                       // weight rows (D columns)
        const int32_t t0 = 16 * (tb * q + min(tb, extra));         // first row of the block
        ui.b_row = m_off[g] + t0;
        ui.cols = 16 * (q + (tb < extra ? 1 : 0));
        ui.narrow = 0;
        ui.kb0 = 0;
        ui.kb1 = k_blocks;
        ui.store_y = t0;                                          // row in group g's D map
        ui.store_z = g;
        ui.n_limit = N;
        ui.m_limit = rows;
        return ui;
    }
    __device__ __forceinline__ void load_a(uint32_t dst, int32_t k, const UnitInfo& ui,
                                           uint32_t bar) const {
        tma_load_3d(dst, &tmW, k, ui.a_row, ui.store_z, bar);
    }
    __device__ __forceinline__ void load_b(uint32_t dst, int32_t k, const UnitInfo& ui,
                                           uint32_t bar) const {
        tma_load_2d(dst, x_map(ui), k, ui.b_row, bar);
    }
    __device__ __forceinline__ void load_a_pair(uint32_t dst, int32_t k, const UnitInfo& ui,
                                                int32_t row_off, uint32_t bar_cluster) const {
        tma_load_3d_pair(dst, &tmW, k, ui.a_row + row_off, ui.store_z, bar_cluster);
    }
    __device__ __forceinline__ void load_b_pair(uint32_t dst, int32_t k, const UnitInfo& ui,
                                                int32_t row_off, uint32_t bar_cluster) const {
        tma_load_2d_pair(dst, x_map(ui), k, ui.b_row + row_off, bar_cluster);
    }
    // A 16-row x 128-column box of D: rows y.. of group z, columns x...
    __device__ __forceinline__ void store_t16(uint32_t buf, int32_t x, int32_t y,
                                              int32_t z) const {
        tma_store_2d(&tmD[z], buf, x, y);
    }
    // A 64-row x 128-column box of D: rows y.. of all of D, columns x...
    __device__ __forceinline__ void store_t64(uint32_t buf, int32_t x, int32_t y) const {
        tma_store_2d(&tmD64, buf, x, y);
    }
};

template <class C, class P>
__global__ void __launch_bounds__(C::kThreads, C::kCtasPerSm)
gemm_tn_f16_kernel(const __grid_constant__ P prob, const uint64_t limit_ns,
                   uint32_t* __restrict__ err) {
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
    // Checked build: the k-blocks the producer issued and the MMA issuer consumed.
    volatile uint32_t* ring_count = reinterpret_cast<volatile uint32_t*>(smem + C::kOffMisc + 8);

    const int warp = __shfl_sync(0xffffffffu, static_cast<int>(threadIdx.x) / 32, 0);
    const int lane = static_cast<int>(threadIdx.x) % 32;

    // Work distribution: single CTAs step by the grid; pairs by the pair count.
    // Cluster roles: a pair is ranks (2p, 2p + 1) of the cluster; `rank` is
    // this CTA's half of its pair, `pair_leader` the pair's first rank.
    const uint32_t cta_rank = (C::kPair || C::kClusterK != 0) ? cluster_ctarank() : 0u;
    const uint32_t rank = C::kPair ? (cta_rank & 1u) : 0u;
    const uint32_t pair_leader = C::kPair ? (cta_rank & ~1u) : 0u;
    const uint16_t pair_mask = static_cast<uint16_t>(0x3u << pair_leader);
    int32_t unit0 =
        C::kPair ? static_cast<int32_t>(blockIdx.x / 2) : static_cast<int32_t>(blockIdx.x);
    int32_t unit_step =
        C::kPair ? static_cast<int32_t>(gridDim.x / 2) : static_cast<int32_t>(gridDim.x);
    // Cluster split: one unit per CTA (or pair), the tile of the cluster and
    // the K slice of this CTA's (pair's) index in it (unit = split * tiles + tile).
    uint32_t ck_rank = 0;
    if constexpr (C::kClusterK != 0) {
        ck_rank = C::kPair ? (cta_rank >> 1) : cta_rank;
        unit0 = static_cast<int32_t>(ck_rank) * prob.w.num_tiles +
                static_cast<int32_t>(blockIdx.x / (C::kClusterK * (C::kPair ? 2 : 1)));
        unit_step = prob.num_units();
    }

    // The next grid on the stream may be scheduled as soon as every CTA of
    // this one is running: it cannot share an SM with this grid's CTAs (shared
    // memory), and it waits (below) before touching global memory.
    grid_launch_dependents();

    // ---- one-time setup: barriers (warp 0), TMEM (warp 1) ----
    if (warp == 0) {
        if (elect_one()) {
            for (uint32_t s = 0; s < (uint32_t)C::STAGES; ++s) {
                mbar_init(full_bar(s), 1);
                mbar_init(empty_bar(s), 1);
            }
            for (uint32_t a = 0; a < 2; ++a) {
                mbar_init(acc_full_bar(a), 1);
                // The leader's acc_empty collects the epilogue warps of both CTAs.
                mbar_init(acc_empty_bar(a), (C::kPair ? 2 : 1) * C::kEpiThreads / 32);
            }
            mbar_init(mma_done_bar, 1);
            *abort_flag = 0;
            if constexpr (kChecked) {
                ring_count[0] = 0;
                ring_count[1] = 0;
            }
            fence_mbarrier_init();
            prob.prefetch();
            // While the previous grid finishes, warm L2 with this CTA's first
            // k-blocks (a prefetch cannot see stale data: L2 is where global
            // memory is coherent), so the first loads after the wait hit L2.
            if (kL2WarmUp && unit0 < prob.num_units()) {
                const UnitInfo ui = prob.unit(unit0, C::kTileM, C::BN, C::kGroupM);
                const int32_t kb_end = min(ui.kb1, ui.kb0 + C::STAGES);
                for (int32_t kb = ui.kb0; kb < kb_end; ++kb)
                    prob.prefetch_l2(kb * C::BK, ui, static_cast<int32_t>(rank) * C::BM,
                                     static_cast<int32_t>(rank) * (ui.cols / 2));
            }
        }
        __syncwarp();
    }
    // TMEM is this CTA's own: allocating it before the previous grid has
    // completed is safe (a CTA of that grid still on this SM only delays the
    // allocation until it frees its columns; it never waits on this grid), so
    // the whole set-up runs under the previous grid's tail.
    if (warp == 1) {
        if constexpr (C::kPair) {
            tmem_alloc_pair(smem_u32(tmem_holder), C::kTmemCols);
            tmem_relinquish_pair();
        } else {
            tmem_alloc(smem_u32(tmem_holder), C::kTmemCols);
            tmem_relinquish();
        }
    }
    tc_fence_before();
    __syncthreads();
    // A pair's barriers must be initialised, and both CTAs' TMEM allocated,
    // before the peer's TMA, MMA or commits can reach them.
    if constexpr (C::kPair) cluster_sync_after_init();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;
    // A, B and D are only touched once the grid before this one on the
    // stream has completed.
    grid_dependency_wait();

    if (warp == 0) {
        // ================= TMA producer =================
        if (elect_one()) {
            uint32_t it = 0;
            bool ok = true;
            for (int32_t u = unit0; ok && u < prob.num_units(); u += unit_step) {
                const UnitInfo ui = prob.unit(u, C::kTileM, C::BN, C::kGroupM);
                // A pair's B rows: this CTA's half of the unit's columns.
                const uint32_t b_bytes =
                    C::kVarCols ? prob.b_box_bytes(ui, C::BK, C::kBBytes) : C::kBBytes;
                const int32_t b_off = static_cast<int32_t>(rank) * (ui.cols / 2);
                for (int32_t kb = ui.kb0; kb < ui.kb1; ++kb) {
                    const uint32_t s = ring_stage(it, C::STAGES);
                    const uint32_t ph = ring_phase(it, C::STAGES);
                    if (!wait_or_abort(empty_bar(s), ph ^ 1u, abort_flag, err, kSiteProducerEmpty,
                                       limit_ns)) {
                        ok = false;
                        break;
                    }
                    if (!check_ok(((kb * C::BK) & 7) == 0 && ui.a_row >= 0 && ui.b_row >= 0, err,
                                  kSiteCheckTma)) {
                        *abort_flag = 1;
                        ok = false;
                        break;
                    }
                    if constexpr (C::kPair) {
                        // Both CTAs' bytes land on the leader's full[s]; only the
                        // leader registers them (its single arrival completes
                        // the phase once all bytes of both CTAs are in).
                        if (rank == 0)
                            mbar_arrive_expect_tx(full_bar(s),
                                                  2 * (prob.a_box_bytes(C::BK) + b_bytes));
                        const uint32_t leader_full = map_to_rank(full_bar(s), pair_leader);
                        const uint32_t stage = sbase + C::kOffA + s * C::kStageBytes;
                        prob.load_a_pair(stage, kb * C::BK, ui,
                                         static_cast<int32_t>(rank) * C::BM, leader_full);
                        prob.load_b_pair(stage + C::kABytes, kb * C::BK, ui, b_off, leader_full);
                    } else {
                        mbar_arrive_expect_tx(full_bar(s), prob.a_box_bytes(C::BK) + b_bytes);
                        const uint32_t stage = sbase + C::kOffA + s * C::kStageBytes;
                        prob.load_a(stage, kb * C::BK, ui, full_bar(s));
                        prob.load_b(stage + C::kABytes, kb * C::BK, ui, full_bar(s));
                    }
                    ++it;
                }
            }
            if constexpr (kChecked) ring_count[0] = it;
            // Drain: the last (up to) STAGES issued stages must have landed
            // before shared memory is released.  In a pair the leader's full
            // barriers count both CTAs' loads; the peer stays until the final
            // cluster barrier.
            if (rank == 0) {
                const uint32_t first = it > (uint32_t)C::STAGES ? it - C::STAGES : 0u;
                for (uint32_t j = first; j < it; ++j)
                    wait_bounded(full_bar(ring_stage(j, C::STAGES)), ring_phase(j, C::STAGES), err,
                                 kSiteDrainFull, limit_ns);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ================= MMA issuer (the leader's, for a pair) =================
        if (rank == 0 && elect_one()) {
            uint32_t it = 0, tcount = 0;
            bool ok = true;
            for (int32_t u = unit0; ok && u < prob.num_units(); u += unit_step, ++tcount) {
                const UnitInfo ui = prob.unit(u, C::kTileM, C::BN, C::kGroupM);
                const int32_t kb0 = ui.kb0;
                const int32_t kb1 = ui.kb1;
                // A narrow unit is an MMA of its own width (N = its columns).
                const uint32_t idesc =
                    C::kVarCols && ui.cols != C::BN
                        ? umma_idesc_16bit_f32(C::kTileM, static_cast<uint32_t>(ui.cols), C::kBF16)
                        : C::kIdesc;
                const uint32_t acc = tcount & 1u;
                const uint32_t acc_ph = (tcount >> 1) & 1u;
                if (!wait_or_abort(acc_empty_bar(acc), acc_ph ^ 1u, abort_flag, err,
                                   kSiteMmaAccEmpty, limit_ns))
                    break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * C::kAccStride;
                for (int32_t kb = kb0; kb < kb1; ++kb) {
                    const uint32_t s = ring_stage(it, C::STAGES);
                    const uint32_t ph = ring_phase(it, C::STAGES);
                    if (!wait_or_abort(full_bar(s), ph, abort_flag, err, kSiteMmaFull, limit_ns)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_addr = sbase + C::kOffA + s * C::kStageBytes;
                    const uint32_t b_addr = a_addr + C::kABytes;
#pragma unroll
                    for (int j = 0; j < C::BK / 16; ++j) {
                        const uint64_t ad = umma_desc_sw128_kmajor(a_addr + 32u * j);
                        const uint64_t bd = umma_desc_sw128_kmajor(b_addr + 32u * j);
                        const uint32_t accum = (kb != kb0 || j != 0) ? 1u : 0u;
                        if constexpr (C::kPair)
                            mma_f16_ss_pair(d_tmem, ad, bd, idesc, accum);
                        else
                            mma_f16_ss(d_tmem, ad, bd, idesc, accum);
                    }
                    // stage s free (in both CTAs of a pair) once these MMAs finish
                    if constexpr (C::kPair)
                        mma_commit_pair(empty_bar(s), pair_mask);
                    else
                        mma_commit(empty_bar(s));
                    ++it;
                }
                if (!ok) break;
                // accumulator ready for the epilogue (of both CTAs of a pair)
                if constexpr (C::kPair)
                    mma_commit_pair(acc_full_bar(acc), pair_mask);
                else
                    mma_commit(acc_full_bar(acc));
            }
            if constexpr (kChecked) ring_count[1] = it;
            // All issued MMAs must finish before TMEM is released.
            if constexpr (C::kPair)
                mma_commit_pair(mma_done_bar, static_cast<uint16_t>(0x1u << pair_leader));
            else
                mma_commit(mma_done_bar);
            wait_bounded(mma_done_bar, 0, err, kSiteDrainMma, limit_ns);
        }
        __syncwarp();
    } else if constexpr (C::kClusterK != 0) {
        // ============ cluster split: accumulator -> this CTA's partial tile ============
        const uint32_t quarter = static_cast<uint32_t>(warp) & 3u;   // TMEM lane quarter
        const uint32_t row = quarter * 32u + static_cast<uint32_t>(lane);
        const bool ok = wait_or_abort(acc_full_bar(0), 0, abort_flag, err, kSiteEpiAccFull,
                                      limit_ns);
        // A warp whose 32 rows all lie past the last row of D (index >= M)
        // holds nothing the reduction reads: it skips the copy.
        const UnitInfo ui0 = prob.unit(unit0, C::kTileM, C::BN, C::kGroupM);
        const bool rows_exist = ui0.a_row + static_cast<int32_t>(rank) * C::BM +
                                    static_cast<int32_t>(quarter) * 32 < prob.w.M;
        if (named_bar_and(1, C::kEpiThreads, ok) && rows_exist) {
            tc_fence_after();
            const uint32_t t_row = tmem_base + ((quarter * 32u) << 16);
            const uint32_t p_row = sbase + C::kOffA + row * C::kPartStride * 4u;
            // Up to four 32-column loads in flight per wait: the copy sits
            // between the last MMA and the cluster's reduction.
            constexpr int kLoads = C::BN / 32;
            constexpr int kBatch = kLoads < 4 ? kLoads : 4;
#pragma unroll 1
            for (int c0 = 0; c0 < kLoads; c0 += kBatch) {
                uint32_t v[kBatch][32];
#pragma unroll
                for (int b = 0; b < kBatch; ++b)
                    if (c0 + b < kLoads) tmem_ld_32x32b_x32(t_row + 32 * (c0 + b), v[b]);
                tmem_ld_wait();
#pragma unroll
                for (int b = 0; b < kBatch; ++b) {
                    if (c0 + b >= kLoads) break;
                    const uint32_t c = static_cast<uint32_t>(c0 + b);
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        st_shared_v4(p_row + (32u * c + 4u * j) * 4u, v[b][4 * j],
                                     v[b][4 * j + 1], v[b][4 * j + 2], v[b][4 * j + 3]);
                }
            }
            if constexpr (C::BN % 32 != 0) {
                // The last 16 columns of a tile whose width is an odd multiple of 16.
                constexpr uint32_t c0 = C::BN / 32 * 32;
                uint32_t v[16];
                tmem_ld_32x32b_x16(t_row + c0, v);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    st_shared_v4(p_row + (c0 + 4u * j) * 4u, v[4 * j], v[4 * j + 1], v[4 * j + 2],
                                 v[4 * j + 3]);
            }
        }
    } else {
        // ================= epilogue (warps 2..5) =================
        const uint32_t quarter = static_cast<uint32_t>(warp) & 3u;   // TMEM lane quarter
        const uint32_t row = quarter * 32u + static_cast<uint32_t>(lane);  // row in tile
        const bool store_thread = threadIdx.x == 64;   // the transposed form's store thread
        uint32_t tcount = 0, box = 0;
        for (int32_t u = unit0; u < prob.num_units(); u += unit_step, ++tcount) {
            UnitInfo ui = prob.unit(u, C::kTileM, C::BN, C::kGroupM);
            if constexpr (!P::kTransposed)
                ui.store_y += static_cast<int32_t>(rank) * C::BM;   // this CTA's 128 rows
            const int32_t n0 = ui.b_row;
            const uint32_t acc = tcount & 1u;
            const uint32_t acc_ph = (tcount >> 1) & 1u;
            bool ok = wait_or_abort(acc_full_bar(acc), acc_ph, abort_flag, err, kSiteEpiAccFull,
                                    limit_ns);
            // All 128 epilogue threads take the same decision.
            if (!named_bar_and(1, C::kEpiThreads, ok)) break;
            tc_fence_after();
            const uint32_t t_row = tmem_base + ((quarter * 32u) << 16) + acc * C::kAccStride;
            // Whole accumulator read: give it back to the MMA warp.
            auto release_acc = [&]() {
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    if constexpr (C::kPair)
                        mbar_arrive_cluster(map_to_rank(acc_empty_bar(acc), pair_leader));
                    else
                        mbar_arrive(acc_empty_bar(acc));
                }
            };
            if constexpr (P::kTransposed) {
                // The accumulator is [weight row n][row t of A]: a chunk is up
                // to 64 rows of D by this CTA's 128 columns, staged as rows of
                // 256 bytes (unswizzled), row t holding column n = `row` at
                // byte 2n, written by this thread from accumulator column t.
                static_assert(C::kEpiBufBytes >= 64 * 256, "a 64-row chunk fits a store buffer");
                const int32_t x = ui.a_row + static_cast<int32_t>(rank) * C::BM;
#pragma unroll 1
                for (int c0 = 0; c0 < ui.cols; c0 += 64, ++box) {
                    const int n16 = min(64, ui.cols - c0) / 16;   // 16-row parts of the chunk
                    uint32_t v[64];
#pragma unroll
                    for (int h = 0; h < 4; ++h)
                        if (h < n16)
                            tmem_ld_32x32b_x16(t_row + c0 + 16 * h,
                                               *reinterpret_cast<uint32_t(*)[16]>(&v[16 * h]));
                    tmem_ld_wait();
                    if (c0 + 64 >= ui.cols) release_acc();
                    const uint32_t buf = sbase + C::kOffD + (box & 1u) * C::kEpiBufBytes;
                    if (store_thread) bulk_wait_group_read<1>();
                    named_bar_sync(1, C::kEpiThreads);
#pragma unroll
                    for (int t = 0; t < 64; ++t)
                        if (t < 16 * n16)
                            st_shared_u16(buf + static_cast<uint32_t>(t) * 256u + row * 2u,
                                          cvt16_rn<C::kBF16>(v[t]));
                    fence_proxy_async_smem();
                    named_bar_sync(1, C::kEpiThreads);
                    if (store_thread) {
                        const int32_t y = ui.store_y + c0;        // row in the group
                        if (x < ui.n_limit &&
                            check_ok((x & 7) == 0 && x >= 0 && y >= 0, err, kSiteCheckTma)) {
                            if (n16 == 4 && y + 64 <= ui.m_limit) {
                                prob.store_t64(buf, x, ui.b_row + c0);   // inside the group
                            } else {
                                for (int j = 0; j < n16 && y + 16 * j < ui.m_limit; ++j)
                                    prob.store_t16(buf + 4096u * j, x, y + 16 * j, ui.store_z);
                            }
                        }
                        bulk_commit_group();
                    }
                }
            } else {
            const int chunks = (C::kVarCols ? ui.cols : C::BN) / C::kEpiCols;
            // Box c's accumulator columns are read from TMEM one box ahead:
            // the read of box c + 1 is issued once box c's registers are in
            // shared memory, so it runs under box c's barrier and store.
            uint32_t v[C::kEpiCols];
            auto load_box = [&](int c) {
                if constexpr (C::kEpiCols == 16) {
                    tmem_ld_32x32b_x16(t_row + c * C::kEpiCols,
                                       *reinterpret_cast<uint32_t(*)[16]>(&v[0]));
                } else {
#pragma unroll
                    for (int h = 0; h < C::kEpiCols / 32; ++h)
                        tmem_ld_32x32b_x32(t_row + c * C::kEpiCols + 32 * h,
                                           *reinterpret_cast<uint32_t(*)[32]>(&v[32 * h]));
                }
            };
            load_box(0);
#pragma unroll 1
            for (int c = 0; c < chunks; ++c, ++box) {
                tmem_ld_wait();
                if (c == chunks - 1) release_acc();
                // Each epilogue warp stages and stores its own 32 rows: a
                // 32-row slice of the box buffer (whole 1024-byte swizzle
                // atoms) and one TMA store of 32 rows issued by its lane 0,
                // so the warps synchronise with nothing but themselves.
                const uint32_t buf = sbase + C::kOffD + (box & 1u) * C::kEpiBufBytes +
                                     quarter * 32u * C::kEpiRowBytes;
                // The store that last read this slice (two boxes ago) must be done.
                if (lane == 0) bulk_wait_group_read<1>();
                __syncwarp();
                // Row `lane` of the slice holds kEpiChunks 16-byte chunks.  The
                // TMA swizzle whose span equals the row width (64B or 128B)
                // XORs the chunk index with address bits 7.. of the row start:
                // chunk j of row r lands at j ^ ((r * row_bytes / 128) % chunks).
                const uint32_t row_addr = buf + static_cast<uint32_t>(lane) * C::kEpiRowBytes;
                const uint32_t xr = ((row * C::kEpiRowBytes) >> 7) & (C::kEpiChunks - 1);
#pragma unroll
                for (uint32_t j = 0; j < C::kEpiChunks; ++j) {
                    if constexpr (C::kOutF32) {
                        st_shared_v4(row_addr + ((j ^ xr) << 4), v[4 * j + 0], v[4 * j + 1],
                                     v[4 * j + 2], v[4 * j + 3]);
                    } else {
                        const uint32_t p0 = pack2_rn<C::kBF16>(v[8 * j + 0], v[8 * j + 1]);
                        const uint32_t p1 = pack2_rn<C::kBF16>(v[8 * j + 2], v[8 * j + 3]);
                        const uint32_t p2 = pack2_rn<C::kBF16>(v[8 * j + 4], v[8 * j + 5]);
                        const uint32_t p3 = pack2_rn<C::kBF16>(v[8 * j + 6], v[8 * j + 7]);
                        st_shared_v4(row_addr + ((j ^ xr) << 4), p0, p1, p2, p3);
                    }
                }
                fence_proxy_async_smem();
                if (c + 1 < chunks) load_box(c + 1);
                __syncwarp();
                if (lane == 0) {
                    const int32_t x = n0 + c * C::kEpiCols;
                    const int32_t y = ui.store_y + static_cast<int32_t>(quarter) * 32;
                    if (x < ui.n_limit && y < ui.m_limit &&
                        check_ok((x & 7) == 0 && x >= 0 && y >= 0, err, kSiteCheckTma))
                        prob.template store<C::kOutF32>(buf, x, y, ui);
                    bulk_commit_group();
                }
            }
            }   // not transposed
            if (store_thread && rank == 0) check_count_unit(err, u);
        }
        if (lane == 0) bulk_wait_group<0>();   // every lane 0 that issued stores
    }

    if constexpr (C::kClusterK != 0) {
        // Every CTA's partial tile is complete and visible cluster-wide.  The
        // outputs of the tile that exist (rows below M, 4-column groups left of
        // N) are dealt out evenly over the CK CTAs (a pair's halves reduce
        // separately: CTA (pair p, half h) adds the partials of ranks 2q + h),
        // so with a few rows every CTA of the cluster still takes a share.
        // Each 4-column group: the CK partials loaded together (consecutive
        // threads read consecutive 16 bytes of a peer's partial row, whole
        // 128-byte lines per quarter warp) and added in slice order
        // (deterministic), one 8-byte store of D; kItems groups per thread
        // have their loads in flight at once.
        tc_fence_before();
        cluster_sync();
        // The accumulator is in shared memory now: a single CTA gives its
        // TMEM back before the reduction rather than at exit.
        if constexpr (!C::kPair) {
            if (warp == 1) {
                tc_fence_after();
                tmem_dealloc(tmem_base, C::kTmemCols);
            }
        }
        constexpr int kGroups = C::BN / 4;
        constexpr int kItems = C::kClusterK <= 4 ? 4 : 2;
        constexpr uint32_t kPeerStride = C::kPair ? 2u : 1u;
        const UnitInfo ui = prob.unit(unit0, C::kTileM, C::BN, C::kGroupM);
        uint16_t* dout = static_cast<uint16_t*>(prob.d_out);
        const int32_t m0 = ui.a_row + static_cast<int32_t>(rank) * C::BM;
        const int rows = max(0, min(C::BM, prob.w.M - m0));
        // (N is a multiple of 8, so a group is either whole or outside.)
        const int groups = max(0, min(kGroups, (prob.w.N - ui.b_row + 3) / 4));
        const int total = rows * groups;
        const int f_begin = static_cast<int>(ck_rank) * total / C::kClusterK;
        const int f_end = (static_cast<int>(ck_rank) + 1) * total / C::kClusterK;
        for (int f0 = f_begin + static_cast<int>(threadIdx.x); f0 < f_end;
             f0 += kItems * C::kThreads) {
            float part[kItems][C::kClusterK][4];
#pragma unroll
            for (int it = 0; it < kItems; ++it) {
                const int f = f0 + it * C::kThreads;
                if (f >= f_end) break;
                const int rl = f / groups, g = f % groups;
                const uint32_t local = sbase + C::kOffA + (rl * C::kPartStride + 4u * g) * 4u;
#pragma unroll
                for (int q = 0; q < C::kClusterK; ++q) {
                    const uint32_t peer = kPeerStride * static_cast<uint32_t>(q) + rank;
                    ld_shared_cluster_v4(map_to_rank(local, peer), part[it][q]);
                }
            }
#pragma unroll
            for (int it = 0; it < kItems; ++it) {
                const int f = f0 + it * C::kThreads;
                if (f >= f_end) break;
                const int rl = f / groups, g = f % groups;
                float a[4] = {part[it][0][0], part[it][0][1], part[it][0][2], part[it][0][3]};
#pragma unroll
                for (int q = 1; q < C::kClusterK; ++q) {
#pragma unroll
                    for (int e = 0; e < 4; ++e) a[e] += part[it][q][e];
                }
                uint2 o;
                o.x = pack2_rn<C::kBF16>(__float_as_uint(a[0]), __float_as_uint(a[1]));
                o.y = pack2_rn<C::kBF16>(__float_as_uint(a[2]), __float_as_uint(a[3]));
                const int32_t m = m0 + rl, n = ui.b_row + 4 * g;
                if (check_ok(rl < C::BM && g < kGroups && m < prob.w.M && n + 4 <= prob.w.N, err,
                             kSiteCheckBounds))
                    *reinterpret_cast<uint2*>(dout + static_cast<int64_t>(m) * prob.w.N + n) = o;
            }
        }
        if (threadIdx.x == 0 && rank == 0 && !*abort_flag) check_count_unit(err, unit0);
        // This CTA has read its peers' partials (the loads above returned
        // before their sums were stored): arrive now; the matching wait, just
        // before exit, keeps every CTA's shared memory alive until all have
        // read it, and the stores and teardown run meanwhile.
        cluster_arrive_release();
    }

    // ---- teardown ----
    tc_fence_before();
    __syncthreads();
    if constexpr (kChecked) {
        if (threadIdx.x == 0 && rank == 0 && !*abort_flag)
            check_ok(ring_count[0] == ring_count[1], err, kSiteCheckRing);
    }
    // A pair stays alive until both CTAs are done with each other's shared
    // memory and barriers (with a cluster split, the wait that completes the
    // barrier arrived at after the reduction).
    if constexpr (C::kClusterK != 0)
        cluster_wait_acquire();
    else if constexpr (C::kPair)
        cluster_sync();
    if (warp == 1 && (C::kPair || C::kClusterK == 0)) {
        tc_fence_after();
        if constexpr (C::kPair)
            tmem_dealloc_pair(tmem_base, C::kTmemCols);
        else
            tmem_dealloc(tmem_base, C::kTmemCols);
    }
}

// D[m][n] = fp16/bf16( sum_{s < S} P[s][m][n] ), summed in split order
// (deterministic).  Each thread handles 8 consecutive outputs: two 16-byte
// loads per split and one 16-byte store.  Grid-stride over M*N/8 (N % 8 == 0).
template <bool BF16>
__global__ void __launch_bounds__(256)
splitk_reduce_kernel(const float4* __restrict__ P, uint4* __restrict__ D, int64_t groups8,
                     int64_t mn4, int32_t splits) {
    grid_launch_dependents();
    grid_dependency_wait();   // the partials come from the grid before this one
    for (int64_t g = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; g < groups8;
         g += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        float4 a = P[2 * g], b = P[2 * g + 1];
        for (int32_t s = 1; s < splits; ++s) {
            const float4 pa = P[s * mn4 + 2 * g];
            const float4 pb = P[s * mn4 + 2 * g + 1];
            a.x += pa.x; a.y += pa.y; a.z += pa.z; a.w += pa.w;
            b.x += pb.x; b.y += pb.y; b.z += pb.z; b.w += pb.w;
        }
        uint4 o;
        o.x = pack2_rn<BF16>(__float_as_uint(a.x), __float_as_uint(a.y));
        o.y = pack2_rn<BF16>(__float_as_uint(a.z), __float_as_uint(a.w));
        o.z = pack2_rn<BF16>(__float_as_uint(b.x), __float_as_uint(b.y));
        o.w = pack2_rn<BF16>(__float_as_uint(b.z), __float_as_uint(b.w));
        D[g] = o;
    }
}

// L2 group height: tiles are visited in groups of GROUP_M tile rows by all
// grid_n tile columns.  When A, B and D fit in L2 together the order hardly
// matters and plain row order (GROUP_M = 1) measured best on GB300 (4096^3:
// 1798 TFLOP/s against 1771 with 8; 4000x3000x4160: 1693 against 1668).
// Otherwise a round of `slots` resident tiles should touch as few A and B
// panels as possible: GROUP_M x (tile rows of A) + (slots / GROUP_M) x (BN
// rows of B) is smallest at GROUP_M = sqrt(slots x BN / tile rows) (8192^3:
// 8, 1864 TFLOP/s; 4: 1830; 2: 1750).
constexpr int64_t kL2FitBytes = 96ll << 20;

int choose_group_m(int64_t M, int64_t N, int64_t K, int64_t grid_m, int64_t slots, int tile_m,
                   int bn, const Tuning& t) {
    const int forced = t.group_m;
    int64_t g = 1;
    if (forced > 0) {
        g = forced;
    } else if (2 * (M + N) * K + 2 * M * N > kL2FitBytes) {
        const double best = std::sqrt(static_cast<double>(slots) * bn / tile_m);
        g = static_cast<int64_t>(best);   // 8.7 at 8192^3 on 76 pairs: 8 measured best
        if (g > 16) g = 16;
    }
    if (g > grid_m) g = grid_m;
    return static_cast<int>(g < 1 ? 1 : g);
}

template <class C>
GemmPlan plan_for(int64_t M, int64_t N, int64_t K, int64_t sms, int64_t splits, const Tuning& t) {
    GemmPlan p{};
    p.m = M;
    p.n = N;
    p.k = K;
    p.bm = C::BM;
    p.bn = C::BN;
    p.bk = C::BK;
    p.stages = C::STAGES;
    p.epi_cols = C::kEpiCols;
    p.grid_m = ceil_div(M, C::kTileM);
    p.grid_n = ceil_div(N, C::BN);
    p.k_blocks = ceil_div(K, C::BK);
    p.tiles = p.grid_m * p.grid_n;
    // Resident work slots: CTAs, or CTA pairs (sms = the device's co-resident
    // pair count for pair configurations).
    const int64_t slots = sms * C::kCtasPerSm;
    if (splits <= 0) {
        // Automatic: enough units to cover the SMs, at least 4 k-blocks each.
        splits = slots / p.tiles;
        const int64_t max_by_k = p.k_blocks / 4 > 0 ? p.k_blocks / 4 : 1;
        if (splits > max_by_k) splits = max_by_k;
        if (splits > 16) splits = 16;
        if (splits < 1) splits = 1;
    }
    if (splits > p.k_blocks) splits = p.k_blocks;
    p.kb_per_unit = ceil_div(p.k_blocks, splits);
    p.splits = ceil_div(p.k_blocks, p.kb_per_unit);   // no empty split
    p.units = p.tiles * p.splits;
    p.full_units = p.units;
    p.narrow_cols = 0;
    p.narrow_b_rows = 0;
    if constexpr (C::kTailSplit) {
        // The last round holds tiles % slots tiles: at most half the slots,
        // its tiles run as two parts each and that round takes about half
        // the time.  (A fuller last round would still need one whole round.)
        const int64_t full = p.tiles / slots * slots;
        const int64_t tail = p.tiles - full;
        if (p.splits == 1 && tail > 0 && 2 * tail <= slots && t.tail_split != 1) {
            p.full_units = full;
            p.units = full + 2 * tail;
            p.narrow_cols = C::kNarrowCols;
            p.narrow_b_rows = C::kNarrowBRows;
        }
    }
    p.group_m = choose_group_m(M, N, K, p.grid_m, slots, C::kTileM, C::BN, t);
    p.grid = static_cast<int>(p.units < slots ? p.units : slots) * (C::kPair ? 2 : 1);
    p.threads = C::kThreads;
    p.smem_bytes = static_cast<int>(C::kSmemBytes);
    p.out_f32 = C::kOutF32;
    p.bf16 = C::kBF16;
    p.pair = C::kPair;
    p.a_rows = C::kARows;
    p.b_box_rows = C::kBRows;
    // With fewer than 128 rows, a box only as tall as the rows that exist
    // (16-row multiples: whole 8-row swizzle atoms) spares the TMA unit the
    // zero fill of the rest; the stage rows above it keep stale data, which
    // reaches only accumulator rows >= M, never stored or reduced.
    p.a_box_rows = M < C::BM ? static_cast<int>((M + 15) / 16 * 16) : C::BM;
    return p;
}

// Modelled time of a plan: the busiest CTA runs ceil(units / grid) units of
// kb_per_unit k-blocks, and a k-block costs about BN + 32 units of time (MMA
// time grows with BN, the A operand traffic per k-block does not).
// Cluster splits against the other plans: each split runs one wave of
// units and then adds CK partial tiles through distributed shared memory
// (about 2 us on GB300, ~2000 units).
int64_t plan_cost(const GemmPlan& p) {
    if (p.cluster_k > 0) return p.kb_per_unit * (p.bn + (p.pair ? 16 : 32)) + 2048;
    const int64_t slots = p.pair ? p.grid / 2 : p.grid;
    // A pair streams half of B per SM: less operand traffic per k-block.
    const int64_t c = p.pair ? 16 : 32;
    if (p.narrow_cols > 0) {
        // Whole rounds, then one round of the wider tail part.  A part moves
        // more operand bytes per output than a whole tile: charge it 8 more.
        // After whole rounds, a last round full of parts is slower still (on
        // GB300, 8192^3: 72 parts on 76 pairs took 0.86 of a whole round,
        // 8 parts at 4096 x 11008 x 4096 about 0.6): charge it 60 % more
        // when every slot holds a part, in proportion below that.  Parts of
        // pair tiles whose operands fit in L2 run near their width instead
        // (1024 x 6144 x 4096: 72 parts in 0.69 of a 224-wide round); single
        // CTAs' parts did not (384 x 14336 x 2048: 146 parts after one
        // round, 26.5 us against 24.8 us for two rounds of pairs).
        const int64_t full_rounds = p.full_units / slots;
        const int64_t parts = p.units - p.full_units;
        int64_t narrow = p.kb_per_unit * (p.narrow_cols + c + 8);
        const bool in_l2 = 2 * (p.m + p.n) * p.k + 2 * p.m * p.n <= kL2FitBytes;
        if (full_rounds > 0 && !(in_l2 && p.pair)) narrow += narrow * 3 * parts / (5 * slots);
        // A single tile row: every B row streams from HBM once, and a part's
        // B stages hold half the bytes of a tile's, too few in flight to hide
        // the latency (256 x 8192 x 8192: 36.9 us in parts, 34.5 us for a
        // 2-pair cluster split; 512 x 4096 x 4096, two tile rows: 24.3
        // against 28.4 us).
        if (full_rounds == 0 && p.grid_m == 1) narrow += narrow / 2;
        return full_rounds * p.kb_per_unit * (p.bn + c) + narrow;
    }
    const int64_t rounds = ceil_div(p.units, slots);
    return rounds * p.kb_per_unit * (p.bn + c);
}

// Cluster splits among themselves (in ns): the mainloop takes the slowest
// of the MMAs, this CTA's own B stream (about 68 GB/s per SM; tile rows that
// share B rows gain little from L2 in one wave) and all unique operand bytes
// at about 6.5 TB/s; then the partial tiles are added through distributed shared memory:
// about 2 us, plus 0.34 ns per remote float, (CK - 1) / CK of the tile's
// existing rows (whole warps of 32) x BN; a CTA pair's coupled loads and
// 256-row MMAs cost about 4.5 us more.  Fitted to GB300 timings of the 2-,
// 4- and 8-CTA splits of 32..256 x 4096..14336 x 4096..14336 (each within
// ~2.5 us; 8-CTA splits measured slower than it says).  Against the k-block
// ranking it replaced it was faster on 10 of 11 shapes checked (up to 27 %,
// 128 x 3072 x 3072) and 3.7 % slower on 384 x 4096 x 14336.
int64_t cluster_split_cost(const GemmPlan& p) {
    const int64_t compute = p.kb_per_unit * (p.bn + (p.pair ? 16 : 32));
    const int64_t stream = p.b_box_rows * p.kb_per_unit * p.bk * 2 / 68;
    const int64_t hbm = (p.m + p.n) * p.k * 2 / 6500;
    const int64_t rows = (p.a_box_rows + 31) / 32 * 32;
    const int64_t reduce = 2048 + rows * p.bn * (p.cluster_k - 1) * 34 / (100 * p.cluster_k);
    return std::max(compute, std::max(stream, hbm)) + reduce + (p.pair ? 4500 : 0);
}

template <class C>
cudaError_t launch_cfg(const GemmPlan& plan, const CUtensorMap& tmA, const CUtensorMap& tmB,
                       const CUtensorMap& tmD, const GemmArgs& args, cudaStream_t stream) {
    auto kernel = gemm_tn_f16_kernel<C, DenseProblem>;
    static ContextMarks attr_done;
    cudaError_t e = smem_opt_in(kernel, static_cast<int>(C::kSmemBytes), attr_done);
    if (e != cudaSuccess) return e;
    DenseProblem prob;
    prob.tmA = tmA;
    prob.tmB = tmB;
    prob.tmD = tmD;
    prob.w.M = args.M;
    prob.w.N = args.N;
    prob.w.grid_m = static_cast<int32_t>(plan.grid_m);
    prob.w.grid_n = static_cast<int32_t>(plan.grid_n);
    prob.w.num_tiles = static_cast<int32_t>(plan.tiles);
    prob.w.num_units = static_cast<int32_t>(plan.units);
    prob.w.k_blocks = static_cast<int32_t>(plan.k_blocks);
    prob.w.kb_per_unit = static_cast<int32_t>(plan.kb_per_unit);
    prob.w.group_m = static_cast<int32_t>(plan.group_m);
    prob.w.a_box_rows = plan.a_box_rows;
    if (plan.a_box_rows > C::kARows || plan.a_rows != C::kARows) return cudaErrorInvalidValue;
    prob.w.full_units = static_cast<int32_t>(plan.full_units);
    prob.w.narrow_cols = plan.narrow_cols;
    prob.w.narrow_b_bytes = plan.narrow_b_rows * C::BK * 2;
    if (plan.narrow_cols > 0) {
        // Tail-split parts: whole store boxes, an MMA N of 16s, whole 8-row
        // swizzle atoms of B in each CTA, and B read through the narrow box
        // whose bytes the kernel counts (narrow_b_rows rows per CTA).
        const int per_cta = C::kPair ? 2 : 1;
        const int second = C::BN - plan.narrow_cols;   // the second part
        if (!C::kTailSplit || args.tmBn == nullptr || plan.narrow_cols >= C::BN ||
            plan.narrow_cols % 16 != 0 || plan.narrow_cols % C::kEpiCols != 0 ||
            plan.narrow_b_rows * per_cta != plan.narrow_cols || plan.narrow_b_rows % 8 != 0 ||
            plan.full_units > plan.units || second % C::kEpiCols != 0 ||
            (second / per_cta) % 8 != 0)
            return cudaErrorInvalidValue;
        prob.tmBn = *args.tmBn;
    } else {
        if (plan.full_units != plan.units) return cudaErrorInvalidValue;
        prob.tmBn = tmB;
    }
    prob.d_out = args.d_out;
    const unsigned cluster = static_cast<unsigned>((C::kPair ? 2 : 1) * (C::kClusterK ? C::kClusterK : 1));
    return launch_kernel(kernel, dim3(static_cast<unsigned>(plan.grid)), dim3(C::kThreads),
                         C::kSmemBytes, stream, cluster, args.pdl, prob, args.wait_limit_ns,
                         args.err_word);
}

template <class C>
cudaError_t launch_grouped_cfg(const GroupedLaunch& g, int num_sms, int num_pairs,
                               const GemmArgs& args, cudaStream_t stream) {
    auto kernel = gemm_tn_f16_kernel<C, GroupedProblem>;
    static ContextMarks attr_done;
    cudaError_t e = smem_opt_in(kernel, static_cast<int>(C::kSmemBytes), attr_done);
    if (e != cudaSuccess) return e;
    GroupedProblem prob;
    prob.tmA = g.tmA;
    prob.tmB = g.tmB;
    prob.groups = static_cast<int32_t>(g.groups);
    prob.grid_n = static_cast<int32_t>(ceil_div(g.N, C::BN));
    prob.N = static_cast<int32_t>(g.N);
    prob.k_blocks = static_cast<int32_t>(ceil_div(g.K, C::BK));
    int32_t t = 0;
    for (int64_t i = 0; i <= g.groups; ++i) {
        prob.m_off[i] = static_cast<int32_t>(g.m_offsets[i]);
        prob.tile_start[i] = t;
        if (i < g.groups) {
            prob.tmD[i] = g.tmD[i];
            const int64_t rows = g.m_offsets[i + 1] - g.m_offsets[i];
            t += static_cast<int32_t>(ceil_div(rows, C::kTileM) * prob.grid_n);
        }
    }
    if (t == 0) return cudaSuccess;   // every group is empty
    const int grid = C::kPair ? 2 * (t < num_pairs ? t : num_pairs) : (t < num_sms ? t : num_sms);
    return launch_kernel(kernel, dim3(static_cast<unsigned>(grid)), dim3(C::kThreads),
                         C::kSmemBytes, stream, C::kPair ? 2u : 1u, args.pdl, prob,
                         args.wait_limit_ns, args.err_word);
}

template <class C>
cudaError_t launch_grouped_t_cfg(const GroupedLaunch& g, int num_sms, int num_pairs,
                                 const GemmArgs& args, cudaStream_t stream) {
    static_assert(C::BN == 256 && C::kEpiBufBytes >= 16 * 256 && !C::kOutF32 && C::kClusterK == 0,
                  "transposed grouped tiles: blocks of up to 256 rows, 16 x 128 store boxes");
    auto kernel = gemm_tn_f16_kernel<C, GroupedTProblem>;
    static ContextMarks attr_done;
    cudaError_t e = smem_opt_in(kernel, static_cast<int>(C::kSmemBytes), attr_done);
    if (e != cudaSuccess) return e;
    if (g.maxw < 16 || g.maxw > C::BN || g.maxw % 16 != 0) return cudaErrorInvalidValue;
    GroupedTProblem prob;
    prob.tmW = g.tmA;
    for (int j = 0; j < 16; ++j) prob.tmX[j] = g.tmXw[j];
    prob.x_used = g.x_used;
    prob.x_ctas = C::kPair ? 2 : 1;
    prob.tmD64 = g.tmD64;
    prob.groups = static_cast<int32_t>(g.groups);
    prob.n_blocks = static_cast<int32_t>(ceil_div(g.N, C::kTileM));
    prob.N = static_cast<int32_t>(g.N);
    prob.k_blocks = static_cast<int32_t>(ceil_div(g.K, C::BK));
    prob.maxw16 = g.maxw / 16;
    int32_t t = 0;
    for (int64_t i = 0; i <= g.groups; ++i) {
        prob.m_off[i] = static_cast<int32_t>(g.m_offsets[i]);
        prob.tile_start[i] = t;
        if (i < g.groups) {
            prob.tmD[i] = g.tmD[i];
            const int64_t steps = ceil_div(g.m_offsets[i + 1] - g.m_offsets[i], 16);
            const int64_t tb = ceil_div(steps, prob.maxw16);
            t += static_cast<int32_t>(tb * prob.n_blocks);
            // Every block width of the group (q or q + 1 steps) has its map.
            if (steps > 0) {
                const int64_t q = steps / tb;
                const uint32_t need = (1u << (q - 1)) | (steps % tb != 0 ? 1u << q : 0u);
                if ((g.x_used & need) != need) return cudaErrorInvalidValue;
            }
        }
    }
    if (t == 0) return cudaSuccess;   // every group is empty
    const int grid = C::kPair ? 2 * (t < num_pairs ? t : num_pairs) : (t < num_sms ? t : num_sms);
    return launch_kernel(kernel, dim3(static_cast<unsigned>(grid)), dim3(C::kThreads),
                         C::kSmemBytes, stream, C::kPair ? 2u : 1u, args.pdl, prob,
                         args.wait_limit_ns, args.err_word);
}

}  // namespace

int grouped_tile_n(const int64_t* m_offsets, int64_t groups, int64_t N, int num_sms, int num_pairs,
                   const Tuning& t, bool* pair) {
    // The width (and single CTAs or pairs) that minimises rounds x (BN + c)
    // over all groups' tiles, as for the dense plan.
    const int widths[3] = {256, 224, 192};
    const int forced = t.tile_n;
    const int pair_mode = t.pair_mode;
    int best = 256;
    bool best_pair = false;
    int64_t best_cost = -1;
    for (int use_pair = 0; use_pair < 2; ++use_pair) {
        if (use_pair && (num_pairs <= 0 || pair_mode == 1)) continue;
        if (!use_pair && num_pairs > 0 && pair_mode == 2) continue;
        const int64_t tile_m = use_pair ? 256 : 128;
        const int64_t slots = use_pair ? num_pairs : (num_sms > 0 ? num_sms : 1);
        for (int bn : widths) {
            if (forced != 0 && bn != forced) continue;
            int64_t tiles = 0;
            for (int64_t i = 0; i < groups; ++i)
                tiles += ceil_div(m_offsets[i + 1] - m_offsets[i], tile_m) * ceil_div(N, bn);
            const int64_t used = tiles < slots ? (tiles > 0 ? tiles : 1) : slots;
            const int64_t cost = ceil_div(tiles, used) * (bn + (use_pair ? 16 : 32));
            if (best_cost < 0 || cost < best_cost) {
                best = bn;
                best_pair = use_pair != 0;
                best_cost = cost;
            }
        }
    }
    *pair = best_pair;
    return best;
}

namespace {

// Largest per-slot load of the transposed grouped schedule (units in the
// order GroupedTProblem numbers them, slot = unit mod slots): the sum over a
// slot's units of (cost of a block of width w + c), in the row-tiled plan's
// unit (one column of a 256-row pair tile per k-block).  The model charges a
// k-block of a block the larger of its MMA (w) and its loads: 128 weight rows
// and w / 2 rows of A per CTA of a pair (w for a single CTA), counting 256
// rows' bytes as long as a 256-column MMA.
int64_t grouped_t_max_load(const int64_t* m_offsets, int64_t groups, int64_t n_blocks,
                           int64_t maxw, int64_t c, int64_t slots, bool pair) {
    int64_t loads[1024] = {};
    if (slots > 1024) return -1;
    // The cost of each row block, in the kernel's order of units.
    std::vector<int64_t> costs;
    for (int64_t g = 0; g < groups; ++g) {
        const int64_t steps = ceil_div(m_offsets[g + 1] - m_offsets[g], 16);
        if (steps == 0) continue;
        const int64_t tb_count = ceil_div(steps, maxw / 16);
        const int64_t q = steps / tb_count, extra = steps % tb_count;
        for (int64_t tb = 0; tb < tb_count; ++tb) {
            const int64_t w = 16 * (q + (tb < extra ? 1 : 0));
            costs.push_back((pair ? std::max(w, 128 + w / 2) : 128 + w) + c);
        }
    }
    int64_t u = 0;
    for (const int64_t cost : costs)
        for (int64_t nb = 0; nb < n_blocks; ++nb, ++u) loads[u % slots] += cost;
    int64_t worst = 0;
    for (int64_t s = 0; s < slots; ++s) worst = std::max(worst, loads[s]);
    return worst;
}

}  // namespace

void plan_grouped(const int64_t* m_offsets, int64_t groups, int64_t N, int num_sms, int num_pairs,
                  const Tuning& t, GroupedLaunch* g) {
    // Row-tiled: rounds x (BN + c) per k-block.
    bool pair = false;
    g->bn = grouped_tile_n(m_offsets, groups, N, num_sms, num_pairs, t, &pair);
    g->pair = pair;
    g->transposed = false;
    g->maxw = 0;
    if (t.grouped_t == 1) return;
    int64_t best = -1;
    {
        const int64_t tile_m = pair ? 256 : 128;
        const int64_t slots = pair ? num_pairs : (num_sms > 0 ? num_sms : 1);
        int64_t tiles = 0;
        for (int64_t i = 0; i < groups; ++i)
            tiles += ceil_div(m_offsets[i + 1] - m_offsets[i], tile_m) * ceil_div(N, g->bn);
        const int64_t used = tiles < slots ? (tiles > 0 ? tiles : 1) : slots;
        best = t.grouped_t == 2 ? -1 : ceil_div(tiles, used) * (g->bn + (pair ? 16 : 32));
    }
    // Transposed: 256 weight rows per CTA pair (128 per single CTA) by blocks
    // of a group's rows of at most maxw, for the maxw whose schedule is best.
    const int pair_mode = t.pair_mode;
    for (int use_pair = 0; use_pair < 2; ++use_pair) {
        if (use_pair && (num_pairs <= 0 || pair_mode == 1)) continue;
        if (!use_pair && num_pairs > 0 && pair_mode == 2) continue;
        if (t.tile_n != 0 && t.tile_n != 256) continue;
        const int64_t tile_m = use_pair ? 256 : 128;
        const int64_t slots = use_pair ? num_pairs : (num_sms > 0 ? num_sms : 1);
        for (int64_t maxw = 256; maxw >= 128; maxw -= 16) {
            const int64_t load = grouped_t_max_load(m_offsets, groups, ceil_div(N, tile_m), maxw,
                                                    use_pair ? 16 : 32, slots, use_pair != 0);
            if (load < 0) continue;
            if (best < 0 || load < best) {
                best = load;
                g->transposed = true;
                g->pair = use_pair != 0;
                g->bn = 256;
                g->maxw = static_cast<int>(maxw);
            }
        }
    }
}

cudaError_t launch_grouped(const GroupedLaunch& g, int num_sms, int num_pairs, const GemmArgs& args,
                           cudaStream_t stream) {
    if (g.transposed)
        return g.pair ? launch_grouped_t_cfg<CfgP256<false>>(g, num_sms, num_pairs, args, stream)
                      : launch_grouped_t_cfg<Cfg256<false>>(g, num_sms, num_pairs, args, stream);
    if (g.pair) {
        switch (g.bn) {
            case 256: return launch_grouped_cfg<CfgP256<false>>(g, num_sms, num_pairs, args, stream);
            case 224: return launch_grouped_cfg<CfgP224<false>>(g, num_sms, num_pairs, args, stream);
            case 192: return launch_grouped_cfg<CfgP192<false>>(g, num_sms, num_pairs, args, stream);
            default: return cudaErrorInvalidValue;
        }
    }
    switch (g.bn) {
        case 256: return launch_grouped_cfg<Cfg256<false>>(g, num_sms, num_pairs, args, stream);
        case 224: return launch_grouped_cfg<Cfg224<false>>(g, num_sms, num_pairs, args, stream);
        case 192: return launch_grouped_cfg<Cfg192<false>>(g, num_sms, num_pairs, args, stream);
        default: return cudaErrorInvalidValue;
    }
}

namespace {

// A cluster split of CK: valid when all tiles x CK CTAs fit in one wave and K
// has at least CK k-blocks (otherwise units == 0).
template <class C>
GemmPlan plan_cluster_split(int64_t M, int64_t N, int64_t K, int64_t slots, int max_clusters,
                            const Tuning& t) {
    GemmPlan p = plan_for<C>(M, N, K, slots, C::kClusterK, t);
    // One cluster per tile, all resident at once (a second wave would double
    // the time).
    const int64_t clusters_fit = max_clusters != 0 ? max_clusters : slots / C::kClusterK;
    if (slots <= 0 || p.splits != C::kClusterK || p.tiles * C::kClusterK > slots ||
        p.tiles > clusters_fit)
        p.units = 0;
    p.full_units = p.units;
    p.grid = static_cast<int>(p.units) * (C::kPair ? 2 : 1);
    p.cluster_k = C::kClusterK;
    return p;
}

template <bool T>
GemmPlan plan_typed(int64_t M, int64_t N, int64_t K, int64_t sms, int64_t pairs, int64_t splits,
                    const ClusterCaps& caps, const Tuning& t) {
    // 3 single-CTA and 3 pair tile plans, up to 10 cluster splits.
    GemmPlan cands[16];
    int n = 0;
    const int pair_mode = t.pair_mode;
    const int forced = t.tile_n;
    const bool pairs_ok = splits == 1 && pairs > 0 && pair_mode != 1;
    const bool singles_ok = !(pairs_ok && pair_mode == 2);
    bool forced_ck = false;   // a forced cluster split size applies (the only candidate)
    if (splits == 1) {
        if (singles_ok) {
            cands[n++] = plan_for<Cfg256<T>>(M, N, K, sms, 1, t);
            cands[n++] = plan_for<Cfg224<T>>(M, N, K, sms, 1, t);
            cands[n++] = plan_for<Cfg192<T>>(M, N, K, sms, 1, t);
        }
        if (pairs_ok) {
            cands[n++] = plan_for<CfgP256<T>>(M, N, K, pairs, 1, t);
            cands[n++] = plan_for<CfgP224<T>>(M, N, K, pairs, 1, t);
            cands[n++] = plan_for<CfgP192<T>>(M, N, K, pairs, 1, t);
        }

        // Few tiles and a long K: split K over clusters (no workspace).
        const int ck_mode = t.cluster_split;
        if (ck_mode != 1) {
            const bool pk = pairs > 0 && pair_mode != 1;
            // The narrower single-CTA tiles take the co-residency measured for
            // the 256-wide ones: all need one CTA per SM, so a cluster of CK
            // CTAs packs the same way.
            GemmPlan ck[10] = {
                plan_cluster_split<CfgCK256<T, 2>>(M, N, K, sms, caps.single_ck[0], t),
                plan_cluster_split<CfgCK256<T, 4>>(M, N, K, sms, caps.single_ck[1], t),
                plan_cluster_split<CfgCK256<T, 8>>(M, N, K, sms, caps.single_ck[2], t),
                plan_cluster_split<CfgPCK256<T, 2>>(M, N, K, pairs, caps.pair_ck[0], t),
                plan_cluster_split<CfgPCK256<T, 4>>(M, N, K, pairs, caps.pair_ck[1], t),
                plan_cluster_split<CfgCK192<T, 2>>(M, N, K, sms, caps.single_ck[0], t),
                plan_cluster_split<CfgCK192<T, 4>>(M, N, K, sms, caps.single_ck[1], t),
                plan_cluster_split<CfgCK128<T, 4>>(M, N, K, sms, caps.single_ck[1], t),
                plan_cluster_split<CfgCK128<T, 8>>(M, N, K, sms, caps.single_ck[2], t),
                plan_cluster_split<CfgCKD128<T>>(M, N, K, sms, caps.decode_ck, t)};
            // The decode split takes problems of at most 64 rows; where it
            // applies, its 9-stage ring replaces the 6-stage one of the same tile.
            if (M > 64) ck[9].units = 0;
            if (M <= 64 && ck[9].units > 0) ck[7].units = 0;
            static_assert(sizeof(ck) / sizeof(ck[0]) + 6 <= sizeof(cands) / sizeof(cands[0]),
                          "every candidate fits");
            if (!pk) ck[3].units = ck[4].units = 0;
            if (pair_mode == 2)
                for (int i : {0, 1, 2, 5, 6, 7, 8, 9}) ck[i].units = 0;
            for (const GemmPlan& c : ck)
                if (c.units > 0 && ck_mode == c.cluster_k && (forced == 0 || c.bn == forced) &&
                    (!forced_ck || plan_cost(c) < plan_cost(cands[0]))) {
                    cands[0] = c;   // a forced split size that applies
                    n = 1;
                    forced_ck = true;
                }
            if (!forced_ck)
                for (const GemmPlan& c : ck)
                    if (c.units > 0) cands[n++] = c;
        }
    } else {
        cands[n++] = plan_for<Cfg256F<T>>(M, N, K, sms, splits, t);
        cands[n++] = plan_for<Cfg224F<T>>(M, N, K, sms, splits, t);
        cands[n++] = plan_for<Cfg192F<T>>(M, N, K, sms, splits, t);
    }
    GemmPlan best = cands[0];
    bool have = false;
    for (int i = 0; i < n; ++i) {
        const GemmPlan& c = cands[i];
        if (forced != 0 && c.bn != forced) continue;
        if (!have || plan_cost(c) < plan_cost(best)) {
            best = c;
            have = true;
        }
    }
    // Where a cluster split wins, which one: its stream, HBM and reduction
    // terms rank the splits better than k-blocks alone (128 x 8192 x 8192:
    // 2-way 192-wide 31.5 us against 4-way 256-wide 32.7 us; 256 x 4096 x
    // 4096: 18.4 against 20.0 us).
    if (have && best.cluster_k > 0 && !forced_ck) {
        for (int i = 0; i < n; ++i) {
            const GemmPlan& c = cands[i];
            if (c.cluster_k > 0 && (forced == 0 || c.bn == forced) &&
                cluster_split_cost(c) < cluster_split_cost(best))
                best = c;
        }
    }
    return best;
}

template <bool T>
cudaError_t launch_typed(const GemmPlan& plan, const CUtensorMap& tmA, const CUtensorMap& tmB,
                         const CUtensorMap& tmD, const GemmArgs& args, cudaStream_t stream) {
    if (plan.cluster_k > 0 && plan.pair) {
        switch (plan.cluster_k) {
            case 2: return launch_cfg<CfgPCK256<T, 2>>(plan, tmA, tmB, tmD, args, stream);
            case 4: return launch_cfg<CfgPCK256<T, 4>>(plan, tmA, tmB, tmD, args, stream);
            default: return cudaErrorInvalidValue;
        }
    }
    if (plan.cluster_k > 0 && plan.a_rows == 64) {
        switch (plan.bn * 16 + plan.cluster_k) {
            case 128 * 16 + 4: return launch_cfg<CfgCKD128<T>>(plan, tmA, tmB, tmD, args, stream);
            default: return cudaErrorInvalidValue;
        }
    }
    if (plan.cluster_k > 0) {
        switch (plan.bn * 16 + plan.cluster_k) {
            case 256 * 16 + 2: return launch_cfg<CfgCK256<T, 2>>(plan, tmA, tmB, tmD, args, stream);
            case 256 * 16 + 4: return launch_cfg<CfgCK256<T, 4>>(plan, tmA, tmB, tmD, args, stream);
            case 256 * 16 + 8: return launch_cfg<CfgCK256<T, 8>>(plan, tmA, tmB, tmD, args, stream);
            case 192 * 16 + 2: return launch_cfg<CfgCK192<T, 2>>(plan, tmA, tmB, tmD, args, stream);
            case 192 * 16 + 4: return launch_cfg<CfgCK192<T, 4>>(plan, tmA, tmB, tmD, args, stream);
            case 128 * 16 + 4: return launch_cfg<CfgCK128<T, 4>>(plan, tmA, tmB, tmD, args, stream);
            case 128 * 16 + 8: return launch_cfg<CfgCK128<T, 8>>(plan, tmA, tmB, tmD, args, stream);
            default: return cudaErrorInvalidValue;
        }
    }
    if (plan.pair) {
        switch (plan.bn) {
            case 256: return launch_cfg<CfgP256<T>>(plan, tmA, tmB, tmD, args, stream);
            case 224: return launch_cfg<CfgP224<T>>(plan, tmA, tmB, tmD, args, stream);
            case 192: return launch_cfg<CfgP192<T>>(plan, tmA, tmB, tmD, args, stream);
            default: return cudaErrorInvalidValue;
        }
    }
    if (!plan.out_f32) {
        switch (plan.bn) {
            case 256: return launch_cfg<Cfg256<T>>(plan, tmA, tmB, tmD, args, stream);
            case 224: return launch_cfg<Cfg224<T>>(plan, tmA, tmB, tmD, args, stream);
            case 192: return launch_cfg<Cfg192<T>>(plan, tmA, tmB, tmD, args, stream);
            default: return cudaErrorInvalidValue;
        }
    }
    switch (plan.bn) {
        case 256: return launch_cfg<Cfg256F<T>>(plan, tmA, tmB, tmD, args, stream);
        case 224: return launch_cfg<Cfg224F<T>>(plan, tmA, tmB, tmD, args, stream);
        case 192: return launch_cfg<Cfg192F<T>>(plan, tmA, tmB, tmD, args, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

namespace {

// Everything a plan depends on.
struct PlanKey {
    int64_t m, n, k, splits;
    int sms, pairs, bf16;
    ClusterCaps caps;
    Tuning t;
    bool operator==(const PlanKey& o) const {
        return m == o.m && n == o.n && k == o.k && splits == o.splits && sms == o.sms &&
               pairs == o.pairs && bf16 == o.bf16 &&
               std::equal(caps.single_ck, caps.single_ck + 3, o.caps.single_ck) &&
               std::equal(caps.pair_ck, caps.pair_ck + 2, o.caps.pair_ck) &&
               caps.decode_ck == o.caps.decode_ck &&
               t.tile_n == o.t.tile_n && t.pair_mode == o.t.pair_mode &&
               t.cluster_split == o.t.cluster_split && t.tail_split == o.t.tail_split &&
               t.group_m == o.t.group_m && t.small_m_route == o.t.small_m_route &&
               t.plain_launch == o.t.plain_launch && t.m1_route == o.t.m1_route &&
               t.grouped_t == o.t.grouped_t;
    }
};

// The last few plans of this host thread (round-robin replacement): a shape
// that repeats skips the search over candidate plans.
struct PlanCache {
    static constexpr int kEntries = 8;
    PlanKey key[kEntries];
    GemmPlan plan[kEntries];
    bool used[kEntries] = {};
    int next = 0;
};
thread_local PlanCache t_plan_cache;

}  // namespace

GemmPlan plan_gemm(int64_t M, int64_t N, int64_t K, int num_sms, const Tuning& t, int64_t splits,
                   bool bf16, int num_pairs, const ClusterCaps& caps) {
    const int64_t sms = num_sms > 0 ? num_sms : 1;
    const PlanKey key{M, N, K, splits, static_cast<int>(sms), num_pairs, bf16 ? 1 : 0, caps, t};
    PlanCache& c = t_plan_cache;
    for (int i = 0; i < PlanCache::kEntries; ++i)
        if (c.used[i] && c.key[i] == key) return c.plan[i];
    const GemmPlan p = bf16 ? plan_typed<true>(M, N, K, sms, num_pairs, splits, caps, t)
                            : plan_typed<false>(M, N, K, sms, num_pairs, splits, caps, t);
    c.key[c.next] = key;
    c.plan[c.next] = p;
    c.used[c.next] = true;
    c.next = (c.next + 1) % PlanCache::kEntries;
    return p;
}

int max_resident_pairs() {
    // How many two-CTA clusters of the pair kernel can be resident at once.
    auto kernel = gemm_tn_f16_kernel<CfgP256<false>, DenseProblem>;
    static ContextMarks attr_done;
    if (smem_opt_in(kernel, static_cast<int>(CfgP256<false>::kSmemBytes), attr_done) != cudaSuccess)
        return 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2, 1, 1);
    cfg.blockDim = dim3(CfgP256<false>::kThreads, 1, 1);
    cfg.dynamicSmemBytes = CfgP256<false>::kSmemBytes;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&clusters, kernel, &cfg) != cudaSuccess) return 0;
    return clusters;
}

namespace {

// Co-resident clusters of CTAS CTAs of configuration C (0 if unknown).
template <class C>
int max_active_clusters(int ctas) {
    auto kernel = gemm_tn_f16_kernel<C, DenseProblem>;
    static ContextMarks attr_done;
    if (smem_opt_in(kernel, static_cast<int>(C::kSmemBytes), attr_done) != cudaSuccess) return 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(ctas), 1, 1);
    cfg.blockDim = dim3(C::kThreads, 1, 1);
    cfg.dynamicSmemBytes = C::kSmemBytes;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(ctas);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&clusters, kernel, &cfg) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return clusters;
}

}  // namespace

ClusterCaps query_cluster_caps() {
    ClusterCaps c;
    c.single_ck[0] = max_active_clusters<CfgCK256<false, 2>>(2);
    c.single_ck[1] = max_active_clusters<CfgCK256<false, 4>>(4);
    c.single_ck[2] = max_active_clusters<CfgCK256<false, 8>>(8);
    c.pair_ck[0] = max_active_clusters<CfgPCK256<false, 2>>(4);
    c.pair_ck[1] = max_active_clusters<CfgPCK256<false, 4>>(8);
    c.decode_ck = max_active_clusters<CfgCKD128<false>>(4);
    // A query that failed must not read as "unknown" (ideal packing): forbid.
    for (int& v : c.single_ck) v = v > 0 ? v : -1;
    for (int& v : c.pair_ck) v = v > 0 ? v : -1;
    c.decode_ck = c.decode_ck > 0 ? c.decode_ck : -1;
    return c;
}

cudaError_t launch_gemm_tn(const GemmPlan& plan, const CUtensorMap& tmA, const CUtensorMap& tmB,
                           const CUtensorMap& tmD, const GemmArgs& args, cudaStream_t stream) {
    return plan.bf16 ? launch_typed<true>(plan, tmA, tmB, tmD, args, stream)
                     : launch_typed<false>(plan, tmA, tmB, tmD, args, stream);
}

GemmPlan plan_small_m(int64_t M, int64_t N, int64_t K, int num_sms, int64_t splits,
                      const Tuning& t) {
    const int64_t sms = num_sms > 0 ? num_sms : 1;
    // The swapped problem: rows = N (weights), columns = Mp, same K.
    if (M <= 16) return plan_for<CfgS16>(N, 16, K, sms, splits, t);
    if (M <= 32) return plan_for<CfgS32>(N, 32, K, sms, splits, t);
    return plan_for<CfgS64>(N, 64, K, sms, splits, t);
}

cudaError_t launch_small_m(const GemmPlan& plan, const CUtensorMap& tmW, const CUtensorMap& tmX,
                           const CUtensorMap& tmP, const GemmArgs& args, cudaStream_t stream) {
    switch (plan.bn) {
        case 16: return launch_cfg<CfgS16>(plan, tmW, tmX, tmP, args, stream);
        case 32: return launch_cfg<CfgS32>(plan, tmW, tmX, tmP, args, stream);
        case 64: return launch_cfg<CfgS64>(plan, tmW, tmX, tmP, args, stream);
        default: return cudaErrorInvalidValue;
    }
}

namespace {

// D[m][n] = fp16( sum_{s < S} P[s][n][m] ) for m < M: the partials of the
// swapped problem are N x Mp (weights' rows by padded activation rows).  A
// thread owns one n and 16 consecutive m: per split it reads 64 contiguous
// bytes (four 16-byte loads), adds in split order, and writes its (up to) 16
// outputs; for a fixed m, consecutive threads write consecutive n (coalesced).
__global__ void __launch_bounds__(256)
small_m_reduce_kernel(const float4* __restrict__ P, __half* __restrict__ D, int32_t M, int32_t N,
                      int32_t Mp, int32_t splits) {
    grid_launch_dependents();
    grid_dependency_wait();   // the partials come from the grid before this one
    const int32_t groups16 = Mp / 16;
    const int64_t t = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x;
    if (t >= static_cast<int64_t>(N) * groups16) return;
    const int32_t n = static_cast<int32_t>(t % N);
    const int32_t m0 = static_cast<int32_t>(t / N) * 16;
    if (m0 >= M) return;
    const int64_t part4 = static_cast<int64_t>(N) * Mp / 4;          // float4s per split
    const float4* p = P + (static_cast<int64_t>(n) * Mp + m0) / 4;
    float4 a0 = p[0], a1 = p[1], a2 = p[2], a3 = p[3];
    for (int32_t s = 1; s < splits; ++s) {
        const float4* q = p + s * part4;
        const float4 b0 = q[0], b1 = q[1], b2 = q[2], b3 = q[3];
        a0.x += b0.x; a0.y += b0.y; a0.z += b0.z; a0.w += b0.w;
        a1.x += b1.x; a1.y += b1.y; a1.z += b1.z; a1.w += b1.w;
        a2.x += b2.x; a2.y += b2.y; a2.z += b2.z; a2.w += b2.w;
        a3.x += b3.x; a3.y += b3.y; a3.z += b3.z; a3.w += b3.w;
    }
    const float v[16] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w,
                         a2.x, a2.y, a2.z, a2.w, a3.x, a3.y, a3.z, a3.w};
#pragma unroll
    for (int i = 0; i < 16; ++i)
        if (m0 + i < M) D[static_cast<int64_t>(m0 + i) * N + n] = __float2half_rn(v[i]);
}

}  // namespace

cudaError_t launch_small_m_reduce(const void* partials, void* D, int64_t M, int64_t N, int64_t Mp,
                                  int64_t splits, bool pdl, cudaStream_t stream) {
    const int64_t threads = N * (Mp / 16);
    const int64_t blocks = (threads + 255) / 256;
    return launch_kernel(small_m_reduce_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0,
                         stream, 1u, pdl, static_cast<const float4*>(partials),
                         static_cast<__half*>(D),
                         static_cast<int32_t>(M), static_cast<int32_t>(N),
                         static_cast<int32_t>(Mp), static_cast<int32_t>(splits));
}

cudaError_t launch_splitk_reduce(const void* partials, void* D, int64_t M, int64_t N,
                                 int64_t splits, bool bf16, int num_sms, bool pdl,
                                 cudaStream_t stream) {
    const int64_t groups8 = M * N / 8;
    int64_t blocks = (groups8 + 255) / 256;
    const int64_t cap = static_cast<int64_t>(num_sms > 0 ? num_sms : 1) * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    auto kernel = bf16 ? splitk_reduce_kernel<true> : splitk_reduce_kernel<false>;
    return launch_kernel(kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream, 1u, pdl,
                         static_cast<const float4*>(partials), static_cast<uint4*>(D), groups8,
                         M * N / 4, static_cast<int32_t>(splits));
}

}  // namespace tmagemm
