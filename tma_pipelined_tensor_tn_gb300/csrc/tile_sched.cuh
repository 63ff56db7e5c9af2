// Persistent tile schedule and pipeline-ring bookkeeping, shared by the host
// (introspection/tests) and the device (the GEMM kernel's roles).
//
// Schedule: a persistent grid of G CTAs; CTA c takes linear tile ids
// c, c + G, c + 2G, ...  ("使用 TMA 为 GEMM 建立 Pipeline", 第 6 步 Persistent
// Kernel 与 Tile Scheduler).  Linear ids are mapped to (m, n) tiles in L2
// groups of `group_m` tile rows: inside a group the id walks down the rows of
// one tile column, then moves to the next column; the last group may be
// shorter ("TensorCore_GEMM_with_TMA" §2.3 kernel, block swizzle; step 6's
// l2_group_size = 8).
//
// Ring: the producer and the MMA issuer both count k-block iterations over the
// CTA's whole life (not per tile), so stage = it % S and the mbarrier phase
// parity = (it / S) & 1 stay right for any K and any number of stages.  Step 6
// resets the phases per tile, which is only valid when every barrier is used an
// even number of times per tile (its K_TILES % (2 * PIPE_DEPTH) == 0 assert);
// the running counter removes that restriction (e.g. K = 4160 gives 65
// k-blocks per tile).
#pragma once

#include <cstdint>

namespace tmagemm {

struct TileCoord {
    int32_t m_blk;
    int32_t n_blk;
};

__host__ __device__ __forceinline__ TileCoord tile_coord(int64_t tile, int64_t grid_m,
                                                        int64_t grid_n, int64_t group_m) {
    const int64_t group_size = group_m * grid_n;
    const int64_t group_id = tile / group_size;
    const int64_t first_m = group_id * group_m;
    const int64_t rows = (grid_m - first_m) < group_m ? (grid_m - first_m) : group_m;
    const int64_t local = tile - group_id * group_size;
    TileCoord c;
    c.m_blk = static_cast<int32_t>(first_m + local % rows);
    c.n_blk = static_cast<int32_t>(local / rows);
    return c;
}

__host__ __device__ __forceinline__ uint32_t ring_stage(uint32_t it, uint32_t stages) {
    return it % stages;
}

__host__ __device__ __forceinline__ uint32_t ring_phase(uint32_t it, uint32_t stages) {
    return (it / stages) & 1u;
}

__host__ __device__ __forceinline__ int64_t ceil_div(int64_t a, int64_t b) {
    return (a + b - 1) / b;
}

}  // namespace tmagemm
