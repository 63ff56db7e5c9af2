// Internal host-side interface between the C ABI (abi.cu) and the kernels'
// translation units.  Not installed; the public interface is include/tmagemm.h.
#pragma once

#include <atomic>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace tmagemm {

// The tuning choices of one call, fixed when the call starts: either the
// caller's per-call options (gemm_f16_ex) or a snapshot of the process-wide
// settings (tmagemm_set_*).  Every field 0 = the automatic choice.
struct Tuning {
    int tile_n = 0;          // 256, 224, 192 (128: cluster splits only) forces that width
    int pair_mode = 0;       // 1 never CTA pairs, 2 pairs only
    int cluster_split = 0;   // 1 never, 2/4/8 that cluster size wherever it applies
    int tail_split = 0;      // 1 never
    int group_m = 0;         // 1..64 forces GROUP_M of the tile order
    int small_m_route = 0;   // 1 swap-AB, 2 register fragments (M <= 16), 3 LSU-fed tcgen05
    int plain_launch = 0;    // 1: launch without programmatic dependent launch
    int m1_route = 0;        // 1: M = 1 through the tile kernel instead of the GEMV
    int grouped_t = 0;       // grouped GEMM: 1 never transposed, 2 always transposed
    bool pdl() const { return plain_launch == 0; }
};

// Snapshot of the process-wide settings.
Tuning process_tuning();

// Unique id (cuCtxGetId) of the CUDA context current on this thread, 0 if
// none is current.  Per-device set-up that lives in a context (function
// attributes, the addresses of __device__ arrays) is keyed on it, so that it
// is redone after cudaDeviceReset replaces the device's context.
uint64_t current_context_id();

// Rows of a D store box: each of the four epilogue warps stores its own 32
// rows of a tile.
constexpr int kEpiWarpRows = 32;

// GEMM tile configuration used by the persistent tcgen05 kernel.
struct GemmPlan {
    int bm, bn, bk, stages;
    int64_t tiles, grid_m, grid_n, k_blocks;
    int64_t splits;        // k-splits (1 = plain GEMM, fp16 output)
    int64_t kb_per_unit;   // k-blocks per work unit
    int64_t units;         // tiles * splits
    int grid, threads;
    int smem_bytes;
    int epi_cols;          // columns per epilogue TMA store box
    bool out_f32;          // split-K partials (FP32 workspace) instead of fp16 D
    bool bf16;             // bf16 operands and output instead of fp16
    bool pair;             // CTA-pair (cta_group::2) tiles of 256 x bn
    int b_box_rows;        // rows of B per CTA (bn, or bn / 2 for a pair)
    int a_box_rows;        // rows of A per TMA box: 128, or M rounded up to 16 when M < 128
    int cluster_k;         // > 0: K split over clusters of this many CTAs (one unit per CTA)
    int a_rows;            // rows of A a stage holds (128; 64 for the decode cluster splits)
    int group_m;           // L2 group height of the tile order, in tiles
    // Tail split: the tiles of the last, partly filled round run as two units
    // each (narrow_cols and bn - narrow_cols columns), when that round is at
    // most half full.  Units < full_units are whole tiles; narrow_cols = 0
    // (full_units = units) without a tail split.
    int64_t full_units;
    int narrow_cols;
    int narrow_b_rows;     // rows of B per CTA in a part's box (narrow_cols, or half for a pair)
    int64_t m, n, k;       // the problem the plan is for
};

// How many clusters of each cluster-split configuration can be co-resident
// (single CTAs with CK = 2, 4, 8; CTA pairs with CK = 2, 4).  0 = unknown:
// the plan then assumes ideal packing (slots / CTAs per cluster).
struct ClusterCaps {
    int single_ck[3] = {0, 0, 0};
    int pair_ck[2] = {0, 0};
    int decode_ck = 0;             // the decode split (4 CTAs, 128 wide, 9 stages)
};

// Pure function of the problem shape, the SM count and the tuning (no CUDA
// calls).  splits == 1: the plain GEMM; splits == 0: choose the split count;
// else that many splits (clamped so that no split is empty).
GemmPlan plan_gemm(int64_t M, int64_t N, int64_t K, int num_sms, const Tuning& t,
                   int64_t splits = 1, bool bf16 = false, int num_pairs = 0,
                   const ClusterCaps& caps = ClusterCaps{});

// The co-residency of the cluster-split kernels on the current device.
ClusterCaps query_cluster_caps();

// Co-resident two-CTA clusters of the pair kernel on the current device
// (0 if clusters cannot be launched).
int max_resident_pairs();

// D = fp16/bf16(sum of `splits` FP32 partial M x N matrices laid out back to back).
cudaError_t launch_splitk_reduce(const void* partials, void* D, int64_t M, int64_t N,
                                 int64_t splits, bool bf16, int num_sms, bool pdl,
                                 cudaStream_t stream);

struct GemmArgs {
    int32_t M, N, K;
    uint64_t wait_limit_ns;
    uint32_t* err_word;   // device address of the sticky error word
    void* d_out = nullptr;   // D itself, for the cluster-split epilogue
    const CUtensorMap* tmBn = nullptr;   // B with box {bk, narrow_b_rows} (tail split only)
    bool pdl = true;      // launch with programmatic dependent launch
};

// Enqueue the GEMM kernel.  Tensor maps: A {K, M} box {bk, bm}; B {K, N} box
// {bk, bn}; D {N, M} box {epi_cols, 32} (fp16), or for split-K the FP32
// workspace {N, M, splits} box {32, 32, 1}.
cudaError_t launch_gemm_tn(const GemmPlan& plan, const CUtensorMap& tmA, const CUtensorMap& tmB,
                           const CUtensorMap& tmD, const GemmArgs& args, cudaStream_t stream);

// Skinny GEMM (2 <= M <= 64) as a swapped split-K problem: rows = N (weights),
// columns = Mp = M rounded up to 16/32/64, same K.  Partials go to an FP32
// workspace [splits][N][Mp]; launch_small_m_reduce transposes and sums them.
GemmPlan plan_small_m(int64_t M, int64_t N, int64_t K, int num_sms, int64_t splits,
                      const Tuning& t);
cudaError_t launch_small_m(const GemmPlan& plan, const CUtensorMap& tmW, const CUtensorMap& tmX,
                           const CUtensorMap& tmP, const GemmArgs& args, cudaStream_t stream);
cudaError_t launch_small_m_reduce(const void* partials, void* D, int64_t M, int64_t N, int64_t Mp,
                                  int64_t splits, bool pdl, cudaStream_t stream);

// Skinny GEMM (2 <= M <= small_m_mma_max_m()) on register fragments: the
// weights stream from HBM straight into mma.sync operands; K is split over
// the 8 CTAs of a cluster and reduced through distributed shared memory.
// No workspace; one launch.
int64_t small_m_mma_max_m();
int64_t small_m_mma_ctas(int64_t N, int num_sms);
int64_t small_m_mma_wave(int num_sms);
cudaError_t launch_small_m_mma(int64_t M, int64_t N, int64_t K, const void* X, const void* W,
                               void* D, cudaStream_t stream, bool bf16, int num_sms,
                               uint32_t* err, bool pdl);

// Skinny GEMM (2 <= M <= 64) on tcgen05 with the weights staged in shared
// memory by the SMs' own 16-byte loads (X by TMA); K split over 8-CTA clusters
// and reduced through distributed shared memory.  tmX: X {K, M} box
// {64, small_m_lsu_cols(M)}, 128B swizzle.  No workspace; one launch.
int64_t small_m_lsu_cols(int64_t M);
cudaError_t launch_small_m_lsu(const CUtensorMap& tmX, int64_t M, int64_t N, int64_t K,
                               const void* W, void* D, uint64_t limit_ns, uint32_t* err,
                               cudaStream_t stream, bool bf16, bool pdl);

// Grouped GEMM: groups g < G with rows [m_offsets[g], m_offsets[g+1]) of A
// and D and weights B[g] (N x K).  Maps: A {K, rows} box {64, 128}; B
// {K, N, G} box {64, bn, 1}; tmD[g] = D rows of group g, {N, M_g} box
// {epi_cols(bn), 32} (unused for empty groups).
constexpr int kMaxGroupsHost = 64;
struct GroupedLaunch {
    CUtensorMap tmA, tmB;
    CUtensorMap tmD[kMaxGroupsHost];
    const int64_t* m_offsets;   // host, groups + 1 entries
    int64_t groups, N, K;
    int bn;
    bool pair;                  // CTA-pair tiles (256 rows; B box bn / 2 rows)
    // Transposed (D_g^T = B_g A_g^T): tmA = B {K, N, G} box {64, 128, 1},
    // tmXw (below) = A by block width, tmD[g] = D rows of group
    // g {N, M_g} box {128, 16} unswizzled (and tmD64); a group's rows in
    // blocks of at most maxw (a multiple of 16 up to bn).
    bool transposed;
    int maxw;
    CUtensorMap tmD64;          // transposed: all of D {N, rows} box {128, 64} unswizzled
    // Transposed: A {K, rows} once per block width 16 (j + 1) in use (bit j of
    // x_used), box {64, 16 (j + 1) / CTAs per tile}; tmB is then unused.
    CUtensorMap tmXw[16];
    uint32_t x_used;
};
// The grouped GEMM's formulation and tiles for these groups: the row-tiled
// form (tiles of 128 or 256 rows of a group by bn columns) or the transposed
// one (256 or 128 weight rows by blocks of up to maxw rows of a group), the
// one whose busiest CTA (pair) of the persistent schedule has the least work.
void plan_grouped(const int64_t* m_offsets, int64_t groups, int64_t N, int num_sms, int num_pairs,
                  const Tuning& t, GroupedLaunch* g);
cudaError_t launch_grouped(const GroupedLaunch& g, int num_sms, int num_pairs, const GemmArgs& args,
                           cudaStream_t stream);

// Enqueue the GEMV: y[n] = sum_k x[k] * W[n][k]; fp16 or bf16 operands and
// output.  One CTA per SM taking pieces of its rows where N / num_sms rows and
// their pieces fit the CTA's slot table, else one warp per row.
cudaError_t launch_gemv(int64_t N, int64_t K, const void* x, const void* W, void* y, bool bf16,
                        int num_sms, cudaStream_t stream, uint32_t* err, bool pdl);

// cudaLaunchKernelEx with a cluster of `cluster_x` CTAs along x (1 = none)
// and, when `pdl` is set, the programmatic-stream-serialization attribute
// (programmatic dependent launch): the next kernel on the stream is scheduled
// while the previous one finishes and runs its set-up (barrier
// initialisation, descriptor prefetch) meanwhile.  Every kernel of the
// library executes griddepcontrol.wait before its first global memory access,
// so the stream order of results is unchanged.
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem_bytes,
                          cudaStream_t stream, unsigned cluster_x, bool pdl, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem_bytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    unsigned n = 0;
    if (cluster_x > 1) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = cluster_x;
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    if (pdl) {
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, args...);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

// Per device, the context (current_context_id) in which a one-time set-up
// was last done; 0 = never.
using ContextMarks = std::atomic<uint64_t>[64];

// Opt-in of `kernel` to `bytes` (> 48 KB) of dynamic shared memory on the
// current device, once per context.  With `max_shared`, the whole
// configurable L1/shared split also goes to shared memory, so CTAs that ask
// for half of it can sit two to an SM.
template <class K>
cudaError_t smem_opt_in(K kernel, int bytes, ContextMarks& done, bool max_shared = true) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t ctx = current_context_id();
    const bool tracked = dev >= 0 && dev < 64 && ctx != 0;
    if (tracked && done[dev].load(std::memory_order_acquire) == ctx) return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess && max_shared)
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 static_cast<int>(cudaSharedmemCarveoutMaxShared));
    if (e == cudaSuccess && tracked) done[dev].store(ctx, std::memory_order_release);
    return e;
}

// Enqueue a one-block kernel that waits on an mbarrier nobody arrives on, with
// the given limit; it must end by recording kSiteTest in the error word.
cudaError_t launch_wait_timeout_probe(uint64_t limit_ns, uint32_t* err_word, cudaStream_t stream);

}  // namespace tmagemm
