/*
 * tmagemm — FP16 "TN" GEMM D = A * B^T and M = 1 GEMV for sm_103a (GB300).
 *
 * C ABI of libtmagemm.so.  Plain pointers and sizes only.  All matrices are
 * dense row-major binary16 (IEEE fp16) with no padding between rows.
 *
 * Operation (both entry points): FP32 accumulation inside the kernel and one
 * round-to-nearest-even conversion to fp16 per output element.
 *   - GEMM and its operand layout: "使用 TMA 为 GEMM 建立 Pipeline" (Modern GPU
 *     programming for MLSys), step 4 "完整 Kernel": A (M, K), B (N, K),
 *     D (M, N), float32 accumulator, float16 output; the Croqtile chapter
 *     "高级数据搬运：TMA、Swizzle 与不规则访问", section "示例：流水线矩阵乘法中的
 *     TMA": matmul(lhs [M, K], rhs [N, K], output [M, N]).
 *   - GEMV: "Learning TileLang with GEMV", §01 GEMV: y = x * W^T with W N x K
 *     row-major (the nn.Linear weight layout), FP32 accumulation.
 *   - Ragged edges: out-of-range operand elements are read as zero and
 *     out-of-range outputs are never written ("高级数据搬运…", section
 *     "零填充：.zfill"; TensorCore_GEMM_with_TMA §2.1: OOB fill NONE = zeros).
 *
 * Ownership: the caller owns every buffer.  The library allocates no device
 * memory in any call.  A, B and D must not overlap.
 *
 * Execution: gemm_f16 / gemv_f16 validate their arguments on the host, enqueue
 * one kernel on `stream` and return without synchronising.  A CUDA launch
 * error is reported as TMAGEMM_ERR_CUDA.  A device-side wait that exceeds its
 * time limit (a pipeline handshake that never completes) makes the kernel stop
 * early and record a sticky error; tmagemm_check() reports it.
 *
 * Thread safety: all entry points may be called from several host threads.
 * The tuning setters (tmagemm_set_*) change process-wide defaults: every call
 * reads them once, when it starts, so a call in progress is never affected,
 * but a setter called while other threads use the library changes those
 * threads' later calls.  Set them before the threads start, or pass per-call
 * options to gemm_f16_ex / gemm_bf16_ex, which read no process-wide setting.
 *
 * Device state: per device and per CUDA context the library looks up its own
 * device addresses and kernel attributes on first use; after cudaDeviceReset
 * the next call in the new context looks them up again.
 */
#ifndef TMAGEMM_H
#define TMAGEMM_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes returned by every entry point. */
typedef enum {
    TMAGEMM_OK = 0,
    TMAGEMM_ERR_INVALID = -1,      /* M, N or K <= 0, or a NULL pointer          */
    TMAGEMM_ERR_ALIGN = -2,        /* pointer not 16-byte aligned, or K % 8 != 0,
                                      or N % 8 != 0 (GEMM with M > 1): the TMA
                                      row strides must be multiples of 16 bytes  */
    TMAGEMM_ERR_UNSUPPORTED = -3,  /* a dimension >= 2^31, or no sm_100-family
                                      device                                     */
    TMAGEMM_ERR_CUDA = -4,         /* a CUDA runtime/driver call failed          */
    TMAGEMM_ERR_TIMEOUT = -5,      /* a device-side pipeline wait timed out      */
    TMAGEMM_ERR_WORKSPACE = -6,    /* split-K workspace missing, misaligned or
                                      smaller than required                      */
    TMAGEMM_ERR_SCRATCH_LIMIT = -7, /* gemm_f16_splitk_noalloc: the problem needs
                                      more than its fixed 32 MiB scratch         */
    TMAGEMM_ERR_CHECK = -8         /* checked build only: a kernel self-check
                                      failed (site in tmagemm_last_error_detail) */
} tmagemm_status;

/*
 * D = fp16(A * B^T), accumulated in FP32.
 *   M, N, K : sizes (> 0).
 *   A       : device pointer, M x K fp16, row-major (K contiguous).
 *   B       : device pointer, N x K fp16, row-major (K contiguous).
 *   D       : device pointer, M x N fp16, row-major; written, never read.
 *   stream  : cudaStream_t (NULL = legacy default stream).
 * Requirements: A, B, D 16-byte aligned; K % 8 == 0; N % 8 == 0 when M > 1.
 * M == 1 is computed by the GEMV kernel (x = A, W = B, y = D); 2 <= M <= 8,
 * and 9 <= M <= 16 where its grid fills at least 80 % of a wave, by the
 * register-fragment kernel of gemm_f16_small_m (B streamed straight into
 * mma.sync operands); other M by the tcgen05 tile kernel, which splits K
 * over clusters when the output has too few tiles to fill the SMs.  The
 * results agree up to FP32 accumulation order.
 * Kernel: persistent, warp-specialised: a TMA producer warp feeding a
 * multi-stage mbarrier ring of 128B-swizzled tiles, one thread issuing
 * tcgen05.mma into a double-buffered TMEM accumulator, and four epilogue warps
 * (tcgen05.ld -> fp16 -> swizzled SMEM -> TMA store).  Tiles are visited in an
 * L2-grouped order ("使用 TMA 为 GEMM 建立 Pipeline", 第 6 步 Persistent
 * Scheduling; TensorCore_GEMM_with_TMA §2.3 block swizzle).
 * Returns a tmagemm_status.
 */
int gemm_f16(int64_t M, int64_t N, int64_t K, const void* A, const void* B, void* D,
             void* stream);

/*
 * Per-call tuning of gemm_f16_ex / gemm_bf16_ex.  Every field 0 = the
 * automatic choice; the other values mean what they mean for the
 * process-wide setters further below:
 *   tile_n        : tmagemm_set_tile_n       (256, 224, 192; 128 cluster splits only)
 *   cta_pair      : tmagemm_set_cta_pair     (1 never, 2 always where possible)
 *   cluster_split : tmagemm_set_cluster_split (1 never, 2, 4 or 8 CTAs)
 *   tail_split    : tmagemm_set_tail_split   (1 never)
 *   group_m       : tmagemm_set_group_m      (1..64)
 *   small_m_route : tmagemm_set_small_m_route (1..3; 1 keeps 2 <= M <= 64 on
 *                   the tile kernel here, since these calls take no workspace)
 *   plain_launch  : 1 = launch without programmatic dependent launch, as
 *                   tmagemm_set_pdl(0) does process-wide
 *   m1_route      : 1 = compute M = 1 with the tcgen05 tile kernel instead of
 *                   the GEMV (N % 8 == 0 is then required, as for M > 1)
 * Results agree with the automatic choice up to FP32 accumulation order.
 */
typedef struct tmagemm_options {
    int32_t tile_n;
    int32_t cta_pair;
    int32_t cluster_split;
    int32_t tail_split;
    int32_t group_m;
    int32_t small_m_route;
    int32_t plain_launch;
    int32_t m1_route;
} tmagemm_options;

/* Sets every field of *opts to 0 (the automatic choices).  NULL is a no-op. */
void tmagemm_options_init(tmagemm_options* opts);

/*
 * gemm_f16 / gemm_bf16 with per-call options instead of the process-wide
 * settings (opts == NULL: the process-wide settings, i.e. gemm_f16 /
 * gemm_bf16 themselves).  Same arguments, requirements and results; a field
 * outside its range returns TMAGEMM_ERR_INVALID and launches nothing.
 */
int gemm_f16_ex(int64_t M, int64_t N, int64_t K, const void* A, const void* B, void* D,
                const tmagemm_options* opts, void* stream);
int gemm_bf16_ex(int64_t M, int64_t N, int64_t K, const void* A, const void* B, void* D,
                 const tmagemm_options* opts, void* stream);

/*
 * Split-K form of gemm_f16 for shapes with too few output tiles to fill the
 * GPU (e.g. small M x N with long K): the K range is cut into `splits` parts,
 * each (tile, part) is one work unit of the same persistent tcgen05 kernel,
 * every unit writes its FP32 partial tile to `workspace`, and a second kernel
 * adds the partials in part order and rounds once to fp16.  Partial sums
 * across blocks need an FP32 destination and one final conversion
 * ("Learning TileLang with GEMV", §5.2 block_split_k).
 *   splits         : 0 = choose automatically; otherwise the requested count,
 *                    clamped so that every part has at least one 64-wide
 *                    k-block.  If the plan ends with one part, the plain
 *                    kernel runs and the workspace is not touched.
 *   workspace      : device pointer, 16-byte aligned, at least
 *                    gemm_f16_splitk_workspace_size(M, N, K, splits) bytes;
 *                    caller-owned scratch, overwritten, no initial contents
 *                    needed.  Calls that overlap on the GPU must not share it.
 *   workspace_bytes: its size.
 * Other arguments, requirements and status codes as gemm_f16, plus
 * TMAGEMM_ERR_WORKSPACE.  Results are deterministic (fixed summation order).
 */
int gemm_f16_splitk(int64_t M, int64_t N, int64_t K, const void* A, const void* B, void* D,
                    int64_t splits, void* workspace, int64_t workspace_bytes, void* stream);

/*
 * gemm_f16_splitk for callers that cannot allocate device memory — code past a
 * no-allocation point (cudaMalloc synchronises the device and would stall a
 * latency-critical loop), plugins whose host framework owns all device memory
 * and exposes no allocator, or users with a fixed budget set at start-up.
 * The pages have no counterpart of this entry point: it exists only so that
 * such callers can use split-K without providing a workspace.
 *   Same arguments, requirements and results as gemm_f16_splitk, without the
 *   workspace: the library uses its own fixed array of 32 MiB in device memory
 *   (part of its device module, so every GPU that loads this entry point holds
 *   it until the process exits).  The caller still passes A, B and D.
 *   Problems whose split-K workspace (gemm_f16_splitk_workspace_size) exceeds
 *   32 MiB are rejected with TMAGEMM_ERR_SCRATCH_LIMIT; nothing is launched.
 *   No call allocates: no cudaMalloc, cudaFree or allocating library routine.
 *   The first call on each device looks up the array's device address on
 *   that device (again after a cudaDeviceReset, in the new context); make
 *   that first call before any stream capture.
 *   Every call shares the one array.  Calls whose kernels may overlap on the
 *   GPU (different streams, or several host threads) race on it; order them
 *   on one stream.  Its contents between calls do not matter: each call
 *   writes every partial it later reads.
 */
int gemm_f16_splitk_noalloc(int64_t M, int64_t N, int64_t K, const void* A, const void* B, void* D,
                            int64_t splits, void* stream);

/*
 * Bytes of workspace gemm_f16_splitk needs for (M, N, K, splits) on the
 * current device (splits = 0: the automatic choice): parts x M x N x 4, or 0
 * when no split is made.  Negative values are status codes.
 */
int64_t gemm_f16_splitk_workspace_size(int64_t M, int64_t N, int64_t K, int64_t splits);

/*
 * y = fp16(x * W^T), accumulated in FP32 ("Learning TileLang with GEMV",
 * §01 GEMV; loads as in §4.5 thread_vectorized_split_k, reduction as in
 * §4.6 Reduction).
 *   N, K   : sizes (> 0).
 *   x      : device pointer, K fp16.
 *   W      : device pointer, N x K fp16, row-major.
 *   y      : device pointer, N fp16; written, never read.
 *   stream : cudaStream_t (NULL = legacy default stream).
 * Requirements: x, W, y 16-byte aligned; K % 8 == 0.
 * Returns a tmagemm_status.
 */
int gemv_f16(int64_t N, int64_t K, const void* x, const void* W, void* y, void* stream);

/*
 * Grouped GEMM: G independent TN GEMMs that share N and K, with run-time row
 * counts (e.g. the tokens routed to each of G experts):
 *   D[r][n] = fp16( sum_k A[r][k] * B[g][n][k] )  for m_offsets[g] <= r < m_offsets[g+1].
 * The same persistent kernel and pipeline run over the tiles of all groups;
 * each group only moves the origin of its A/D window ("高级数据搬运：TMA、
 * Swizzle 与不规则访问", section "任意偏移窗口：view 与 from", the MoE case).
 *   G         : 1 <= G <= 64 groups.
 *   m_offsets : HOST array of G + 1 row offsets, m_offsets[0] = 0,
 *               non-decreasing; group g owns rows [m_offsets[g], m_offsets[g+1])
 *               (empty groups allowed).  Read during the call only.
 *   A         : device pointer, m_offsets[G] x K fp16 row-major.
 *   B         : device pointer, G x N x K fp16 (G stacked row-major N x K).
 *   D         : device pointer, m_offsets[G] x N fp16 row-major.
 * Requirements as gemm_f16 (16-byte alignment, K % 8 == 0, N % 8 == 0).
 * Status codes as gemm_f16; G > 64 returns TMAGEMM_ERR_UNSUPPORTED.
 */
int gemm_f16_grouped(int64_t G, const int64_t* m_offsets, int64_t N, int64_t K, const void* A,
                     const void* B, void* D, void* stream);

/*
 * Skinny GEMM for a few rows of activations, D = fp16(X * W^T) with
 * 2 <= M <= 64: the decode step of "Learning TileLang with GEMV" (§01 GEMV:
 * every linear layer is a GEMV when tokens are decoded one by one) for a
 * batch of M tokens.  Like the GEMV it is bound by reading W once.  The
 * automatic choice (tmagemm_set_small_m_route overrides it):
 *   - M <= 8, and M <= 16 when N is such that this kernel's grid fills at
 *     least 80 % of a wave (4 CTAs per SM; e.g. N = 4096 or 8192): W streams
 *     from HBM straight into mma.sync register fragments (16-byte loads, no
 *     shared-memory staging); the CTAs of a cluster split K and add their
 *     FP32 partials in fixed order through distributed shared memory.
 *   - otherwise: the tcgen05 tile kernel of gemm_f16, which splits K over
 *     clusters when the output has too few tiles to fill the SMs.
 * Neither needs a workspace.  Two more kernels are available by route: the
 * tcgen05 kernel with the roles swapped (W the 128-row MMA operand, X the
 * 16- or 64-wide one, rows past M zero; K split, FP32 partials in
 * `workspace`, a second kernel adds them in fixed order, transposes and
 * rounds), and tcgen05 with W staged in shared memory by the SMs' own loads.
 *   X         : device pointer, M x K fp16 row-major (activations).
 *   W         : device pointer, N x K fp16 row-major (weights).
 *   D         : device pointer, M x N fp16 row-major.
 *   workspace : device pointer, 16-byte aligned, at least
 *               gemm_f16_small_m_workspace_size(M, N, K) bytes; scratch,
 *               overwritten, no initial contents needed; not shared by calls
 *               that overlap on the GPU.
 * Requirements as gemm_f16; M outside [2, 64] returns TMAGEMM_ERR_UNSUPPORTED
 * (M = 1 is gemv_f16, larger M is gemm_f16).  Deterministic.
 */
int gemm_f16_small_m(int64_t M, int64_t N, int64_t K, const void* X, const void* W, void* D,
                     void* workspace, int64_t workspace_bytes, void* stream);

/* Workspace bytes gemm_f16_small_m needs on the current device (negative =
 * status; 0 unless route 1 sends this M to the swap-AB kernel). */
int64_t gemm_f16_small_m_workspace_size(int64_t M, int64_t N, int64_t K);

/*
 * Route of gemm_f16_small_m, process-wide: 0 = automatic (above), 2 = the
 * register fragments wherever they apply (M <= 16) and the tile kernel
 * above, 1 = always the swap-AB kernel (needs the workspace), 3 = always the
 * LSU-fed tcgen05 kernel.
 * gemm_f16 / gemm_bf16 with 2 <= M <= 64 follow routes 0, 2 and 3 and take
 * the tile kernel under route 1.  Results
 * agree up to FP32 accumulation order.  The workspace size depends on the
 * route: query it after setting the route.  Returns TMAGEMM_ERR_INVALID for
 * other values.
 */
int tmagemm_set_small_m_route(int route);

/*
 * bfloat16 forms of gemm_f16 and gemv_f16: A, B, D (x, W, y) hold bf16
 * values; accumulation is FP32 and each output is rounded once to bf16
 * (nearest even).  Same kernels, tiles, shape routing (M = 1 the GEMV, a
 * few rows the register-fragment kernel, as for gemm_f16), requirements and
 * status codes; only the element type of the tensor maps, the MMA operand format and
 * the final conversion change.  "TensorCore_GEMM_with_TMA" runs this TN GEMM in bf16
 * (§2.1 init tensor map: CU_TENSOR_MAP_DATA_TYPE_BFLOAT16; §2.3: bf16 output
 * rounded to nearest).
 */
int gemm_bf16(int64_t M, int64_t N, int64_t K, const void* A, const void* B, void* D,
              void* stream);
int gemv_bf16(int64_t N, int64_t K, const void* x, const void* W, void* y, void* stream);

/*
 * Synchronises `stream`, then reads and clears the current device's sticky
 * device-side error word.  Returns TMAGEMM_OK, TMAGEMM_ERR_TIMEOUT (a kernel
 * stopped after a pipeline wait ran out of time) or TMAGEMM_ERR_CUDA.
 */
int tmagemm_check(void* stream);

/*
 * Detail of the last device-side error on the current device (0 = none):
 * bits 0..7 the wait site, bits 8..31 the block index.  Does not clear it.
 */
int tmagemm_last_error_detail(void);

/*
 * Checked build (libtmagemm_checked.so, compiled with -DTMAGEMM_CHECKED): the
 * kernels check their own invariants in place of a sanitizer.  A TMA
 * coordinate that breaks the 16-byte rule or is negative, an epilogue index
 * outside its tile or D, or producer and MMA issuer that consumed different
 * numbers of k-blocks record a site (11..13) in the error word, skip the
 * access, and make tmagemm_check return TMAGEMM_ERR_CHECK.  Every work unit
 * that completes (an output tile, or one K part of it) increments a counter.
 * tmagemm_checked_unit_counts waits for `stream`, copies the first n counters
 * (unit u at index u mod 65536; the tile kernel numbers its units as
 * tmagemm_gemm_plan does: K part * tiles + tile, the grouped GEMM the groups'
 * tiles one after the other; the small-M kernels count one unit per CTA and
 * the GEMV one per output row) to host memory `counts` and zeroes all of
 * them.  In the normal build it returns TMAGEMM_ERR_UNSUPPORTED.
 */
int tmagemm_checked_unit_counts(uint32_t* counts, int64_t n, void* stream);

/* Static text for a status code (never NULL). */
const char* tmagemm_strerror(int status);

/* Library version, (major << 16) | (minor << 8) | patch. */
int tmagemm_version(void);

/*
 * Diagnostics for the failure path: enqueues a one-block kernel whose only
 * thread waits, with the same bounded wait the GEMM roles use, on an mbarrier
 * that nothing ever arrives on.  After `limit_ms` (1..10000) the wait gives up
 * and records a timeout in the device error word; the kernel then returns
 * normally and the context stays usable.  tmagemm_check() afterwards must
 * return TMAGEMM_ERR_TIMEOUT.  No TMA or tensor-core work is involved.
 */
int tmagemm_selftest_wait_timeout(int64_t limit_ms, void* stream);

/*
 * Tuning/test override of the CTA-pair tiles of gemm_f16 / gemm_bf16: 0 =
 * automatic (a pair of CTAs on two SMs runs one 256 x N tile with cta_group::2
 * MMAs when the plan's cost model prefers it), 1 = never use pairs, 2 = use
 * pairs whenever the device can co-schedule them.  Process-wide; results are
 * the same up to FP32 accumulation order.  Returns TMAGEMM_ERR_INVALID for
 * other values.
 */
int tmagemm_set_cta_pair(int mode);

/*
 * Tuning/test override of the GEMM's tile width N: 256, 224 or 192 forces that
 * tile shape for every later gemm_f16 call in the process (128 exists only for
 * cluster splits, so it applies where one does); 0 restores the automatic
 * choice (the width that minimises the number of tile rounds on the device's
 * SMs, weighted by tile cost).  Results are the same for every width up to
 * FP32 accumulation order.  Returns TMAGEMM_ERR_INVALID for other values.
 */
int tmagemm_set_tile_n(int bn);

/*
 * Tuning override of the dense GEMM's tile order: tiles are visited in groups
 * of GROUP_M tile rows (by all tile columns), so that tiles sharing A and B
 * panels run close together in time.  0 = automatic (about one round of
 * resident tiles per group), 1..64 = that GROUP_M.  Results are identical
 * (the order changes which CTA computes a tile, not how).  Returns
 * TMAGEMM_ERR_INVALID for other values.
 */
int tmagemm_set_group_m(int g);

/*
 * Cluster split-K of gemm_f16 / gemm_bf16, process-wide: 0 = automatic (for
 * shapes whose output tiles fill at most half of the SMs, when the plan's cost
 * model prefers it, the CTAs of a 2-, 4- or 8-CTA cluster compute one
 * 128 x 256, 128 x 192 or 128 x 128 tile (or a 256 x 256 tile in CTA pairs)
 * over separate K ranges and add their FP32 accumulators through distributed
 * shared memory, in fixed order, before writing D: no workspace, one launch),
 * 1 = never, 2, 4 or 8 = that cluster size whenever all tiles x that many
 * CTAs fit in one wave.  Results agree up to FP32
 * accumulation order.  Returns TMAGEMM_ERR_INVALID for other values.
 */
int tmagemm_set_cluster_split(int mode);

/*
 * Tail split of gemm_f16 / gemm_bf16, process-wide: 0 = automatic, 1 = never.
 * A persistent schedule whose last round of output tiles fills at most half
 * of the resident CTAs (or CTA pairs) runs each tile of that round as two
 * work units of its column range — 128 columns and the rest of the tile
 * (128, 96 or 64 for tiles 256, 224 or 192 wide) — so the round takes about
 * half as long; the plan's cost model weighs it against the other tile
 * widths.  Every output is still summed over all of K by one unit, in the
 * same k order as in an unsplit tile.  Returns TMAGEMM_ERR_INVALID for other
 * values.
 */
int tmagemm_set_tail_split(int mode);

/*
 * Formulation of gemm_f16_grouped, process-wide: 0 = automatic, 1 = always
 * row tiles (tiles of 128 or 256 rows of one group), 2 = always transposed
 * (each group computed as D_g^T = B_g A_g^T: tiles of 256 or 128 weight rows
 * by blocks of up to 256 rows of the group, so a group's rows are padded to
 * a multiple of 16 instead of 128 or 256; the accumulator is stored
 * transposed).  Results agree up to FP32 accumulation order.  Returns
 * TMAGEMM_ERR_INVALID for other values.
 */
int tmagemm_set_grouped_transposed(int mode);

/*
 * The plan gemm_f16_grouped runs for these groups (G, m_offsets and N as for
 * gemm_f16_grouped) on `num_sms` SMs with `num_pairs` co-resident CTA pairs:
 * out[0] = 1 if transposed, out[1] = 1 if CTA pairs, out[2] = tile width of
 * the row tiles (256 when transposed), out[3] = the widest block of a group's
 * rows when transposed (else 0).  `out` holds 4 values.  No GPU needed.
 */
int tmagemm_grouped_plan(int64_t G, const int64_t* m_offsets, int64_t N, int64_t num_sms,
                         int64_t num_pairs, int64_t* out);

/*
 * Programmatic dependent launch of the library's kernels: 1 (the default)
 * launches each kernel with CUDA's programmatic-stream-serialization
 * attribute, so a kernel queued behind another on the same stream is
 * scheduled while that one finishes and prepares its barriers meanwhile; it
 * still waits for the earlier kernel to complete (and its writes to become
 * visible) before it reads or writes any argument buffer, so results and
 * stream order are the same either way.  0 launches the kernels plainly.
 * Process-wide.  Returns TMAGEMM_ERR_INVALID for other values.
 */
int tmagemm_set_pdl(int on);

/* ---- host-side introspection of the kernels' schedule (no GPU needed) ---- */

/*
 * Output tile visited as linear id `tile` of a grid of grid_m x grid_n tiles
 * with `group_m` tile rows per L2 group: *m_blk, *n_blk receive the tile's row
 * and column.  This is the same function the GEMM kernel runs.  Returns
 * TMAGEMM_ERR_INVALID for out-of-range input.
 */
int tmagemm_tile_coord(int64_t tile, int64_t grid_m, int64_t grid_n, int64_t group_m,
                       int64_t* m_blk, int64_t* n_blk);

/*
 * Position of k-block iteration `it` (counted over the whole life of a CTA,
 * across tiles) in a ring of `stages` SMEM stages: *stage = it % stages and
 * *phase = parity of the stage's mbarrier phase for that use.  Same function
 * as the kernel's producer and MMA loops.
 */
int tmagemm_ring_position(int64_t it, int64_t stages, int64_t* stage, int64_t* phase);

/*
 * The GEMM launch configuration for (M, N, K) on a device with `num_sms` SMs,
 * of which `num_pairs` two-CTA clusters can be co-resident (0 = no pairs), and
 * a split request (1 = gemm_f16, 0 = automatic split-K, > 1 = that many
 * parts): written to out[0..13] in the order BM, BN, BK, STAGES, tiles, grid
 * (CTAs), threads, smem bytes, parts, k-blocks per part, work units, pair
 * (1 if CTA pairs; then tiles are 256 rows high), cluster split (0, or the
 * number of CTAs (pairs) per cluster that split K for gemm_f16; then parts
 * == that number), GROUP_M (tile rows per L2 group of the tile order).
 * `out` holds 14 values.  No GPU needed: cluster splits
 * assume ideal packing of clusters here, while gemm_f16 also checks how many
 * clusters the device can hold at once.  num_sms == 0 asks instead for the
 * plan gemm_f16 runs on the current device (its SMs, CTA pairs and cluster
 * co-residency; num_pairs is then ignored and a CUDA device is required).
 */
int tmagemm_gemm_plan(int64_t M, int64_t N, int64_t K, int64_t num_sms, int64_t num_pairs,
                      int64_t splits, int64_t* out);

/*
 * The tail split of the gemm_f16 plan for (M, N, K) on `num_sms` SMs with
 * `num_pairs` co-resident CTA pairs (num_sms == 0: the current device, as for
 * tmagemm_gemm_plan): out[0] = work units that are whole tiles, out[1] = tiles
 * of the last round split in two (each two units; tmagemm_gemm_plan's unit
 * count includes both), out[2] = columns of each split tile's first part
 * (0 when nothing is split).  `out` holds 3 values.
 */
int tmagemm_gemm_tail_plan(int64_t M, int64_t N, int64_t K, int64_t num_sms, int64_t num_pairs,
                           int64_t* out);

/*
 * Host-buffer executor: GEMMs whose operands and results live in host memory.
 * The paper pages have no counterpart; it is the end-to-end path of the
 * library.  A step copies A_i (M x K) and B_i (N x K) host -> device, runs
 * gemm_f16 (gemm_bf16 when created with bf16 = 1) and copies D_i (M x N)
 * device -> host.  Three streams carry the three phases and `depth` device
 * slots rotate, so the input copies of step i+1, the GEMM of step i and the
 * result copy of step i-1 overlap; events order the phases of one slot.
 * Every step moves all of its own bytes (one cudaMemcpyAsync per copy).
 *   create     : allocates `depth` (1..16) slots of device memory for A, B
 *                and D on the current device (the only device allocation the
 *                library makes), three non-blocking streams and the events.
 *                TMAGEMM_ERR_INVALID for bad sizes, TMAGEMM_ERR_CUDA if an
 *                allocation fails.
 *   run        : enqueues `steps` steps and returns without waiting; A_host,
 *                B_host, D_host are arrays of `steps` host pointers (host
 *                memory should be page-locked for the copies to overlap; the
 *                caller keeps the buffers alive and unchanged until
 *                synchronize returns).  Status as gemm_f16.
 *   synchronize: waits for every enqueued step and reports a device-side
 *                timeout like tmagemm_check.
 *   destroy    : waits, then frees everything (NULL is a no-op).
 * One object per thread at a time; the object is tied to the device that was
 * current at create.
 */
typedef struct tmagemm_host_pipeline tmagemm_host_pipeline;
int tmagemm_host_pipeline_create(int64_t M, int64_t N, int64_t K, int depth, int bf16,
                                 tmagemm_host_pipeline** out);
int tmagemm_host_pipeline_run(tmagemm_host_pipeline* p, int64_t steps, const void* const* A_host,
                              const void* const* B_host, void* const* D_host);
int tmagemm_host_pipeline_synchronize(tmagemm_host_pipeline* p);
void tmagemm_host_pipeline_destroy(tmagemm_host_pipeline* p);

#ifdef __cplusplus
}
#endif

#endif /* TMAGEMM_H */
