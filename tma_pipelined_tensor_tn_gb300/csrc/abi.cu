// C ABI of libtmagemm.so (declared in include/tmagemm.h): argument
// validation, TMA tensor-map encoding, per-device state, kernel dispatch and
// the sticky device-side error word.
//
// Tensor maps follow "TensorCore_GEMM_with_TMA" §2.1 init tensor map: a rank-2
// map per operand with sizes {inner, outer} (fastest first), one byte stride
// for the outer dimension, a box of {64 fp16, rows} and 128-byte swizzle for a
// 64-element fp16 row; out-of-range elements read as zero (OOB fill NONE).
// Unlike the page, errors are returned as status codes, never printed.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <cstdlib>
#include <mutex>

#include "../../include/tmagemm.h"
#include "launch.h"
#include "ptx.cuh"
#include "tile_sched.cuh"

namespace tmagemm {

// Sticky per-device error word written by the kernels' bounded waits (and, in
// the checked build, their self-checks), followed there by the work-unit
// counters.
#ifdef TMAGEMM_CHECKED
__device__ uint32_t g_err_word[1 + kCheckUnits];
#else
__device__ uint32_t g_err_word[1];
#endif

namespace {

constexpr int kMaxDevices = 64;

// Process-wide tuning defaults (tmagemm_set_*); each call reads them once, at
// its start, into a Tuning of its own.
int g_force_tile_n = 0;
int g_pair_mode = 0;
int g_cluster_split = 0;
int g_tail_split = 0;
int g_force_group_m = 0;
int g_small_m_route = 0;
int g_pdl = 1;
int g_grouped_t = 0;

struct DeviceState {
    bool ready = false;
    uint64_t ctx_id = 0;    // the context the set-up below belongs to
    int sms = 0;
    int pairs = 0;          // co-resident two-CTA clusters of the pair kernel
    ClusterCaps caps;       // co-resident clusters of the cluster-split kernels
    int cc_major = 0;
    uint32_t* err_word = nullptr;
};

std::mutex g_mutex;
DeviceState g_dev[kMaxDevices];
std::atomic<int> g_last_detail{0};
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
PFN_cuCtxGetCurrent_v4000 g_ctx_current = nullptr;
PFN_cuCtxGetId_v12000 g_ctx_id = nullptr;
std::once_flag g_ctx_fns_once;

uint64_t wait_limit_ns() {
    static const uint64_t v = [] {
        const char* s = std::getenv("TMAGEMM_WAIT_LIMIT_MS");
        long ms = s ? std::strtol(s, nullptr, 10) : 0;
        if (ms <= 0) ms = 2000;
        return static_cast<uint64_t>(ms) * 1000000ull;
    }();
    return v;
}

}  // namespace

Tuning process_tuning() {
    Tuning t;
    t.tile_n = __atomic_load_n(&g_force_tile_n, __ATOMIC_ACQUIRE);
    t.pair_mode = __atomic_load_n(&g_pair_mode, __ATOMIC_ACQUIRE);
    t.cluster_split = __atomic_load_n(&g_cluster_split, __ATOMIC_ACQUIRE);
    t.tail_split = __atomic_load_n(&g_tail_split, __ATOMIC_ACQUIRE);
    t.group_m = __atomic_load_n(&g_force_group_m, __ATOMIC_ACQUIRE);
    t.small_m_route = __atomic_load_n(&g_small_m_route, __ATOMIC_ACQUIRE);
    t.plain_launch = __atomic_load_n(&g_pdl, __ATOMIC_ACQUIRE) ? 0 : 1;
    t.grouped_t = __atomic_load_n(&g_grouped_t, __ATOMIC_ACQUIRE);
    return t;
}

uint64_t current_context_id() {
    std::call_once(g_ctx_fns_once, [] {
        cudaDriverEntryPointQueryResult q{};
        void* fn = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 4000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_ctx_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(fn);
        fn = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_ctx_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(fn);
    });
    if (!g_ctx_current || !g_ctx_id) return 0;
    CUcontext ctx = nullptr;
    if (g_ctx_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
    unsigned long long id = 0;
    if (g_ctx_id(ctx, &id) != CUDA_SUCCESS) return 0;
    return static_cast<uint64_t>(id);
}

namespace {

// Per-device set-up, with that device current: once per context of the
// device (a cudaDeviceReset ends the context; the next call finds a new one
// and repeats the set-up, since the error word's address may have moved).
int device_state(DeviceState** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return TMAGEMM_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return TMAGEMM_ERR_UNSUPPORTED;
    uint64_t ctx = current_context_id();
    if (ctx == 0) {
        // No context current yet: the runtime creates the device's primary
        // context on its first call that needs one, e.g. this look-up.
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_err_word) != cudaSuccess) return TMAGEMM_ERR_CUDA;
        ctx = current_context_id();
    }
    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceState& d = g_dev[dev];
    if (!d.ready || d.ctx_id != ctx) {
        d.ready = false;
        if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return TMAGEMM_ERR_CUDA;
        if (cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev) !=
            cudaSuccess)
            return TMAGEMM_ERR_CUDA;
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_err_word) != cudaSuccess) return TMAGEMM_ERR_CUDA;
        d.err_word = static_cast<uint32_t*>(p);
        if (!g_encode) {
            cudaDriverEntryPointQueryResult q{};
            void* fn = nullptr;
            if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                 cudaEnableDefault, &q) != cudaSuccess ||
                q != cudaDriverEntryPointSuccess || fn == nullptr)
                return TMAGEMM_ERR_CUDA;
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
        }
        if (d.cc_major == 10) {
            d.pairs = max_resident_pairs();
            d.caps = query_cluster_caps();
        }
        d.ctx_id = ctx;
        d.ready = true;
    }
    if (d.cc_major != 10) return TMAGEMM_ERR_UNSUPPORTED;   // sm_100 family only
    *out = &d;
    return TMAGEMM_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Row-major 16-bit (fp16 or bf16) matrix of `rows` x `cols` (cols contiguous)
// as a rank-2 map.
int encode_2d(CUtensorMap* map, const void* base, uint64_t cols, uint64_t rows, uint32_t box_cols,
              uint32_t box_rows, CUtensorMapSwizzle swz, CUtensorMapL2promotion l2,
              bool bf16 = false) {
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * 2};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t estr[2] = {1, 1};
    const CUtensorMapDataType dt =
        bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    CUresult r = g_encode(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, swz, l2,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? TMAGEMM_OK : TMAGEMM_ERR_CUDA;
}

// FP32 split-K workspace [splits][rows][cols] as a rank-3 map, box
// {box_cols, box_rows, 1}; the swizzle span equals the box row (64 or 128 B).
int encode_ws_3d(CUtensorMap* map, void* base, uint64_t cols, uint64_t rows, uint64_t splits,
                 uint32_t box_rows, uint32_t box_cols = 32) {
    cuuint64_t dims[3] = {cols, rows, splits};
    cuuint64_t strides[2] = {cols * 4, cols * rows * 4};
    cuuint32_t box[3] = {box_cols, box_rows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    const CUtensorMapSwizzle swz =
        box_cols * 4 == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B;
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, base, dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? TMAGEMM_OK : TMAGEMM_ERR_CUDA;
}

int validate_common(int64_t a, int64_t b, int64_t c) {
    if (a <= 0 || b <= 0 || c <= 0) return TMAGEMM_ERR_INVALID;
    const int64_t lim = (int64_t(1) << 31) - 1;
    if (a > lim || b > lim || c > lim) return TMAGEMM_ERR_UNSUPPORTED;
    return TMAGEMM_OK;
}

int gemv_impl(int64_t N, int64_t K, const void* x, const void* W, void* y, void* stream, bool bf16,
              const Tuning& t) {
    if (!x || !W || !y) return TMAGEMM_ERR_INVALID;
    if (int s = validate_common(N, K, 1)) return s;
    if (!aligned16(x) || !aligned16(W) || !aligned16(y) || (K % 8) != 0) return TMAGEMM_ERR_ALIGN;
    DeviceState* d = nullptr;
    if (int s = device_state(&d)) return s;
    cudaError_t e = launch_gemv(N, K, x, W, y, bf16, d->sms, static_cast<cudaStream_t>(stream),
                                d->err_word, t.pdl());
    return e == cudaSuccess ? TMAGEMM_OK : TMAGEMM_ERR_CUDA;
}

// Encodes the tensor maps for `plan` and launches it; for a split-K plan also
// the reduction of the workspace into D.
int run_gemm(const GemmPlan& plan, DeviceState* d, int64_t M, int64_t N, int64_t K, const void* A,
             const void* B, void* D, void* workspace, void* stream, const Tuning& t) {
    CUtensorMap tmA, tmB, tmD;
    if (int s = encode_2d(&tmA, A, K, M, plan.bk, plan.a_box_rows, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, plan.bf16))
        return s;
    if (int s = encode_2d(&tmB, B, K, N, plan.bk, plan.b_box_rows, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, plan.bf16))
        return s;
    // Store boxes: 32 rows (each epilogue warp stores its own rows) by one
    // swizzle span: 64 columns (128 B) or 32 columns (64 B) of fp16, 32 of fp32.
    if (plan.out_f32) {
        if (int s = encode_ws_3d(&tmD, workspace, N, M, plan.splits, kEpiWarpRows)) return s;
    } else {
        const CUtensorMapSwizzle dswz =
            plan.epi_cols == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
        if (int s = encode_2d(&tmD, D, N, M, plan.epi_cols, kEpiWarpRows, dswz,
                              CU_TENSOR_MAP_L2_PROMOTION_NONE, plan.bf16))
            return s;
    }
    GemmArgs args;
    args.M = static_cast<int32_t>(M);
    args.N = static_cast<int32_t>(N);
    args.K = static_cast<int32_t>(K);
    args.wait_limit_ns = wait_limit_ns();
    args.err_word = d->err_word;
    args.d_out = D;
    args.pdl = t.pdl();
    // Tail-split parts read B through a box of narrow_b_rows rows.
    CUtensorMap tmBn;
    if (plan.narrow_cols > 0) {
        if (int s = encode_2d(&tmBn, B, K, N, plan.bk, plan.narrow_b_rows,
                              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              plan.bf16))
            return s;
        args.tmBn = &tmBn;
    }
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = launch_gemm_tn(plan, tmA, tmB, tmD, args, st);
    if (e == cudaSuccess && plan.out_f32)
        e = launch_splitk_reduce(workspace, D, M, N, plan.splits, plan.bf16, d->sms, t.pdl(), st);
    return e == cudaSuccess ? TMAGEMM_OK : TMAGEMM_ERR_CUDA;
}

}  // namespace
}  // namespace tmagemm

using namespace tmagemm;

namespace {

enum class SmallMKernel { kSwapAB, kFragments, kLsu, kTile };

// Which kernel gemm_f16_small_m runs for M rows against N weight rows (see
// tmagemm_set_small_m_route).  The automatic choice follows GB300
// measurements:
// - up to 8 rows the register-fragment kernel, fastest everywhere measured
//   (4096 x 14336, M = 8: 19.6 us against 22-23 us for the tile kernel);
// - 9..16 rows the fragments only when their grid fills at least 80 % of its
//   wave (512 of 608 CTAs at N = 4096 or 8192), otherwise the tile kernel's
//   cluster split (M = 16: 14336 x 4096 22.4 against 24.9 us, 11008 x 4096
//   18.9 against 23.8, 6144 x 4096 12.6 against 14.9, where the fragment
//   grid fills 57-74 %);
// - above 16 rows the tile kernel, the fastest or within 7 % of it
//   everywhere (14336 x 4096, M = 17..64: 23-26 us; swap-AB 29-30, LSU-fed
//   49-89).
// Route 2 forces the fragments wherever they apply (M <= 16).
SmallMKernel small_m_kernel(int64_t M, int64_t N, int num_sms, const Tuning& t) {
    const int route = t.small_m_route;
    if (route == 1) return SmallMKernel::kSwapAB;
    if (route == 3) return SmallMKernel::kLsu;
    if (M > small_m_mma_max_m()) return SmallMKernel::kTile;
    if (route == 2 || M <= 8) return SmallMKernel::kFragments;
    return 5 * small_m_mma_ctas(N, num_sms) >= 4 * small_m_mma_wave(num_sms)
               ? SmallMKernel::kFragments
               : SmallMKernel::kTile;
}

// The workspace-free small-M kernels (register fragments, LSU-fed tcgen05),
// fp16 or bf16 operands and output.
int small_m_no_workspace(SmallMKernel k, int64_t M, int64_t N, int64_t K, const void* X,
                         const void* W, void* D, void* stream, bool bf16, const Tuning& t) {
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    DeviceState* d = nullptr;
    if (int s = device_state(&d)) return s;
    if (k == SmallMKernel::kFragments)
        return launch_small_m_mma(M, N, K, X, W, D, st, bf16, d->sms, d->err_word, t.pdl()) ==
                       cudaSuccess
                   ? TMAGEMM_OK
                   : TMAGEMM_ERR_CUDA;
    // X {K, M} in boxes of 64 k x Mp token rows (rows past M read as zero).
    CUtensorMap tmX;
    if (int s = encode_2d(&tmX, X, K, M, 64, small_m_lsu_cols(M), CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, bf16))
        return s;
    return launch_small_m_lsu(tmX, M, N, K, W, D, wait_limit_ns(), d->err_word, st, bf16,
                              t.pdl()) == cudaSuccess
               ? TMAGEMM_OK
               : TMAGEMM_ERR_CUDA;
}

// gemm_f16 / gemm_bf16 with a few rows: runs the register-fragment kernel
// where small_m_kernel picks it (or the LSU-fed kernel up to 64 rows when
// route 3 forces it) and returns true with its status in *status; false if
// the tile kernel should run.
bool few_rows(int64_t M, int64_t N, int64_t K, const void* A, const void* B, void* D,
              void* stream, bool bf16, const Tuning& t, int* status) {
    if (M < 2 || M > 64) return false;
    DeviceState* d = nullptr;
    if (int s = device_state(&d)) {
        *status = s;
        return true;
    }
    const SmallMKernel k = small_m_kernel(M, N, d->sms, t);
    if (k != SmallMKernel::kFragments && k != SmallMKernel::kLsu) return false;
    *status = small_m_no_workspace(k, M, N, K, A, B, D, stream, bf16, t);
    return true;
}

// gemm_f16 / gemm_bf16 under tuning `t`: M = 1 the GEMV (or, with
// m1_route = 1, the tile kernel), a few rows the register-fragment kernel,
// otherwise the tile kernel with the plan for this shape.
int gemm_impl(int64_t M, int64_t N, int64_t K, const void* A, const void* B, void* D, void* stream,
              bool bf16, const Tuning& t) {
    if (!A || !B || !D) return TMAGEMM_ERR_INVALID;
    if (int s = validate_common(M, N, K)) return s;
    if (M == 1 && t.m1_route == 0) return gemv_impl(N, K, A, B, D, stream, bf16, t);
    if (!aligned16(A) || !aligned16(B) || !aligned16(D) || (K % 8) != 0 || (N % 8) != 0)
        return TMAGEMM_ERR_ALIGN;
    // A few rows: the register-fragment kernel streams B fastest up to 16
    // rows (GB300, N = 4096, K = 14336: 21.5 us against 30 us for the tile
    // kernel); above that the tile kernel with its cluster split.
    int fr = TMAGEMM_OK;
    if (few_rows(M, N, K, A, B, D, stream, bf16, t, &fr)) return fr;
    DeviceState* d = nullptr;
    if (int s = device_state(&d)) return s;
    return run_gemm(plan_gemm(M, N, K, d->sms, t, 1, bf16, d->pairs, d->caps), d, M, N, K, A, B, D,
                    nullptr, stream, t);
}

// The per-call options as a Tuning; TMAGEMM_ERR_INVALID for a value outside
// its documented range.
int tuning_from_options(const tmagemm_options* o, Tuning* t) {
    if (!o) {
        *t = process_tuning();
        return TMAGEMM_OK;
    }
    const int32_t bn = o->tile_n, ck = o->cluster_split;
    if ((bn != 0 && bn != 256 && bn != 224 && bn != 192 && bn != 128) || o->cta_pair < 0 ||
        o->cta_pair > 2 || (ck != 0 && ck != 1 && ck != 2 && ck != 4 && ck != 8) ||
        o->tail_split < 0 || o->tail_split > 1 || o->group_m < 0 || o->group_m > 64 ||
        o->small_m_route < 0 || o->small_m_route > 3 || o->plain_launch < 0 ||
        o->plain_launch > 1 || o->m1_route < 0 || o->m1_route > 1)
        return TMAGEMM_ERR_INVALID;
    t->tile_n = bn;
    t->pair_mode = o->cta_pair;
    t->cluster_split = ck;
    t->tail_split = o->tail_split;
    t->group_m = o->group_m;
    t->small_m_route = o->small_m_route;
    t->plain_launch = o->plain_launch;
    t->m1_route = o->m1_route;
    return TMAGEMM_OK;
}

// Columns of the tcgen05 swap-AB tile for M activation rows: 16, else 64.
// Rows 17..32 run padded to 64: on GB300 the 64-wide configuration measured
// 33 us against 37 us for the 32-wide one at N = 4096, K = 14336.
int64_t small_m_tile_rows(int64_t M) { return M <= 16 ? M : 64; }

}  // namespace

extern "C" {

int gemm_f16(int64_t M, int64_t N, int64_t K, const void* A, const void* B, void* D,
             void* stream) {
    return gemm_impl(M, N, K, A, B, D, stream, false, process_tuning());
}

int gemm_bf16(int64_t M, int64_t N, int64_t K, const void* A, const void* B, void* D,
              void* stream) {
    return gemm_impl(M, N, K, A, B, D, stream, true, process_tuning());
}

void tmagemm_options_init(tmagemm_options* opts) {
    if (opts) *opts = tmagemm_options{};
}

int gemm_f16_ex(int64_t M, int64_t N, int64_t K, const void* A, const void* B, void* D,
                const tmagemm_options* opts, void* stream) {
    Tuning t;
    if (int s = tuning_from_options(opts, &t)) return s;
    return gemm_impl(M, N, K, A, B, D, stream, false, t);
}

int gemm_bf16_ex(int64_t M, int64_t N, int64_t K, const void* A, const void* B, void* D,
                 const tmagemm_options* opts, void* stream) {
    Tuning t;
    if (int s = tuning_from_options(opts, &t)) return s;
    return gemm_impl(M, N, K, A, B, D, stream, true, t);
}

int64_t gemm_f16_splitk_workspace_size(int64_t M, int64_t N, int64_t K, int64_t splits) {
    if (splits < 0 || splits > 4096) return TMAGEMM_ERR_INVALID;
    if (int s = validate_common(M, N, K)) return s;
    if (M == 1) return 0;
    DeviceState* d = nullptr;
    if (int s = device_state(&d)) return s;
    const GemmPlan p = plan_gemm(M, N, K, d->sms, process_tuning(), splits == 0 ? 0 : splits);
    // No FP32 partials (one part, or gemm_f16's own plan): no workspace.
    if (!p.out_f32 || p.splits <= 1) return 0;
    return p.splits * M * N * 4;
}

int gemm_f16_splitk(int64_t M, int64_t N, int64_t K, const void* A, const void* B, void* D,
                    int64_t splits, void* workspace, int64_t workspace_bytes, void* stream) {
    if (!A || !B || !D) return TMAGEMM_ERR_INVALID;
    if (splits < 0 || splits > 4096) return TMAGEMM_ERR_INVALID;
    if (int s = validate_common(M, N, K)) return s;
    const Tuning t = process_tuning();
    if (M == 1) return gemv_impl(N, K, A, B, D, stream, false, t);
    if (!aligned16(A) || !aligned16(B) || !aligned16(D) || (K % 8) != 0 || (N % 8) != 0)
        return TMAGEMM_ERR_ALIGN;
    DeviceState* d = nullptr;
    if (int s = device_state(&d)) return s;
    const GemmPlan p = plan_gemm(M, N, K, d->sms, t, splits == 0 ? 0 : splits);
    if (!p.out_f32 || p.splits <= 1)   // no FP32 partials: gemm_f16's plan, no workspace
        return run_gemm(plan_gemm(M, N, K, d->sms, t, 1, false, d->pairs, d->caps), d, M, N, K, A,
                        B, D, nullptr, stream, t);
    if (!workspace || !aligned16(workspace) || workspace_bytes < p.splits * M * N * 4)
        return TMAGEMM_ERR_WORKSPACE;
    return run_gemm(p, d, M, N, K, A, B, D, workspace, stream, t);
}

int gemv_f16(int64_t N, int64_t K, const void* x, const void* W, void* y, void* stream) {
    return gemv_impl(N, K, x, W, y, stream, false, process_tuning());
}

int gemv_bf16(int64_t N, int64_t K, const void* x, const void* W, void* y, void* stream) {
    return gemv_impl(N, K, x, W, y, stream, true, process_tuning());
}

int gemm_f16_grouped(int64_t G, const int64_t* m_offsets, int64_t N, int64_t K, const void* A,
                     const void* B, void* D, void* stream) {
    if (!m_offsets || !A || !B || !D || G <= 0) return TMAGEMM_ERR_INVALID;
    if (G > kMaxGroupsHost) return TMAGEMM_ERR_UNSUPPORTED;
    if (m_offsets[0] != 0) return TMAGEMM_ERR_INVALID;
    for (int64_t g = 0; g < G; ++g)
        if (m_offsets[g + 1] < m_offsets[g]) return TMAGEMM_ERR_INVALID;
    const int64_t rows = m_offsets[G];
    if (rows == 0) return TMAGEMM_OK;                     // nothing to compute
    if (int s = validate_common(rows, N, K)) return s;
    if (G * N > (int64_t(1) << 31) - 1) return TMAGEMM_ERR_UNSUPPORTED;
    if (!aligned16(A) || !aligned16(B) || !aligned16(D) || (K % 8) != 0 || (N % 8) != 0)
        return TMAGEMM_ERR_ALIGN;
    const Tuning t = process_tuning();
    DeviceState* d = nullptr;
    if (int s = device_state(&d)) return s;
    GroupedLaunch g{};
    g.m_offsets = m_offsets;
    g.groups = G;
    g.N = N;
    g.K = K;
    plan_grouped(m_offsets, G, N, d->sms, d->pairs, t, &g);
    // The weights B as {K, N, G}: the narrow operand of row tiles (box of bn
    // rows, bn / 2 per CTA of a pair), the 128-row operand of transposed ones.
    {
        const uint32_t b_rows = g.transposed ? 128u : static_cast<uint32_t>(g.pair ? g.bn / 2 : g.bn);
        cuuint64_t dims[3] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(N),
                              static_cast<cuuint64_t>(G)};
        cuuint64_t strides[2] = {static_cast<cuuint64_t>(K) * 2, static_cast<cuuint64_t>(N * K) * 2};
        cuuint32_t box[3] = {64, b_rows, 1};
        cuuint32_t estr[3] = {1, 1, 1};
        if (g_encode(&g.tmB, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void*>(B), dims, strides,
                     box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return TMAGEMM_ERR_CUDA;
    }
    if (g.transposed) {
        // A's rows are the narrow operand, the weights "A".  A block of w rows
        // loads exactly its rows (w / 2 per CTA of a pair): one map per block
        // width in use, box {64, w / CTAs per tile}.  A group of `steps`
        // 16-row steps has blocks of q and (if the division leaves a
        // remainder) q + 1 steps.
        g.tmA = g.tmB;
        g.x_used = 0;
        const int64_t maxw16 = g.maxw / 16;
        for (int64_t i = 0; i < G; ++i) {
            const int64_t steps = (m_offsets[i + 1] - m_offsets[i] + 15) / 16;
            if (steps == 0) continue;
            const int64_t tb = (steps + maxw16 - 1) / maxw16;
            const int64_t q = steps / tb;
            g.x_used |= 1u << (q - 1);
            if (steps % tb != 0) g.x_used |= 1u << q;
        }
        for (int j = 0; j < 16; ++j) {
            if (!(g.x_used & (1u << j))) continue;
            const int64_t box_rows = 16 * (j + 1) / (g.pair ? 2 : 1);
            if (int s = encode_2d(&g.tmXw[j], A, K, rows, 64, box_rows, CU_TENSOR_MAP_SWIZZLE_128B,
                                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B))
                return s;
        }
        // D as one map (64 rows x 128 columns per store, inside a group) and
        // per group (16 x 128, clipped at the group's last row); unswizzled.
        if (int s = encode_2d(&g.tmD64, D, N, rows, 128, 64, CU_TENSOR_MAP_SWIZZLE_NONE,
                              CU_TENSOR_MAP_L2_PROMOTION_NONE))
            return s;
        for (int64_t i = 0; i < G; ++i) {
            const int64_t mg = m_offsets[i + 1] - m_offsets[i];
            if (mg == 0) continue;   // an empty group has no tiles and no map
            const void* base = static_cast<const uint16_t*>(D) + m_offsets[i] * N;
            if (int s = encode_2d(&g.tmD[i], base, N, mg, 128, 16, CU_TENSOR_MAP_SWIZZLE_NONE,
                                  CU_TENSOR_MAP_L2_PROMOTION_NONE))
                return s;
        }
    } else {
        const int epi_cols = g.bn == 224 ? 32 : 64;
        if (int s = encode_2d(&g.tmA, A, K, rows, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B))
            return s;
        const CUtensorMapSwizzle dswz =
            epi_cols == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
        for (int64_t i = 0; i < G; ++i) {
            const int64_t mg = m_offsets[i + 1] - m_offsets[i];
            if (mg == 0) continue;   // an empty group has no tiles and no map
            const void* base = static_cast<const uint16_t*>(D) + m_offsets[i] * N;
            if (int s = encode_2d(&g.tmD[i], base, N, mg, epi_cols, kEpiWarpRows, dswz,
                                  CU_TENSOR_MAP_L2_PROMOTION_NONE))
                return s;
        }
    }
    GemmArgs args;
    args.M = static_cast<int32_t>(rows);
    args.N = static_cast<int32_t>(N);
    args.K = static_cast<int32_t>(K);
    args.wait_limit_ns = wait_limit_ns();
    args.err_word = d->err_word;
    args.pdl = t.pdl();
    cudaError_t e = launch_grouped(g, d->sms, d->pairs, args, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? TMAGEMM_OK : TMAGEMM_ERR_CUDA;
}

int64_t gemm_f16_small_m_workspace_size(int64_t M, int64_t N, int64_t K) {
    if (int s = validate_common(M, N, K)) return s;
    if (M < 2 || M > 64) return TMAGEMM_ERR_UNSUPPORTED;
    // Only swap-AB needs one (route 1, which does not depend on the shape).
    const Tuning t = process_tuning();
    if (small_m_kernel(M, N, 0, t) != SmallMKernel::kSwapAB) return 0;
    DeviceState* d = nullptr;
    if (int s = device_state(&d)) return s;
    const GemmPlan p = plan_small_m(small_m_tile_rows(M), N, K, d->sms, 0, t);
    return p.splits * N * p.bn * 4;
}

int gemm_f16_small_m(int64_t M, int64_t N, int64_t K, const void* X, const void* W, void* D,
                     void* workspace, int64_t workspace_bytes, void* stream) {
    if (!X || !W || !D) return TMAGEMM_ERR_INVALID;
    if (int s = validate_common(M, N, K)) return s;
    if (M < 2 || M > 64) return TMAGEMM_ERR_UNSUPPORTED;
    if (!aligned16(X) || !aligned16(W) || !aligned16(D) || (K % 8) != 0 || (N % 8) != 0)
        return TMAGEMM_ERR_ALIGN;
    const Tuning t = process_tuning();
    DeviceState* d = nullptr;
    if (int s = device_state(&d)) return s;
    const SmallMKernel kern = small_m_kernel(M, N, d->sms, t);
    if (kern == SmallMKernel::kTile) return gemm_impl(M, N, K, X, W, D, stream, false, t);
    if (kern != SmallMKernel::kSwapAB)
        return small_m_no_workspace(kern, M, N, K, X, W, D, stream, false, t);
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    const GemmPlan p = plan_small_m(small_m_tile_rows(M), N, K, d->sms, 0, t);
    const int64_t need = p.splits * N * p.bn * 4;
    if (!workspace || !aligned16(workspace) || workspace_bytes < need) return TMAGEMM_ERR_WORKSPACE;
    // Swapped roles: the weights are the 128-row operand, the activations the
    // narrow one (rows past M read as zero), partials [splits][N][Mp].
    CUtensorMap tmW, tmX, tmP;
    if (int s = encode_2d(&tmW, W, K, N, p.bk, p.a_box_rows, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B))
        return s;
    if (int s = encode_2d(&tmX, X, K, M, p.bk, p.bn, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B))
        return s;
    if (int s = encode_ws_3d(&tmP, workspace, p.bn, N, p.splits, kEpiWarpRows, p.epi_cols))
        return s;
    GemmArgs args;
    args.M = static_cast<int32_t>(N);
    args.N = static_cast<int32_t>(p.bn);
    args.K = static_cast<int32_t>(K);
    args.wait_limit_ns = wait_limit_ns();
    args.err_word = d->err_word;
    args.pdl = t.pdl();
    cudaError_t e = launch_small_m(p, tmW, tmX, tmP, args, st);
    if (e == cudaSuccess)
        e = launch_small_m_reduce(workspace, D, M, N, p.bn, p.splits, t.pdl(), st);
    return e == cudaSuccess ? TMAGEMM_OK : TMAGEMM_ERR_CUDA;
}

int tmagemm_check(void* stream) {
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return TMAGEMM_ERR_CUDA;
    DeviceState* d = nullptr;
    if (int s = device_state(&d)) return s;
    uint32_t v = 0;
    if (cudaMemcpy(&v, d->err_word, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess)
        return TMAGEMM_ERR_CUDA;
    if (v == 0) return TMAGEMM_OK;
    g_last_detail.store(static_cast<int>(v));
    const uint32_t zero = 0;
    if (cudaMemcpy(d->err_word, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess)
        return TMAGEMM_ERR_CUDA;
    const uint32_t site = v & 0xffu;
    return site >= kSiteCheckRing && site <= kSiteCheckBounds ? TMAGEMM_ERR_CHECK
                                                             : TMAGEMM_ERR_TIMEOUT;
}

int tmagemm_checked_unit_counts(uint32_t* counts, int64_t n, void* stream) {
    if (!kChecked) return TMAGEMM_ERR_UNSUPPORTED;
    if (n < 0 || n > static_cast<int64_t>(kCheckUnits) || (n > 0 && !counts))
        return TMAGEMM_ERR_INVALID;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return TMAGEMM_ERR_CUDA;
    DeviceState* d = nullptr;
    if (int s = device_state(&d)) return s;
    if (n > 0 && cudaMemcpy(counts, d->err_word + 1, static_cast<size_t>(n) * sizeof(uint32_t),
                            cudaMemcpyDeviceToHost) != cudaSuccess)
        return TMAGEMM_ERR_CUDA;
    if (cudaMemset(d->err_word + 1, 0, kCheckUnits * sizeof(uint32_t)) != cudaSuccess)
        return TMAGEMM_ERR_CUDA;
    return TMAGEMM_OK;
}

int tmagemm_last_error_detail(void) { return g_last_detail.load(); }

const char* tmagemm_strerror(int status) {
    switch (status) {
        case TMAGEMM_OK: return "ok";
        case TMAGEMM_ERR_INVALID: return "invalid argument (non-positive size or NULL pointer)";
        case TMAGEMM_ERR_ALIGN:
            return "alignment: pointers must be 16-byte aligned, K % 8 == 0 and N % 8 == 0";
        case TMAGEMM_ERR_UNSUPPORTED: return "unsupported size or device";
        case TMAGEMM_ERR_CUDA: return "CUDA runtime or driver call failed";
        case TMAGEMM_ERR_TIMEOUT: return "device-side pipeline wait timed out";
        case TMAGEMM_ERR_CHECK:
            return "a self-check of the checked build failed (site in tmagemm_last_error_detail)";
        case TMAGEMM_ERR_WORKSPACE:
            return "split-K workspace missing, not 16-byte aligned, or smaller than required";
        case TMAGEMM_ERR_SCRATCH_LIMIT:
            return "problem needs more split-K scratch than the fixed 32 MiB of the "
                   "no-allocation entry point";
        default: return "unknown status";
    }
}

int tmagemm_version(void) { return (0 << 16) | (1 << 8) | 0; }

int tmagemm_set_cta_pair(int mode) {
    if (mode < 0 || mode > 2) return TMAGEMM_ERR_INVALID;
    __atomic_store_n(&g_pair_mode, mode, __ATOMIC_RELEASE);
    return TMAGEMM_OK;
}

int tmagemm_set_tile_n(int bn) {
    if (bn != 0 && bn != 256 && bn != 224 && bn != 192 && bn != 128) return TMAGEMM_ERR_INVALID;
    __atomic_store_n(&g_force_tile_n, bn, __ATOMIC_RELEASE);
    return TMAGEMM_OK;
}

int tmagemm_set_small_m_route(int route) {
    if (route < 0 || route > 3) return TMAGEMM_ERR_INVALID;
    __atomic_store_n(&g_small_m_route, route, __ATOMIC_RELEASE);
    return TMAGEMM_OK;
}

int tmagemm_set_group_m(int g) {
    if (g < 0 || g > 64) return TMAGEMM_ERR_INVALID;
    __atomic_store_n(&g_force_group_m, g, __ATOMIC_RELEASE);
    return TMAGEMM_OK;
}

int tmagemm_set_cluster_split(int mode) {
    if (mode != 0 && mode != 1 && mode != 2 && mode != 4 && mode != 8) return TMAGEMM_ERR_INVALID;
    __atomic_store_n(&g_cluster_split, mode, __ATOMIC_RELEASE);
    return TMAGEMM_OK;
}

int tmagemm_set_tail_split(int mode) {
    if (mode != 0 && mode != 1) return TMAGEMM_ERR_INVALID;
    __atomic_store_n(&g_tail_split, mode, __ATOMIC_RELEASE);
    return TMAGEMM_OK;
}

int tmagemm_set_grouped_transposed(int mode) {
    if (mode < 0 || mode > 2) return TMAGEMM_ERR_INVALID;
    __atomic_store_n(&g_grouped_t, mode, __ATOMIC_RELEASE);
    return TMAGEMM_OK;
}

int tmagemm_grouped_plan(int64_t G, const int64_t* m_offsets, int64_t N, int64_t num_sms,
                         int64_t num_pairs, int64_t* out) {
    if (!out || !m_offsets || G <= 0 || G > kMaxGroupsHost || N <= 0 || num_sms <= 0 ||
        num_pairs < 0 || num_pairs > num_sms / 2 || m_offsets[0] != 0)
        return TMAGEMM_ERR_INVALID;
    for (int64_t g = 0; g < G; ++g)
        if (m_offsets[g + 1] < m_offsets[g]) return TMAGEMM_ERR_INVALID;
    GroupedLaunch gl{};
    plan_grouped(m_offsets, G, N, static_cast<int>(num_sms), static_cast<int>(num_pairs),
                 process_tuning(), &gl);
    out[0] = gl.transposed ? 1 : 0;
    out[1] = gl.pair ? 1 : 0;
    out[2] = gl.bn;
    out[3] = gl.maxw;
    return TMAGEMM_OK;
}

int tmagemm_set_pdl(int on) {
    if (on != 0 && on != 1) return TMAGEMM_ERR_INVALID;
    __atomic_store_n(&g_pdl, on, __ATOMIC_RELEASE);
    return TMAGEMM_OK;
}

int tmagemm_tile_coord(int64_t tile, int64_t grid_m, int64_t grid_n, int64_t group_m,
                       int64_t* m_blk, int64_t* n_blk) {
    if (!m_blk || !n_blk || grid_m <= 0 || grid_n <= 0 || group_m <= 0 || tile < 0 ||
        tile >= grid_m * grid_n)
        return TMAGEMM_ERR_INVALID;
    const TileCoord c = tile_coord(tile, grid_m, grid_n, group_m);
    *m_blk = c.m_blk;
    *n_blk = c.n_blk;
    return TMAGEMM_OK;
}

int tmagemm_ring_position(int64_t it, int64_t stages, int64_t* stage, int64_t* phase) {
    if (!stage || !phase || it < 0 || it > 0xffffffffll || stages <= 0 || stages > 64)
        return TMAGEMM_ERR_INVALID;
    *stage = ring_stage(static_cast<uint32_t>(it), static_cast<uint32_t>(stages));
    *phase = ring_phase(static_cast<uint32_t>(it), static_cast<uint32_t>(stages));
    return TMAGEMM_OK;
}

}  // extern "C"

namespace {

int plan_query(int64_t M, int64_t N, int64_t K, int64_t num_sms, int64_t num_pairs, int64_t splits,
               GemmPlan* p) {
    if (num_sms < 0 || num_pairs < 0 || num_pairs > num_sms / 2 || splits < 0 || splits > 4096)
        return TMAGEMM_ERR_INVALID;
    if (int s = validate_common(M, N, K)) return s;
    if (num_sms == 0) {
        // The plan gemm_f16 runs on the current device.
        DeviceState* d = nullptr;
        if (int s = device_state(&d)) return s;
        *p = plan_gemm(M, N, K, d->sms, process_tuning(), splits, false, d->pairs, d->caps);
    } else {
        *p = plan_gemm(M, N, K, static_cast<int>(num_sms), process_tuning(), splits, false,
                       static_cast<int>(num_pairs));
    }
    return TMAGEMM_OK;
}

}  // namespace

extern "C" {

int tmagemm_gemm_tail_plan(int64_t M, int64_t N, int64_t K, int64_t num_sms, int64_t num_pairs,
                           int64_t* out) {
    if (!out) return TMAGEMM_ERR_INVALID;
    GemmPlan p;
    if (int s = plan_query(M, N, K, num_sms, num_pairs, 1, &p)) return s;
    out[0] = p.full_units;
    out[1] = (p.units - p.full_units) / 2;
    out[2] = p.narrow_cols;
    return TMAGEMM_OK;
}

int tmagemm_gemm_plan(int64_t M, int64_t N, int64_t K, int64_t num_sms, int64_t num_pairs,
                      int64_t splits, int64_t* out) {
    if (!out) return TMAGEMM_ERR_INVALID;
    GemmPlan p;
    if (int s = plan_query(M, N, K, num_sms, num_pairs, splits, &p)) return s;
    out[0] = p.bm;
    out[1] = p.bn;
    out[2] = p.bk;
    out[3] = p.stages;
    out[4] = p.tiles;
    out[5] = p.grid;
    out[6] = p.threads;
    out[7] = p.smem_bytes;
    out[8] = p.splits;
    out[9] = p.kb_per_unit;
    out[10] = p.units;
    out[11] = p.pair ? 1 : 0;
    out[12] = p.cluster_k;
    out[13] = p.group_m;
    return TMAGEMM_OK;
}

int tmagemm_selftest_wait_timeout(int64_t limit_ms, void* stream) {
    if (limit_ms <= 0 || limit_ms > 10000) return TMAGEMM_ERR_INVALID;
    DeviceState* d = nullptr;
    if (int s = device_state(&d)) return s;
    cudaError_t e = launch_wait_timeout_probe(static_cast<uint64_t>(limit_ms) * 1000000ull,
                                              d->err_word, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? TMAGEMM_OK : TMAGEMM_ERR_CUDA;
}

}  // extern "C"

namespace tmagemm {
namespace {

// One block; thread 0 inits an mbarrier expecting one arrival that never
// comes and waits on it with the same bounded wait the GEMM roles use.
__global__ void wait_timeout_probe_kernel(uint64_t limit_ns, uint32_t* err) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        abort_flag = 0;
        mbar_init(smem_u32(&bar), 1);
        fence_mbarrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        (void)wait_or_abort(smem_u32(&bar), 0, &abort_flag, err, kSiteTest, limit_ns);
    }
    __syncthreads();
}

}  // namespace

cudaError_t launch_wait_timeout_probe(uint64_t limit_ns, uint32_t* err_word, cudaStream_t stream) {
    wait_timeout_probe_kernel<<<1, 32, 0, stream>>>(limit_ns, err_word);
    return cudaGetLastError();
}

}  // namespace tmagemm
