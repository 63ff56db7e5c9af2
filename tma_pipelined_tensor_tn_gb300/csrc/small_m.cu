// Skinny GEMM for a few tokens, D = fp16(X W^T) with 2 <= M <= 16 (and the
// same with bf16 operands and output), streamed
// like the GEMV: the weights go from HBM straight into tensor-core register
// fragments, with no shared-memory staging.
//
// The decode step reads each weight once ("Learning TileLang with GEMV", §01
// GEMV, §02 Bandwidth Bound), so the weight stream sets the time.  Per-thread
// 16-byte loads with enough of them in flight keep HBM busier on this part
// than the TMA-fed tcgen05 kernels do at these sizes (the swap-AB kernel
// streams at about 4 TB/s).  The arithmetic, 2 M flops per weight byte,
// still wants tensor cores: mma.sync m16n8k16 (FP16 in, FP32 accumulate)
// takes its operands from registers, which is what lets the weights skip
// shared memory.
//
// Fragment layout.  In m16n8k16 a thread with groupID g = lane / 4 and
// t = lane % 4 holds A(row g and g + 8; k slots 2t, 2t+1, 2t+8, 2t+9) and
// B(k slots 2t, 2t+1, 2t+8, 2t+9; column g).  A dot product does not depend
// on the order of its k terms, so any map from slots to physical k that is
// the same for A and B gives the same sum.  Here two consecutive MMAs (j = 0,
// 1) cover 32 physical k: slot 2t+e of MMA j is k = 8t + 4j + e and slot
// 2t+8+e is k = 8t + 4j + 2 + e.  Thread (g, t) then needs exactly the eight
// consecutive k values 8t .. 8t+7 of weight rows g and g+8 and of token row
// g: one 16-byte load each, and the four threads of a group read 64
// contiguous bytes of each row.
//
// Work split.  A CTA of 4 warps owns 64 weight rows (16 per warp, one MMA
// row tile); the S CTAs of a thread-block cluster (S = 8, 4, 2 or 1, so that
// the grid stays one wave) own the same rows and split K into S slices.  Each CTA leaves its 64 x 8NT FP32 partial
// tile in shared memory; after a cluster barrier each CTA finishes 64 / S of
// the rows, adding the S partials in slice order through distributed shared
// memory, rounding once to fp16 and writing D.  No workspace, one launch,
// deterministic.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "launch.h"
#include "ptx.cuh"

namespace tmagemm {

namespace {

constexpr int kSmWarps = 4;               // warps per CTA, 16 weight rows each
constexpr int kSmRows = 16 * kSmWarps;    // weight rows per CTA and per cluster
constexpr int kSmMaxSlices = 8;           // CTAs per cluster (K slices), at most

__device__ __forceinline__ uint4 ld_weights(const uint4* p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

// c += A * B for one m16n8k16 tile (fp16 or bf16 operands, FP32 accumulators).
template <bool BF16>
__device__ __forceinline__ void mma_m16n8k16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                             uint32_t a3, uint32_t b0, uint32_t b1) {
    if constexpr (BF16)
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
            "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
            : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
    else
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
            "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
            : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ float ld_shared_cluster_f32(uint32_t addr) {
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
    return v;
}

// One group: U steps of 32 k.  Lane (g, t) of step u reads chunk
// c = chunk0 + 4u (8 fp16; chunk0 already includes t) of weight rows g and
// g + 8 and, when XB, of token rows g + 8j; chunks past the slice and rows
// past N or M read as zero.  Without XB the token fragments are read just
// before their MMAs instead (every warp of the CTA reads the same slice of X,
// so those loads hit in L1), which saves 4 U NT registers.
template <int NT, int U, bool XB>
struct Group {
    uint4 wa[U], wb[U];
    uint4 x[XB ? U : 1][XB ? NT : 1];
};

template <int NT, int U, bool XB>
__device__ __forceinline__ void load_group(Group<NT, U, XB>& G, const uint4* wrow_a,
                                           const uint4* wrow_b, const uint4* const (&xrow)[NT],
                                           int32_t chunk0, int32_t c_end) {
    const uint4 z = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const int32_t c = chunk0 + 4 * u;
        const bool ok = c < c_end;
        G.wa[u] = (ok && wrow_a) ? ld_weights(wrow_a + c) : z;
        G.wb[u] = (ok && wrow_b) ? ld_weights(wrow_b + c) : z;
        if constexpr (XB) {
#pragma unroll
            for (int j = 0; j < NT; ++j) G.x[u][j] = (ok && xrow[j]) ? __ldg(xrow[j] + c) : z;
        }
    }
}

template <bool BF16, int NT, int U, bool XB>
__device__ __forceinline__ void mma_group(const Group<NT, U, XB>& G, const uint4* const (&xrow)[NT],
                                          int32_t chunk0, int32_t c_end, float (&acc)[NT][4]) {
    const uint4 z = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const int32_t c = chunk0 + 4 * u;
        const bool ok = c < c_end;
#pragma unroll
        for (int j = 0; j < NT; ++j) {
            uint4 x;
            if constexpr (XB)
                x = G.x[u][j];
            else
                x = (ok && xrow[j]) ? __ldg(xrow[j] + c) : z;
            // MMA 0: physical k 8t + {0,1} (slots 2t, 2t+1) and 8t + {2,3}
            // (slots 2t+8, 2t+9); MMA 1: 8t + {4,5} and 8t + {6,7}.
            mma_m16n8k16<BF16>(acc[j], G.wa[u].x, G.wb[u].x, G.wa[u].y, G.wb[u].y, x.x, x.y);
            mma_m16n8k16<BF16>(acc[j], G.wa[u].z, G.wb[u].z, G.wa[u].w, G.wb[u].w, x.z, x.w);
        }
    }
}

template <int NT, int U, bool XB, int MIN_CTAS, int S, bool BF16>
__global__ void __launch_bounds__(kSmWarps * 32, MIN_CTAS)
small_m_mma_kernel(const uint4* __restrict__ X, const uint4* __restrict__ W,
                   uint16_t* __restrict__ D, int32_t M, int32_t N, int32_t K8, int32_t slice8,
                   uint32_t* __restrict__ err) {
    constexpr int kMp = 8 * NT;
    __shared__ float part[kSmRows][kMp];

    grid_launch_dependents();
    const int lane = static_cast<int>(threadIdx.x) & 31;
    const int warp = static_cast<int>(threadIdx.x) >> 5;
    const int g = lane >> 2, t = lane & 3;
    const uint32_t rank = cluster_ctarank();
    static_assert(S >= 1 && S <= kSmMaxSlices, "cluster of 1..8 CTAs");
    const int32_t row0 = static_cast<int32_t>(blockIdx.x / S) * kSmRows;
    const int32_t ra = row0 + warp * 16 + g, rb = ra + 8;
    const int32_t c_begin = static_cast<int32_t>(rank) * slice8;
    const int32_t c_end = min(K8, c_begin + slice8);

    const uint4* wrow_a = ra < N ? W + static_cast<int64_t>(ra) * K8 : nullptr;
    const uint4* wrow_b = rb < N ? W + static_cast<int64_t>(rb) * K8 : nullptr;
    const uint4* xrow[NT];
#pragma unroll
    for (int j = 0; j < NT; ++j)
        xrow[j] = g + 8 * j < M ? X + static_cast<int64_t>(g + 8 * j) * K8 : nullptr;

    float acc[NT][4] = {};
    // While the previous grid finishes, pull the first eighth of this CTA's K
    // slice of its weight rows into L2 (a prefetch cannot see stale data: L2
    // is where global memory is coherent), so the first loads after the wait
    // hit L2 instead of HBM.
    if (t == 0 && c_end > c_begin) {
        const uint32_t bytes = static_cast<uint32_t>(max(1, (c_end - c_begin) / 8)) * 16u;
        if (wrow_a) prefetch_l2_bytes(wrow_a + c_begin, bytes);
        if (wrow_b) prefetch_l2_bytes(wrow_b + c_begin, bytes);
    }
    grid_dependency_wait();   // X and W may come from the grid before this one

    // Groups of kSmUnroll steps (4 chunks each); group i+1's loads are issued
    // before group i is multiplied.
    constexpr int32_t kGroupChunks = 4 * U;
    const int32_t groups = c_end > c_begin ? (c_end - c_begin + kGroupChunks - 1) / kGroupChunks : 0;
    Group<NT, U, XB> ga, gb;
    if (groups > 0) load_group(ga, wrow_a, wrow_b, xrow, c_begin + t, c_end);
    for (int32_t i = 0; i < groups; i += 2) {
        const int32_t ca = c_begin + t + i * kGroupChunks;
        const int32_t cb = ca + kGroupChunks;
        if (i + 1 < groups) load_group(gb, wrow_a, wrow_b, xrow, cb, c_end);
        mma_group<BF16>(ga, xrow, ca, c_end, acc);
        if (i + 2 < groups) load_group(ga, wrow_a, wrow_b, xrow, cb + kGroupChunks, c_end);
        if (i + 1 < groups) mma_group<BF16>(gb, xrow, cb, c_end, acc);
    }

    // This slice's partial tile: C rows g, g+8 of the warp's 16 weight rows,
    // columns (tokens) 8j + 2t + {0, 1}.
#pragma unroll
    for (int j = 0; j < NT; ++j) {
        part[warp * 16 + g][8 * j + 2 * t] = acc[j][0];
        part[warp * 16 + g][8 * j + 2 * t + 1] = acc[j][1];
        part[warp * 16 + g + 8][8 * j + 2 * t] = acc[j][2];
        part[warp * 16 + g + 8][8 * j + 2 * t + 1] = acc[j][3];
    }
    cluster_sync();   // every slice's partial tile is visible cluster-wide

    // CTA `rank` finishes weight rows [64 rank / S, 64 (rank + 1) / S) of the
    // cluster's 64 (consecutive outputs are consecutive rows, so D is written
    // in runs): each output is the sum of the S slice partials, loaded from
    // the peers' shared memory together and added in slice order.
    const int r_begin = static_cast<int>(rank) * kSmRows / S;
    const int nrows = (static_cast<int>(rank) + 1) * kSmRows / S - r_begin;
    for (int o = static_cast<int>(threadIdx.x); o < nrows * kMp; o += kSmWarps * 32) {
        const int rl = r_begin + o % nrows;
        const int m = o / nrows;
        const uint32_t local = smem_u32(&part[rl][m]);
        float v[S];
#pragma unroll
        for (int q = 0; q < S; ++q) v[q] = ld_shared_cluster_f32(map_to_rank(local, q));
        float sum = v[0];
#pragma unroll
        for (int q = 1; q < S; ++q) sum += v[q];
        const int32_t n = row0 + rl;
        if (m < M && n < N) {
            if constexpr (BF16)
                D[static_cast<int64_t>(m) * N + n] = __bfloat16_as_ushort(__float2bfloat16_rn(sum));
            else
                D[static_cast<int64_t>(m) * N + n] = __half_as_ushort(__float2half_rn(sum));
        }
    }
    cluster_sync();   // peers' shared memory stays alive until every CTA has read it
    if (threadIdx.x == 0) check_count_unit(err, static_cast<int32_t>(blockIdx.x));
}

}  // namespace

int64_t small_m_mma_max_m() { return 16; }

// CTAs the register-fragment kernel launches for N weight rows, and the wave
// it sizes them against (4 per SM): the same slice choice as launch_sliced.
int64_t small_m_mma_ctas(int64_t N, int num_sms) {
    const int64_t groups = (N + kSmRows - 1) / kSmRows;
    const int64_t wave = small_m_mma_wave(num_sms);
    for (int64_t s : {8, 4, 2})
        if (groups * s <= wave) return groups * s;
    return groups;
}

int64_t small_m_mma_wave(int num_sms) { return 4ll * (num_sms > 0 ? num_sms : 152); }

namespace {

// Grid of S-CTA clusters over ceil(N / 64) row groups; K is cut into S
// ranges of whole 4-chunk (32-k) steps.
template <int NT, int U, bool XB, int MIN_CTAS, int S, bool BF16>
cudaError_t launch_variant(int64_t M, int64_t N, int64_t K, const void* X, const void* W, void* D,
                           cudaStream_t stream, uint32_t* err, bool pdl) {
    const int32_t K8 = static_cast<int32_t>(K / 8);
    const int32_t per = (K8 + S - 1) / S;
    const int32_t slice8 = (per + 3) / 4 * 4;
    const int64_t clusters = (N + kSmRows - 1) / kSmRows;
    return launch_kernel(small_m_mma_kernel<NT, U, XB, MIN_CTAS, S, BF16>,
                         dim3(static_cast<unsigned>(clusters * S)), dim3(kSmWarps * 32), 0,
                         stream, static_cast<unsigned>(S), pdl, static_cast<const uint4*>(X),
                         static_cast<const uint4*>(W), static_cast<uint16_t*>(D),
                         static_cast<int32_t>(M), static_cast<int32_t>(N), K8, slice8, err);
}

// Slices per cluster: 8 when the clusters of 64 weight rows are few enough
// for one wave of CTAs (4 per SM: 512 CTAs at N = 4096), fewer for more rows
// so that the grid stays one wave with longer K slices (N = 14336: 2), and
// none (one CTA per 64 rows, whole K) when even 2 slices would not fit in one
// wave (N = 28672: 448 CTAs).
template <int NT, int U, bool BF16>
cudaError_t launch_sliced(int64_t M, int64_t N, int64_t K, const void* X, const void* W, void* D,
                          int num_sms, cudaStream_t stream, uint32_t* err, bool pdl) {
    const int64_t clusters = (N + kSmRows - 1) / kSmRows;
    const int64_t wave = 4ll * (num_sms > 0 ? num_sms : 152);
    if (clusters * 8 <= wave)
        return launch_variant<NT, U, true, 1, 8, BF16>(M, N, K, X, W, D, stream, err, pdl);
    if (clusters * 4 <= wave)
        return launch_variant<NT, U, true, 1, 4, BF16>(M, N, K, X, W, D, stream, err, pdl);
    if (clusters * 2 <= wave)
        return launch_variant<NT, U, true, 1, 2, BF16>(M, N, K, X, W, D, stream, err, pdl);
    return launch_variant<NT, U, true, 1, 1, BF16>(M, N, K, X, W, D, stream, err, pdl);
}

template <bool BF16>
cudaError_t launch_typed(int64_t M, int64_t N, int64_t K, const void* X, const void* W, void* D,
                         int num_sms, cudaStream_t stream, uint32_t* err, bool pdl) {
    if (M <= 8) return launch_sliced<1, 4, BF16>(M, N, K, X, W, D, num_sms, stream, err, pdl);
    if (M <= 16) return launch_sliced<2, 2, BF16>(M, N, K, X, W, D, num_sms, stream, err, pdl);
    return cudaErrorInvalidValue;
}

}  // namespace

// Measured on GB300 at N = 4096, K = 14336 over unroll 2..6, X prefetched or
// not, 1..4 CTAs per SM and 4..8 slices: the best keep every CTA resident
// with loads of both operands in flight.  M <= 8: unroll 4, 128 registers,
// 8 slices (512 CTAs, 4 per SM), 21.3 us.  M <= 16: unroll 2, 110 registers,
// 8 slices, 23.1 us.  A slice count read at run time instead of fixed at
// compile time cost 2 us; above 16 tokens the tcgen05 kernel is faster.
cudaError_t launch_small_m_mma(int64_t M, int64_t N, int64_t K, const void* X, const void* W,
                               void* D, cudaStream_t stream, bool bf16, int num_sms,
                               uint32_t* err, bool pdl) {
    return bf16 ? launch_typed<true>(M, N, K, X, W, D, num_sms, stream, err, pdl)
                : launch_typed<false>(M, N, K, X, W, D, num_sms, stream, err, pdl);
}

}  // namespace tmagemm
