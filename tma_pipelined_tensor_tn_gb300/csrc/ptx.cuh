// Device primitives for sm_100-family (sm_103a) kernels, written as inline PTX
// from the public PTX ISA: mbarrier, elect.sync, proxy fences, TMA tensor
// loads/stores with bulk groups, and tcgen05 (TMEM alloc, MMA, commit, ld).
//
// The protocol these wrap is the one the pages build GEMM pipelines on:
//   - one thread issues TMA loads and registers the expected bytes with
//     mbarrier.arrive.expect_tx; the TMA engine's complete_tx counts them down
//     ("使用 TMA 为 GEMM 建立 Pipeline", 第 4 步, 等待 TMA Load 和 Store 完成;
//     TensorCore_GEMM_with_TMA §1.2 mbarrier, §1.3 TMA);
//   - waiters poll mbarrier.try_wait.parity with the phase parity they expect;
//   - TMA stores are grouped with commit_group and waited with wait_group;
//   - the tensor-core MMA is tcgen05.mma into TMEM, completion signalled by
//     tcgen05.commit onto an mbarrier (step 4, "完整 Kernel").
//
// Every wait here is bounded (see wait_or_abort): a handshake that never
// completes ends the kernel with an error code instead of hanging the GPU.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

namespace tmagemm {

// ---------------------------------------------------------------- basics ----

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// One lane of the (fully active) warp returns true.
__device__ __forceinline__ bool elect_one() {
    uint32_t pred = 0;
    asm volatile(
        "{\n\t.reg .pred P;\n\t"
        "elect.sync _|P, 0xffffffff;\n\t"
        "selp.u32 %0, 1, 0, P;\n\t}"
        : "=r"(pred));
    return pred != 0;
}

// Named barrier over `count` threads (a multiple of 32).
__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// Named barrier over `count` threads that also ANDs a per-thread predicate:
// every participant gets the same result.
__device__ __forceinline__ bool named_bar_and(uint32_t id, uint32_t count, bool v) {
    uint32_t out;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 q, %1, 0;\n\t"
        "bar.red.and.pred p, %2, %3, q;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(out)
        : "r"(static_cast<uint32_t>(v)), "r"(id), "r"(count)
        : "memory");
    return out != 0;
}

// -------------------------------------------------------------- mbarrier ----

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Makes mbarrier.init visible to the async proxy (TMA, tcgen05.commit).
__device__ __forceinline__ void fence_mbarrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// One arrival plus `bytes` of expected asynchronous transactions.
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;"
                 ::"r"(bar), "r"(bytes) : "memory");
}

// True once the phase with parity `parity` has completed.
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred P;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 P, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, P;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// ----------------------------------------------------------- error word ----

// Wait-site ids recorded in the error word (bits 0..7).
enum WaitSite : uint32_t {
    kSiteProducerEmpty = 1,
    kSiteMmaFull = 2,
    kSiteMmaAccEmpty = 3,
    kSiteEpiAccFull = 4,
    kSiteDrainFull = 5,
    kSiteDrainMma = 6,
    kSiteTest = 7,
    kSiteGemvFull = 8,
    kSiteGemvX = 9,
    // Checked build only (TMAGEMM_CHECKED): a self-check failed.
    kSiteCheckRing = 11,     // producer and MMA issuer saw different k-block counts
    kSiteCheckTma = 12,      // a TMA coordinate broke the 16-byte rule or was negative
    kSiteCheckBounds = 13,   // an epilogue index left its tile or D
};

// Sticky per-device error word: 0 = fine, otherwise site | (block << 8).
__device__ __forceinline__ void record_error(uint32_t* err_word, uint32_t site) {
    uint32_t code = (site & 0xffu) | ((blockIdx.x & 0xffffffu) << 8);
    atomicCAS(err_word, 0u, code == 0u ? 1u : code);
}

// ----------------------------------------------------------- checked build ----
// Built with -DTMAGEMM_CHECKED, the kernels check their own invariants in place
// of a sanitizer: a failed check records its site in the error word and the
// kernel skips the access (no trap, no assert), and every work unit that
// completes increments its counter in the words after the error word
// (err_word[1 + unit % kCheckUnits]), so the host can see that each unit ran
// exactly once.  In the normal build the checks compile away.
#ifdef TMAGEMM_CHECKED
constexpr bool kChecked = true;
#else
constexpr bool kChecked = false;
#endif
constexpr uint32_t kCheckUnits = 1u << 16;   // unit counters after the error word

__device__ __forceinline__ void check_count_unit(uint32_t* err_word, int32_t unit) {
    if constexpr (kChecked)
        atomicAdd(err_word + 1 + (static_cast<uint32_t>(unit) % kCheckUnits), 1u);
}

// True if `cond` holds (always, in the normal build); otherwise records `site`.
__device__ __forceinline__ bool check_ok(bool cond, uint32_t* err_word, uint32_t site) {
    if constexpr (kChecked) {
        if (!cond) {
            record_error(err_word, site);
            return false;
        }
    }
    return true;
}

// Waits are timed with the SM cycle counter (cheap to read, unlike the global
// timer).  A limit in nanoseconds is converted at 2.5 cycles/ns, above the
// maximum SM clock, so the real time before giving up is never shorter than
// the limit (about 1.2x at the 2.07 GHz maximum, more at lower clocks).
__device__ __forceinline__ uint64_t limit_cycles(uint64_t limit_ns) { return limit_ns * 5u / 2u; }

// Polls `bar` for `parity`.  Gives up (returns false) when the CTA-wide abort
// flag is raised by another role, or after `limit_ns`, in which case it raises
// the flag itself and records `site` in the device error word.
__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity,
                                              volatile int* abort_flag, uint32_t* err_word,
                                              uint32_t site, uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = clock64();
    const uint64_t lim = limit_cycles(limit_ns);
    for (uint32_t spin = 0;; ++spin) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if ((spin & 15u) == 15u && static_cast<uint64_t>(clock64()) - t0 > lim) {
            *abort_flag = 1;
            record_error(err_word, site);
            return false;
        }
    }
}

// Same, but ignores the abort flag: used while draining in-flight copies
// before the CTA exits.
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, uint32_t* err_word,
                                             uint32_t site, uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = clock64();
    const uint64_t lim = limit_cycles(limit_ns);
    for (uint32_t spin = 0;; ++spin) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((spin & 15u) == 15u && static_cast<uint64_t>(clock64()) - t0 > lim) {
            record_error(err_word, site);
            return false;
        }
    }
}

// ------------------------------------------------------------------- TMA ----

__device__ __forceinline__ void tma_prefetch_desc(const void* tmap) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tmap)) : "memory");
}

// 2-D tiled load of box (x = inner coordinate, y = outer) into this CTA's
// shared memory; completion is counted on mbarrier `bar` in bytes.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void* tmap, int32_t x, int32_t y,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];"
        ::"r"(dst), "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

// Prefetch of a 2-D box into L2 only (no shared memory, no completion to
// wait for).  L2 is where global memory is kept coherent, so a prefetched line
// is never stale: a kernel may issue this for its inputs even before the grid
// that writes them has finished.
__device__ __forceinline__ void tma_prefetch_l2_2d(const void* tmap, int32_t x, int32_t y) {
    asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];"
                 ::"l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y)
                 : "memory");
}

// 3-D form of tma_prefetch_l2_2d (x inner, then y, then z).
__device__ __forceinline__ void tma_prefetch_l2_3d(const void* tmap, int32_t x, int32_t y,
                                                   int32_t z) {
    asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];"
                 ::"l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(z)
                 : "memory");
}

// Prefetch of `bytes` contiguous bytes (16-byte aligned start and size) into L2.
__device__ __forceinline__ void prefetch_l2_bytes(const void* p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;"
                 ::"l"(reinterpret_cast<uint64_t>(p)), "r"(bytes)
                 : "memory");
}

// 3-D tiled load (x inner, then y, then z), completion counted on `bar`.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const void* tmap, int32_t x, int32_t y,
                                            int32_t z, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];"
        ::"r"(dst), "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(z), "r"(bar)
        : "memory");
}

// 2-D tiled store of a shared-memory box to global memory (bulk group).
// Elements outside the tensor are not written.
__device__ __forceinline__ void tma_store_2d(const void* tmap, uint32_t src, int32_t x, int32_t y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];"
        ::"l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(src)
        : "memory");
}

// 3-D tiled store (x inner, then y, then z), same rules as the 2-D store.
__device__ __forceinline__ void tma_store_3d(const void* tmap, uint32_t src, int32_t x, int32_t y,
                                             int32_t z) {
    asm volatile(
        "cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%1, %2, %3}], [%4];"
        ::"l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(z), "r"(src)
        : "memory");
}

__device__ __forceinline__ void bulk_commit_group() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// Wait until at most N committed store groups still read shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_group_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

// Wait until at most N committed store groups are still incomplete.
template <int N>
__device__ __forceinline__ void bulk_wait_group() {
    asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}

// Generic-proxy shared-memory writes become visible to the async proxy.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// --------------------------------------------------------------- tcgen05 ----

// Whole warp: allocate `ncols` TMEM columns (power of two >= 32); the TMEM
// address is written to shared memory at `dst`.
__device__ __forceinline__ void tmem_alloc(uint32_t dst, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 ::"r"(dst), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;"
                 ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D(tmem) (+)= A(smem desc) * B(smem desc)^T, kind::f16, one CTA.
__device__ __forceinline__ void mma_f16_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                           uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
        ::"r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive (once) on `bar` when all previously issued tcgen05 async operations
// of this thread have completed.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
        ::"r"(bar) : "memory");
}

// Warp-collective: 32 lanes x 32 consecutive 32-bit columns from TMEM.
// Lane i of the warp reads TMEM lane (taddr.lane + i); v[j] = column (taddr.col + j).
__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&v)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
          "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]),
          "=r"(v[13]), "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]),
          "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]),
          "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]),
          "=r"(v[31])
        : "r"(taddr));
}

// Warp-collective: 32 lanes x 16 consecutive 32-bit columns from TMEM.
__device__ __forceinline__ void tmem_ld_32x32b_x16(uint32_t taddr, uint32_t (&v)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
          "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]),
          "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld_wait() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// ------------------------------------------------ CTA pair (cluster of 2) ----
// A CTA pair runs one 256-row MMA: each CTA holds 128 rows of A and half of
// B in its own shared memory and 128 lanes of the accumulator in its own TMEM;
// the pair's leader (cluster rank 0) issues the MMAs for both.

__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// The shared::cluster address of `addr` (a shared::cta address of this CTA)
// in the shared memory of cluster rank `rank`.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t addr, uint32_t rank) {
    uint32_t out;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(out) : "r"(addr), "r"(rank));
    return out;
}

// Programmatic dependent launch (PTX griddepcontrol).  grid_dependency_wait
// returns once the grids this one depends on have completed and their memory
// writes are visible to it; for a launch without the programmatic-serialization
// attribute it returns at once.  grid_launch_dependents allows the next grid
// on the stream to be scheduled once every CTA of this grid has issued it or
// exited (issuing it more than once per CTA has no further effect).
__device__ __forceinline__ void grid_dependency_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void grid_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// All threads of all CTAs of the cluster.
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// The two halves of cluster_sync, for work placed between them.  Every
// thread of the cluster arrives once and then waits once.
__device__ __forceinline__ void cluster_arrive_release() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait_acquire() {
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Cluster barrier whose arrive carries no release: for the set-up barrier of
// a CTA pair, where the only writes the peer must see are mbarrier
// initialisations already released to the cluster by fence.mbarrier_init,
// and the TMEM allocation, ordered by the tcgen05 fences around it.  (An
// arrive with release waits for the thread's outstanding memory operations;
// on GB300 that cost the pair set-up about 1.3 us.)
__device__ __forceinline__ void cluster_sync_after_init() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Four floats from shared memory at a shared::cluster address (any CTA of
// the cluster); 16-byte aligned.
__device__ __forceinline__ void ld_shared_cluster_v4(uint32_t cluster_addr, float (&v)[4]) {
    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v[0]), "=f"(v[1]), "=f"(v[2]), "=f"(v[3])
                 : "r"(cluster_addr)
                 : "memory");
}

// One arrival on an mbarrier given by its shared::cluster address (any CTA).
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];"
                 ::"r"(cluster_addr) : "memory");
}

// 2-D tiled load into this CTA's shared memory whose bytes are counted on an
// mbarrier of either CTA of the pair (cluster address).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const void* tmap, int32_t x, int32_t y,
                                                 uint32_t bar_cluster) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];"
        ::"r"(dst), "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(bar_cluster)
        : "memory");
}

// 3-D form of tma_load_2d_pair.
__device__ __forceinline__ void tma_load_3d_pair(uint32_t dst, const void* tmap, int32_t x, int32_t y,
                                                 int32_t z, uint32_t bar_cluster) {
    asm volatile(
        "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];"
        ::"r"(dst), "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(z), "r"(bar_cluster)
        : "memory");
}

// Pair-wide TMEM allocation: one warp in EACH CTA of the pair executes it.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;"
                 ::"r"(dst), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tmem_relinquish_pair() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;"
                 ::"r"(taddr), "r"(ncols) : "memory");
}

// D (+)= A * B^T for the pair: M = 256 (128 rows from each CTA's A), N split
// over the two CTAs' B halves; issued by one thread of the leader CTA.
__device__ __forceinline__ void mma_f16_ss_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                                uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}"
        ::"r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive once on the mbarrier at offset `bar` in every CTA of `cta_mask` when
// the pair's previously issued tcgen05 operations complete.
__device__ __forceinline__ void mma_commit_pair(uint32_t bar, uint16_t cta_mask) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
        " [%0], %1;"
        ::"r"(bar), "h"(cta_mask) : "memory");
}

// ------------------------------------------------- UMMA descriptor fields ----

// Shared-memory matrix descriptor (tcgen05 "matrix descriptor"): start address,
// leading/stride byte offsets (all >> 4), the fixed 0b001 at bits 46..48 and
// the swizzle mode in bits 61..63 (2 = 128-byte swizzle).
//
// For a K-major operand tile whose rows are exactly one 128-byte swizzle atom
// wide (64 fp16), rows are grouped in 8-row / 1024-byte atoms: SBO = 1024 B;
// LBO is unused for this layout.  Stepping K by 16 elements (32 bytes) inside
// the atom advances the start address by 32 bytes — the swizzle XOR is taken
// from the address bits, exactly as the TMA engine applied it when writing.
__device__ __forceinline__ uint64_t umma_desc_sw128_kmajor(uint32_t smem_addr) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((smem_addr & 0x3FFFFu) >> 4);      // start address
    d |= static_cast<uint64_t>(1u) << 16;                          // LBO (unused) = 16 B
    d |= static_cast<uint64_t>(1024u >> 4) << 32;                  // SBO = 1024 B
    d |= static_cast<uint64_t>(1u) << 46;                          // fixed 0b001
    d |= static_cast<uint64_t>(2u) << 61;                          // SWIZZLE_128B
    return d;
}

// Instruction descriptor for kind::f16: D fp32, A and B both fp16 or both
// bf16 (never mixed), both K-major, shape M x N (M in {64,128}, N multiple of
// 16 up to 256).
__host__ __device__ constexpr uint32_t umma_idesc_16bit_f32(uint32_t M, uint32_t N, bool bf16) {
    return (1u << 4)                    // D format: F32
         | ((bf16 ? 1u : 0u) << 7)      // A format: F16 (0) or BF16 (1)
         | ((bf16 ? 1u : 0u) << 10)     // B format: the same as A
         | (0u << 15)                   // A K-major
         | (0u << 16)                   // B K-major
         | ((N >> 3) << 17)             // N / 8
         | ((M >> 4) << 24);            // M / 16
}

// Two fp32 -> one packed half2, round to nearest even.
__device__ __forceinline__ uint32_t pack_half2_rn(uint32_t lo_bits, uint32_t hi_bits) {
    __half2 h = __floats2half2_rn(__uint_as_float(lo_bits), __uint_as_float(hi_bits));
    return *reinterpret_cast<uint32_t*>(&h);
}

// Two fp32 -> one packed bfloat162, round to nearest even.
__device__ __forceinline__ uint32_t pack_bf162_rn(uint32_t lo_bits, uint32_t hi_bits) {
    __nv_bfloat162 h = __floats2bfloat162_rn(__uint_as_float(lo_bits), __uint_as_float(hi_bits));
    return *reinterpret_cast<uint32_t*>(&h);
}

template <bool BF16>
__device__ __forceinline__ uint32_t pack2_rn(uint32_t lo_bits, uint32_t hi_bits) {
    if constexpr (BF16)
        return pack_bf162_rn(lo_bits, hi_bits);
    else
        return pack_half2_rn(lo_bits, hi_bits);
}

__device__ __forceinline__ void st_shared_u16(uint32_t addr, uint16_t v) {
    asm volatile("st.shared.u16 [%0], %1;" ::"r"(addr), "h"(v) : "memory");
}

// fp32 bits -> one fp16 or bf16, round to nearest even.
template <bool BF16>
__device__ __forceinline__ uint16_t cvt16_rn(uint32_t f_bits) {
    return static_cast<uint16_t>(pack2_rn<BF16>(f_bits, 0u) & 0xffffu);
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};"
                 ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

}  // namespace tmagemm
