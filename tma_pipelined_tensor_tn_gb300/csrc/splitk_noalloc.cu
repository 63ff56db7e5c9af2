// Split-K GEMM for callers that cannot allocate device memory.
//
// gemm_f16_splitk needs a caller-provided FP32 workspace.  Some callers have
// no way to provide one: code that runs after a no-allocation point (a
// latency-critical serving loop where cudaMalloc, which synchronises the
// device, would stall every stream), plugins whose host framework owns all
// device memory through its own pool and exposes no allocator to C, or
// embedded users with a fixed memory budget set at start-up.  For them this
// file holds the workspace itself, as a fixed-size array in the library's own
// device memory, and gemm_f16_splitk_noalloc passes it to the same split-K
// path.  Nothing here calls cudaMalloc, cudaFree or any allocating routine.
//
// The array is part of this file's device module: every GPU that loads it
// keeps its kSplitkScratchBytes until the process exits.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "../../include/tmagemm.h"
#include "launch.h"

namespace tmagemm {
namespace {

// 32 MiB: enough for, e.g., 8 parts of a 1024 x 1024 output or 2 parts of 2048 x 2048.
constexpr int64_t kSplitkScratchBytes = int64_t(32) << 20;

static __device__ __align__(256) float g_splitk_scratch[kSplitkScratchBytes / 4];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
struct ScratchAddress {
    uint64_t ctx = 0;      // the context the address was looked up in
    void* ptr = nullptr;
};
ScratchAddress g_scratch[kMaxDevices];

// The array's device address on the current device.  In host code the name
// g_splitk_scratch is a host-side stand-in, not a device address, so the
// address is looked up with the device current: on the first call in each
// context of the device (after cudaDeviceReset the device's next context
// loads this module anew, and the array may sit elsewhere).
int scratch_for_current_device(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return TMAGEMM_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return TMAGEMM_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    ScratchAddress& a = g_scratch[dev];
    const uint64_t ctx = current_context_id();
    if (a.ptr == nullptr || ctx == 0 || a.ctx != ctx) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_splitk_scratch) != cudaSuccess || p == nullptr)
            return TMAGEMM_ERR_CUDA;
        a.ptr = p;
        // The look-up creates the primary context if there was none yet.
        a.ctx = ctx != 0 ? ctx : current_context_id();
    }
    *out = a.ptr;
    return TMAGEMM_OK;
}

}  // namespace
}  // namespace tmagemm

extern "C" {

int gemm_f16_splitk_noalloc(int64_t M, int64_t N, int64_t K, const void* A, const void* B, void* D,
                            int64_t splits, void* stream) {
    if (!A || !B || !D) return TMAGEMM_ERR_INVALID;
    const int64_t need = gemm_f16_splitk_workspace_size(M, N, K, splits);
    if (need < 0) return static_cast<int>(need);
    if (need > tmagemm::kSplitkScratchBytes) return TMAGEMM_ERR_SCRATCH_LIMIT;
    void* scratch = nullptr;
    if (int s = tmagemm::scratch_for_current_device(&scratch)) return s;
    // The split-K partial kernel writes every element of every part before the
    // reduction reads it, so the array needs no clearing between calls.
    return gemm_f16_splitk(M, N, K, A, B, D, splits, scratch, tmagemm::kSplitkScratchBytes, stream);
}

}  // extern "C"
