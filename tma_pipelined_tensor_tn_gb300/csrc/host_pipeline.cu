// Host-buffer GEMM executor: operands and results in host memory, copies of
// neighbouring steps overlapped with the GEMMs.
//
// A step copies A_i and B_i host -> device, runs gemm_f16 (or gemm_bf16) and
// copies D_i device -> host.  Three streams carry the three phases and
// `depth` device slots rotate, so the input copies of step i+1, the GEMM of
// step i and the result copy of step i-1 run at the same time.  Events order
// the phases of one slot:
//   input copies of step i   wait until the slot's previous GEMM has read it,
//   GEMM of step i           waits for its inputs and for the slot's previous
//                            result to have left the device,
//   result copy of step i    waits for its GEMM.
// Every step moves all of its own bytes; nothing is cached between steps.
// One cudaMemcpyAsync per copy.  Host buffers should be page-locked for the
// copies to overlap (pageable memory works but serialises).
#include <cuda_runtime.h>
#include <cstdint>
#include <new>
#include <vector>

#include "../../include/tmagemm.h"

struct tmagemm_host_pipeline {
    int64_t M = 0, N = 0, K = 0;
    int depth = 0;
    bool bf16 = false;
    int device = 0;
    cudaStream_t s_h2d = nullptr, s_cmp = nullptr, s_d2h = nullptr;
    std::vector<void*> dA, dB, dD;
    std::vector<cudaEvent_t> ev_h2d, ev_cmp, ev_d2h;
    std::vector<bool> used;
    int64_t next = 0;
};

namespace {

// Makes `device` current for one call and restores the caller's device.
struct DeviceGuard {
    int prev = -1;
    bool ok = false;
    explicit DeviceGuard(int device) {
        ok = cudaGetDevice(&prev) == cudaSuccess && cudaSetDevice(device) == cudaSuccess;
    }
    ~DeviceGuard() {
        if (prev >= 0) cudaSetDevice(prev);
    }
};

void release(tmagemm_host_pipeline* p) {
    if (!p) return;
    DeviceGuard guard(p->device);
    for (cudaStream_t s : {p->s_h2d, p->s_cmp, p->s_d2h})
        if (s) cudaStreamSynchronize(s);
    for (auto* v : {&p->dA, &p->dB, &p->dD})
        for (void* q : *v)
            if (q) cudaFree(q);
    for (auto* v : {&p->ev_h2d, &p->ev_cmp, &p->ev_d2h})
        for (cudaEvent_t e : *v)
            if (e) cudaEventDestroy(e);
    for (cudaStream_t s : {p->s_h2d, p->s_cmp, p->s_d2h})
        if (s) cudaStreamDestroy(s);
    delete p;
}

}  // namespace

extern "C" {

int tmagemm_host_pipeline_create(int64_t M, int64_t N, int64_t K, int depth, int bf16,
                                 tmagemm_host_pipeline** out) {
    if (!out) return TMAGEMM_ERR_INVALID;
    *out = nullptr;
    if (M <= 0 || N <= 0 || K <= 0 || depth < 1 || depth > 16 || (bf16 != 0 && bf16 != 1))
        return TMAGEMM_ERR_INVALID;
    auto* p = new (std::nothrow) tmagemm_host_pipeline();
    if (!p) return TMAGEMM_ERR_CUDA;
    p->M = M;
    p->N = N;
    p->K = K;
    p->depth = depth;
    p->bf16 = bf16 != 0;
    bool ok = cudaGetDevice(&p->device) == cudaSuccess;
    for (cudaStream_t* s : {&p->s_h2d, &p->s_cmp, &p->s_d2h})
        ok = ok && cudaStreamCreateWithFlags(s, cudaStreamNonBlocking) == cudaSuccess;
    p->dA.assign(depth, nullptr);
    p->dB.assign(depth, nullptr);
    p->dD.assign(depth, nullptr);
    p->ev_h2d.assign(depth, nullptr);
    p->ev_cmp.assign(depth, nullptr);
    p->ev_d2h.assign(depth, nullptr);
    p->used.assign(depth, false);
    for (int k = 0; ok && k < depth; ++k) {
        ok = cudaMalloc(&p->dA[k], static_cast<size_t>(M * K * 2)) == cudaSuccess &&
             cudaMalloc(&p->dB[k], static_cast<size_t>(N * K * 2)) == cudaSuccess &&
             cudaMalloc(&p->dD[k], static_cast<size_t>(M * N * 2)) == cudaSuccess &&
             cudaEventCreateWithFlags(&p->ev_h2d[k], cudaEventDisableTiming) == cudaSuccess &&
             cudaEventCreateWithFlags(&p->ev_cmp[k], cudaEventDisableTiming) == cudaSuccess &&
             cudaEventCreateWithFlags(&p->ev_d2h[k], cudaEventDisableTiming) == cudaSuccess;
    }
    if (!ok) {
        release(p);
        return TMAGEMM_ERR_CUDA;
    }
    *out = p;
    return TMAGEMM_OK;
}

int tmagemm_host_pipeline_run(tmagemm_host_pipeline* p, int64_t steps, const void* const* A_host,
                              const void* const* B_host, void* const* D_host) {
    if (!p || steps < 0 || (steps > 0 && (!A_host || !B_host || !D_host)))
        return TMAGEMM_ERR_INVALID;
    for (int64_t i = 0; i < steps; ++i)
        if (!A_host[i] || !B_host[i] || !D_host[i]) return TMAGEMM_ERR_INVALID;
    DeviceGuard guard(p->device);
    if (!guard.ok) return TMAGEMM_ERR_CUDA;
    const size_t a_bytes = static_cast<size_t>(p->M * p->K * 2);
    const size_t b_bytes = static_cast<size_t>(p->N * p->K * 2);
    const size_t d_bytes = static_cast<size_t>(p->M * p->N * 2);
    for (int64_t i = 0; i < steps; ++i) {
        const int k = static_cast<int>(p->next % p->depth);
        const bool again = p->used[k];
        bool ok = true;
        // Inputs: after the slot's previous GEMM has read A and B.
        if (again) ok = cudaStreamWaitEvent(p->s_h2d, p->ev_cmp[k], 0) == cudaSuccess;
        ok = ok &&
             cudaMemcpyAsync(p->dA[k], A_host[i], a_bytes, cudaMemcpyHostToDevice, p->s_h2d) ==
                 cudaSuccess &&
             cudaMemcpyAsync(p->dB[k], B_host[i], b_bytes, cudaMemcpyHostToDevice, p->s_h2d) ==
                 cudaSuccess &&
             cudaEventRecord(p->ev_h2d[k], p->s_h2d) == cudaSuccess;
        // GEMM: after its inputs, and after the slot's previous result left.
        ok = ok && cudaStreamWaitEvent(p->s_cmp, p->ev_h2d[k], 0) == cudaSuccess;
        if (ok && again) ok = cudaStreamWaitEvent(p->s_cmp, p->ev_d2h[k], 0) == cudaSuccess;
        if (!ok) return TMAGEMM_ERR_CUDA;
        const int s = p->bf16 ? gemm_bf16(p->M, p->N, p->K, p->dA[k], p->dB[k], p->dD[k], p->s_cmp)
                              : gemm_f16(p->M, p->N, p->K, p->dA[k], p->dB[k], p->dD[k], p->s_cmp);
        if (s != TMAGEMM_OK) return s;
        // Result: after its GEMM.
        ok = cudaEventRecord(p->ev_cmp[k], p->s_cmp) == cudaSuccess &&
             cudaStreamWaitEvent(p->s_d2h, p->ev_cmp[k], 0) == cudaSuccess &&
             cudaMemcpyAsync(D_host[i], p->dD[k], d_bytes, cudaMemcpyDeviceToHost, p->s_d2h) ==
                 cudaSuccess &&
             cudaEventRecord(p->ev_d2h[k], p->s_d2h) == cudaSuccess;
        if (!ok) return TMAGEMM_ERR_CUDA;
        p->used[k] = true;
        ++p->next;
    }
    return TMAGEMM_OK;
}

int tmagemm_host_pipeline_synchronize(tmagemm_host_pipeline* p) {
    if (!p) return TMAGEMM_ERR_INVALID;
    DeviceGuard guard(p->device);
    if (!guard.ok) return TMAGEMM_ERR_CUDA;
    for (cudaStream_t s : {p->s_h2d, p->s_cmp, p->s_d2h})
        if (cudaStreamSynchronize(s) != cudaSuccess) return TMAGEMM_ERR_CUDA;
    return tmagemm_check(p->s_cmp);
}

void tmagemm_host_pipeline_destroy(tmagemm_host_pipeline* p) { release(p); }

}  // extern "C"
