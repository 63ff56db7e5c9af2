"""Host-buffer GEMM executor: overlaps each step's copies with other steps' work.

A thin binding over the library's native executor (`tmagemm_host_pipeline_*`
in include/tmagemm.h): a step copies A and B from host memory to the device,
runs gemm_f16 (or gemm_bf16) and copies D back.  Three CUDA streams carry the
three phases and `depth` device slots rotate, so the host->device copies of
step i+1, the GEMM of step i and the device->host copy of step i-1 run at the
same time; events order the phases of one slot.  Every step still moves all
of its own inputs and its result across the host link; nothing is cached
between steps.  This module only marshals pointers.
"""
from __future__ import annotations

import ctypes

from . import _binding as B


class HostGemmPipeline:
    def __init__(self, M, N, K, dtype=None, depth=2, device=None):
        import torch
        self.torch = torch
        self.M, self.N, self.K = int(M), int(N), int(K)
        self.dtype = dtype or torch.float16
        if self.dtype not in (torch.float16, torch.bfloat16):
            raise TypeError("dtype must be float16 or bfloat16")
        self.device = torch.device(device if device is not None else "cuda")
        self.depth = int(depth)
        if self.depth < 1:
            raise ValueError("depth must be >= 1")
        self._handle = ctypes.c_void_p()
        self._keep = []   # host tensors of enqueued steps, alive until synchronize()
        with torch.cuda.device(self.device):
            s = B.lib().tmagemm_host_pipeline_create(
                self.M, self.N, self.K, self.depth, 1 if self.dtype == torch.bfloat16 else 0,
                ctypes.byref(self._handle))
        if s != B.TMAGEMM_OK:
            raise B.TmaGemmError(s, "tmagemm_host_pipeline_create")

    def h2d_bytes_per_step(self):
        return 2 * (self.M * self.K + self.N * self.K)

    def d2h_bytes_per_step(self):
        return 2 * self.M * self.N

    def _check_host(self, t, shape, what):
        if t.device.type != "cpu" or t.dtype != self.dtype or tuple(t.shape) != shape \
                or not t.is_contiguous():
            raise ValueError(f"{what} must be a contiguous CPU {self.dtype} tensor of shape {shape}")

    def run(self, host_a, host_b, host_d):
        """Enqueue len(host_a) steps; host_* are lists of CPU tensors (pinned for
        overlap; A_i: M x K, B_i: N x K, D_i: M x N).  Returns without waiting;
        call synchronize() before reading host_d or reusing the inputs."""
        if not (len(host_a) == len(host_b) == len(host_d)):
            raise ValueError("host_a, host_b and host_d must have the same length")
        n = len(host_a)
        for a, b, d in zip(host_a, host_b, host_d):
            self._check_host(a, (self.M, self.K), "A")
            self._check_host(b, (self.N, self.K), "B")
            self._check_host(d, (self.M, self.N), "D")
        arr = ctypes.c_void_p * max(n, 1)
        pa = arr(*[t.data_ptr() for t in host_a])
        pb = arr(*[t.data_ptr() for t in host_b])
        pd = arr(*[t.data_ptr() for t in host_d])
        self._keep.extend(list(host_a) + list(host_b) + list(host_d))
        with self.torch.cuda.device(self.device):
            s = B.lib().tmagemm_host_pipeline_run(self._handle, n, ctypes.cast(pa, ctypes.c_void_p),
                                                  ctypes.cast(pb, ctypes.c_void_p),
                                                  ctypes.cast(pd, ctypes.c_void_p))
        if s != B.TMAGEMM_OK:
            raise B.TmaGemmError(s, "tmagemm_host_pipeline_run")

    def synchronize(self):
        with self.torch.cuda.device(self.device):
            s = B.lib().tmagemm_host_pipeline_synchronize(self._handle)
        self._keep.clear()
        if s != B.TMAGEMM_OK:
            raise B.TmaGemmError(s, "tmagemm_host_pipeline_synchronize")

    def close(self):
        if self._handle:
            B.lib().tmagemm_host_pipeline_destroy(self._handle)
            self._handle = ctypes.c_void_p()
            self._keep.clear()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
