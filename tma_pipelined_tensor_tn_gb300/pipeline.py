"""Host-buffer GEMM executor: overlaps each step's copies with other steps' work.

A step is: copy A_i and B_i from pinned host memory to the device, run
gemm_f16 (or gemm_bf16), copy D_i back to pinned host memory.  Three CUDA
streams carry the three phases and `depth` device buffer slots rotate, so the
host->device copy of step i+1, the GEMM of step i and the device->host copy of
step i-1 run at the same time; events order the phases of one slot:

    h2d[i]     waits until the slot's previous GEMM has read A and B
    compute[i] waits for h2d[i] and for the slot's previous D to be copied out
    d2h[i]     waits for compute[i]

The input copies of a step can also be cut into row blocks on several
streams (copy_streams).

Every step still moves all of its own inputs and its result across the host
link; nothing is cached between steps.  The GEMM itself is the library's C ABI
call (argument marshalling only, through the ctypes binding).
"""
from __future__ import annotations

from . import _binding as B


class HostGemmPipeline:
    def __init__(self, M, N, K, dtype=None, depth=2, device=None, copy_streams=1):
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
        mk = dict(dtype=self.dtype, device=self.device)
        self.slots = [(torch.empty((M, K), **mk), torch.empty((N, K), **mk),
                       torch.empty((M, N), **mk)) for _ in range(self.depth)]
        # Input copies may be cut into `copy_streams` row blocks on their own
        # streams (measured on GB300 at 4096^3: 4 streams gave 332 TFLOP/s end
        # to end against 357 for one, so one is the default).
        self.n_copy = max(1, int(copy_streams))
        self.s_h2d = torch.cuda.Stream(self.device)
        self.s_h2d_extra = [torch.cuda.Stream(self.device) for _ in range(self.n_copy - 1)]
        self.s_cmp = torch.cuda.Stream(self.device)
        self.s_d2h = torch.cuda.Stream(self.device)
        ev = lambda: torch.cuda.Event()   # noqa: E731
        self.ev_h2d = [ev() for _ in range(self.depth)]
        self.ev_cmp = [ev() for _ in range(self.depth)]
        self.ev_d2h = [ev() for _ in range(self.depth)]
        self._used = [False] * self.depth
        self._fn = B.lib().gemm_bf16 if self.dtype == torch.bfloat16 else B.lib().gemm_f16

    def h2d_bytes_per_step(self):
        return 2 * (self.M * self.K + self.N * self.K)

    def d2h_bytes_per_step(self):
        return 2 * self.M * self.N

    def run(self, host_a, host_b, host_d):
        """Enqueue len(host_a) steps; host_* are lists of pinned CPU tensors
        (A_i: M x K, B_i: N x K, D_i: M x N).  Returns without waiting; call
        synchronize() (or wait on the returned event) before reading host_d."""
        torch = self.torch
        if not (len(host_a) == len(host_b) == len(host_d)):
            raise ValueError("host_a, host_b and host_d must have the same length")
        for i, (ha, hb, hd) in enumerate(zip(host_a, host_b, host_d)):
            k = i % self.depth
            dA, dB, dD = self.slots[k]
            streams = [self.s_h2d] + self.s_h2d_extra
            if self._used[k]:
                for st in streams:
                    st.wait_event(self.ev_cmp[k])   # GEMM of the slot's last step read A, B
            pieces = self._row_blocks(dA, ha) + self._row_blocks(dB, hb)
            for j, (dst, src) in enumerate(pieces):
                with torch.cuda.stream(streams[j % len(streams)]):
                    dst.copy_(src, non_blocking=True)
            for st in self.s_h2d_extra:                  # join the copy streams
                ev = torch.cuda.Event()
                ev.record(st)
                self.s_h2d.wait_event(ev)
            self.ev_h2d[k].record(self.s_h2d)
            self.s_cmp.wait_event(self.ev_h2d[k])
            if self._used[k]:
                self.s_cmp.wait_event(self.ev_d2h[k])       # previous D of this slot is out
            s = self._fn(self.M, self.N, self.K, dA.data_ptr(), dB.data_ptr(), dD.data_ptr(),
                         B.ctypes.c_void_p(self.s_cmp.cuda_stream))
            if s != B.TMAGEMM_OK:
                raise B.TmaGemmError(s, "gemm in HostGemmPipeline")
            self.ev_cmp[k].record(self.s_cmp)
            with torch.cuda.stream(self.s_d2h):
                self.s_d2h.wait_event(self.ev_cmp[k])
                hd.copy_(dD, non_blocking=True)
                self.ev_d2h[k].record(self.s_d2h)
            self._used[k] = True
        done = torch.cuda.Event()
        done.record(self.s_d2h)
        return done

    def _row_blocks(self, dst, src):
        """`n_copy` matching row blocks of a device tensor and its host source."""
        rows = dst.shape[0]
        step = -(-rows // self.n_copy)
        return [(dst[r:r + step], src[r:r + step]) for r in range(0, rows, step)]

    def synchronize(self):
        for s in [self.s_h2d] + self.s_h2d_extra + [self.s_cmp, self.s_d2h]:
            s.synchronize()
