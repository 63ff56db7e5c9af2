"""Thin ctypes binding to libtmagemm.so (C ABI in include/tmagemm.h).

Argument marshalling only: every step of the GEMM/GEMV runs in the library's
CUDA kernels.  If the library is missing this module raises; there is no
fallback implementation.
"""
from __future__ import annotations

import ctypes
import os
import threading

_PKG = os.path.dirname(os.path.abspath(__file__))
# TMAGEMM_CHECKED=1 selects the checked build (kernels that check their own
# invariants and count their work units; see tmagemm_checked_unit_counts).
CHECKED = os.environ.get("TMAGEMM_CHECKED", "") == "1"
LIB_PATH = os.path.join(_PKG, "libtmagemm_checked.so" if CHECKED else "libtmagemm.so")

TMAGEMM_OK = 0
TMAGEMM_ERR_INVALID = -1
TMAGEMM_ERR_ALIGN = -2
TMAGEMM_ERR_UNSUPPORTED = -3
TMAGEMM_ERR_CUDA = -4
TMAGEMM_ERR_TIMEOUT = -5
TMAGEMM_ERR_WORKSPACE = -6
TMAGEMM_ERR_SCRATCH_LIMIT = -7
TMAGEMM_ERR_CHECK = -8



class TmagemmOptions(ctypes.Structure):
    """struct tmagemm_options: per-call tuning of gemm_f16_ex / gemm_bf16_ex
    (every field 0 = automatic)."""
    _fields_ = [(name, ctypes.c_int32) for name in (
        "tile_n", "cta_pair", "cluster_split", "tail_split", "group_m", "small_m_route",
        "plain_launch", "m1_route")]


# Every symbol include/tmagemm.h declares, with (argtypes, restype).
_i64, _p, _int = ctypes.c_int64, ctypes.c_void_p, ctypes.c_int
_P64 = ctypes.POINTER(ctypes.c_int64)
_POPT = ctypes.POINTER(TmagemmOptions)
SIGNATURES = {
    "gemm_f16": ([_i64, _i64, _i64, _p, _p, _p, _p], _int),
    "gemm_f16_ex": ([_i64, _i64, _i64, _p, _p, _p, _POPT, _p], _int),
    "gemm_bf16_ex": ([_i64, _i64, _i64, _p, _p, _p, _POPT, _p], _int),
    "tmagemm_options_init": ([_POPT], None),
    "gemv_f16": ([_i64, _i64, _p, _p, _p, _p], _int),
    "gemm_bf16": ([_i64, _i64, _i64, _p, _p, _p, _p], _int),
    "gemm_f16_grouped": ([_i64, _P64, _i64, _i64, _p, _p, _p, _p], _int),
    "gemm_f16_small_m": ([_i64, _i64, _i64, _p, _p, _p, _p, _i64, _p], _int),
    "gemm_f16_small_m_workspace_size": ([_i64, _i64, _i64], _i64),
    "gemv_bf16": ([_i64, _i64, _p, _p, _p, _p], _int),
    "gemm_f16_splitk": ([_i64, _i64, _i64, _p, _p, _p, _i64, _p, _i64, _p], _int),
    "gemm_f16_splitk_workspace_size": ([_i64, _i64, _i64, _i64], _i64),
    "gemm_f16_splitk_noalloc": ([_i64, _i64, _i64, _p, _p, _p, _i64, _p], _int),
    "tmagemm_check": ([_p], _int),
    "tmagemm_last_error_detail": ([], _int),
    "tmagemm_checked_unit_counts": ([ctypes.POINTER(ctypes.c_uint32), _i64, _p], _int),
    "tmagemm_strerror": ([_int], ctypes.c_char_p),
    "tmagemm_version": ([], _int),
    "tmagemm_selftest_wait_timeout": ([_i64, _p], _int),
    "tmagemm_tile_coord": ([_i64, _i64, _i64, _i64, _P64, _P64], _int),
    "tmagemm_ring_position": ([_i64, _i64, _P64, _P64], _int),
    "tmagemm_gemm_plan": ([_i64, _i64, _i64, _i64, _i64, _i64, _P64], _int),
    "tmagemm_gemm_tail_plan": ([_i64, _i64, _i64, _i64, _i64, _P64], _int),
    "tmagemm_set_cta_pair": ([_int], _int),
    "tmagemm_set_tile_n": ([_int], _int),
    "tmagemm_set_pdl": ([_int], _int),
    "tmagemm_set_small_m_route": ([_int], _int),
    "tmagemm_set_cluster_split": ([_int], _int),
    "tmagemm_set_tail_split": ([_int], _int),
    "tmagemm_set_group_m": ([_int], _int),
    "tmagemm_set_grouped_transposed": ([_int], _int),
    "tmagemm_grouped_plan": ([_i64, _P64, _i64, _i64, _i64, _P64], _int),
    "tmagemm_host_pipeline_create": ([_i64, _i64, _i64, _int, _int, ctypes.POINTER(_p)], _int),
    "tmagemm_host_pipeline_run": ([_p, _i64, _p, _p, _p], _int),
    "tmagemm_host_pipeline_synchronize": ([_p], _int),
    "tmagemm_host_pipeline_destroy": ([_p], None),
}

_lock = threading.Lock()
_lib = None


class TmaGemmError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: {strerror(status)} (status {status})" if what else strerror(status))


def lib() -> ctypes.CDLL:
    """The loaded library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"{LIB_PATH} not found: build it first (python -c "
                    "'import __graft_entry__ as g; g.build()')")
            L = ctypes.CDLL(LIB_PATH)
            for name, (argt, rest) in SIGNATURES.items():
                fn = getattr(L, name)
                fn.argtypes = argt
                fn.restype = rest
            _lib = L
    return _lib


def strerror(status: int) -> str:
    return lib().tmagemm_strerror(int(status)).decode()


# ---- raw C-ABI calls (same names as the header) ------------------------------

def gemm_f16(M, N, K, A, B, D, stream=None) -> int:
    return lib().gemm_f16(M, N, K, A, B, D, stream)


def options(**fields) -> TmagemmOptions:
    """A tmagemm_options with the named fields set (tmagemm_options_init first)."""
    o = TmagemmOptions()
    lib().tmagemm_options_init(ctypes.byref(o))
    for k, v in fields.items():
        if k not in dict(TmagemmOptions._fields_):
            raise TypeError(f"unknown option {k!r}")
        setattr(o, k, int(v))
    return o


def gemm_f16_ex(M, N, K, A, B, D, opts=None, stream=None) -> int:
    return lib().gemm_f16_ex(M, N, K, A, B, D, ctypes.byref(opts) if opts is not None else None,
                             stream)


def gemm_bf16_ex(M, N, K, A, B, D, opts=None, stream=None) -> int:
    return lib().gemm_bf16_ex(M, N, K, A, B, D, ctypes.byref(opts) if opts is not None else None,
                              stream)


def gemm_f16_grouped(G, m_offsets, N, K, A, B, D, stream=None) -> int:
    """m_offsets: a sequence of G + 1 host integers."""
    offs = (ctypes.c_int64 * (G + 1))(*[int(v) for v in m_offsets])
    return lib().gemm_f16_grouped(G, offs, N, K, A, B, D, stream)


def gemm_grouped(A, B, m_offsets, out=None, stream=None):
    """Grouped D[rows of g] = A[rows of g] @ B[g].T for CUDA fp16 A (R, K), B (G, N, K)."""
    import torch
    _check_f16_cuda("A", A)
    _check_f16_cuda("B", B)
    G, N, K = B.shape
    R, K2 = A.shape
    if K != K2 or len(m_offsets) != G + 1 or int(m_offsets[-1]) != R:
        raise ValueError("shapes and m_offsets disagree")
    if out is None:
        out = torch.empty((R, N), dtype=torch.float16, device=A.device)
    _check_f16_cuda("out", out)
    with torch.cuda.device(A.device):
        s = gemm_f16_grouped(G, m_offsets, N, K, A.data_ptr(), B.data_ptr(), out.data_ptr(),
                             _stream_handle(stream, A.device))
    if s != TMAGEMM_OK:
        raise TmaGemmError(s, "gemm_f16_grouped")
    return out


def gemm_f16_small_m(M, N, K, X, W, D, workspace, workspace_bytes, stream=None) -> int:
    return lib().gemm_f16_small_m(M, N, K, X, W, D, workspace, workspace_bytes, stream)


def gemm_f16_small_m_workspace_size(M, N, K) -> int:
    return lib().gemm_f16_small_m_workspace_size(M, N, K)


def gemm_small_m(X, W, workspace=None, out=None, stream=None):
    """D = X @ W.T for CUDA fp16 X (M, K) with 2 <= M <= 64 and W (N, K)."""
    import torch
    _check_f16_cuda("X", X)
    _check_f16_cuda("W", W)
    M, K = X.shape
    N, K2 = W.shape
    if K != K2:
        raise ValueError("X and W must share K")
    if out is None:
        out = torch.empty((M, N), dtype=torch.float16, device=X.device)
    _check_f16_cuda("out", out)
    with torch.cuda.device(X.device):
        need = lib().gemm_f16_small_m_workspace_size(M, N, K)
        if need < 0:
            raise TmaGemmError(int(need), "gemm_f16_small_m_workspace_size")
        if workspace is None and need > 0:
            workspace = torch.empty((int(need),), dtype=torch.uint8, device=X.device)
        ws_ptr = workspace.data_ptr() if workspace is not None else None
        ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
        s = lib().gemm_f16_small_m(M, N, K, X.data_ptr(), W.data_ptr(), out.data_ptr(),
                                   ws_ptr, ws_bytes, _stream_handle(stream, X.device))
    if s != TMAGEMM_OK:
        raise TmaGemmError(s, "gemm_f16_small_m")
    return out


def gemm_bf16(M, N, K, A, B, D, stream=None) -> int:
    return lib().gemm_bf16(M, N, K, A, B, D, stream)


def gemv_bf16(N, K, x, W, y, stream=None) -> int:
    return lib().gemv_bf16(N, K, x, W, y, stream)


def gemm_f16_splitk(M, N, K, A, B, D, splits, workspace, workspace_bytes, stream=None) -> int:
    return lib().gemm_f16_splitk(M, N, K, A, B, D, splits, workspace, workspace_bytes, stream)


def gemm_f16_splitk_noalloc(M, N, K, A, B, D, splits, stream=None) -> int:
    """Split-K GEMM using the library's fixed device scratch (no allocation)."""
    return lib().gemm_f16_splitk_noalloc(M, N, K, A, B, D, splits, stream)


def gemm_f16_splitk_workspace_size(M, N, K, splits) -> int:
    return lib().gemm_f16_splitk_workspace_size(M, N, K, splits)


def gemv_f16(N, K, x, W, y, stream=None) -> int:
    return lib().gemv_f16(N, K, x, W, y, stream)


def tmagemm_check(stream=None) -> int:
    return lib().tmagemm_check(stream)


def tmagemm_last_error_detail() -> int:
    return lib().tmagemm_last_error_detail()


def tmagemm_version() -> int:
    return lib().tmagemm_version()


def tmagemm_selftest_wait_timeout(limit_ms, stream=None) -> int:
    return lib().tmagemm_selftest_wait_timeout(limit_ms, stream)


def tmagemm_set_tile_n(bn) -> int:
    return lib().tmagemm_set_tile_n(bn)


def tmagemm_tile_coord(tile, grid_m, grid_n, group_m):
    m, n = ctypes.c_int64(), ctypes.c_int64()
    s = lib().tmagemm_tile_coord(tile, grid_m, grid_n, group_m, ctypes.byref(m), ctypes.byref(n))
    if s != TMAGEMM_OK:
        raise TmaGemmError(s, "tmagemm_tile_coord")
    return m.value, n.value


def tmagemm_ring_position(it, stages):
    st, ph = ctypes.c_int64(), ctypes.c_int64()
    s = lib().tmagemm_ring_position(it, stages, ctypes.byref(st), ctypes.byref(ph))
    if s != TMAGEMM_OK:
        raise TmaGemmError(s, "tmagemm_ring_position")
    return st.value, ph.value


def tmagemm_gemm_plan(M, N, K, num_sms, splits=1, num_pairs=0):
    out = (ctypes.c_int64 * 14)()
    s = lib().tmagemm_gemm_plan(M, N, K, num_sms, num_pairs, splits, out)
    if s != TMAGEMM_OK:
        raise TmaGemmError(s, "tmagemm_gemm_plan")
    keys = ("BM", "BN", "BK", "STAGES", "tiles", "grid", "threads", "smem", "splits",
            "kb_per_unit", "units", "pair", "cluster_k", "group_m")
    return dict(zip(keys, list(out)))


def tmagemm_gemm_tail_plan(M, N, K, num_sms, num_pairs=0):
    out = (ctypes.c_int64 * 3)()
    s = lib().tmagemm_gemm_tail_plan(M, N, K, num_sms, num_pairs, out)
    if s != TMAGEMM_OK:
        raise TmaGemmError(s, "tmagemm_gemm_tail_plan")
    return dict(zip(("full_units", "split_tiles", "narrow_cols"), list(out)))


def tmagemm_set_cta_pair(mode) -> int:
    return lib().tmagemm_set_cta_pair(mode)


def tmagemm_set_pdl(on) -> int:
    return lib().tmagemm_set_pdl(on)


def tmagemm_set_small_m_route(route) -> int:
    return lib().tmagemm_set_small_m_route(route)


def tmagemm_set_cluster_split(mode) -> int:
    return lib().tmagemm_set_cluster_split(mode)


def tmagemm_set_tail_split(mode) -> int:
    return lib().tmagemm_set_tail_split(mode)


def tmagemm_set_grouped_transposed(mode) -> int:
    return lib().tmagemm_set_grouped_transposed(mode)


def tmagemm_grouped_plan(m_offsets, N, num_sms, num_pairs=0):
    G = len(m_offsets) - 1
    offs = (ctypes.c_int64 * (G + 1))(*[int(v) for v in m_offsets])
    out = (ctypes.c_int64 * 4)()
    s = lib().tmagemm_grouped_plan(G, offs, N, num_sms, num_pairs, out)
    if s != TMAGEMM_OK:
        raise TmaGemmError(s, "tmagemm_grouped_plan")
    return dict(zip(("transposed", "pair", "bn", "maxw"), list(out)))


def tmagemm_set_group_m(g) -> int:
    return lib().tmagemm_set_group_m(g)


# ---- torch-tensor conveniences (marshalling only) ----------------------------

def _stream_handle(stream, device):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream)


def _check_f16_cuda(name, t, dtype=None):
    import torch
    dtype = dtype or torch.float16
    if not isinstance(t, torch.Tensor) or t.device.type != "cuda":
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous (row-major)")


def gemm(A, B, out=None, stream=None, opts=None):
    """D = A @ B.T for CUDA fp16 or bf16 tensors A (M, K), B (N, K); returns D (M, N).
    `opts` (a TmagemmOptions, see options()) selects gemm_f16_ex / gemm_bf16_ex."""
    import torch
    dt = A.dtype if A.dtype in (torch.float16, torch.bfloat16) else torch.float16
    _check_f16_cuda("A", A, dt)
    _check_f16_cuda("B", B, dt)
    M, K = A.shape
    N, K2 = B.shape
    if K != K2:
        raise ValueError("A and B must share K")
    if out is None:
        out = torch.empty((M, N), dtype=dt, device=A.device)
    _check_f16_cuda("out", out, dt)
    if tuple(out.shape) != (M, N):
        raise ValueError("out must be (M, N)")
    name = "gemm_bf16" if dt == torch.bfloat16 else "gemm_f16"
    with torch.cuda.device(A.device):
        args = (M, N, K, A.data_ptr(), B.data_ptr(), out.data_ptr())
        if opts is None:
            s = getattr(lib(), name)(*args, _stream_handle(stream, A.device))
        else:
            name += "_ex"
            s = getattr(lib(), name)(*args, ctypes.byref(opts), _stream_handle(stream, A.device))
    if s != TMAGEMM_OK:
        raise TmaGemmError(s, name)
    return out


def gemm_splitk(A, B, workspace=None, splits=0, out=None, stream=None):
    """Split-K D = A @ B.T; `workspace` is a CUDA tensor of at least
    gemm_f16_splitk_workspace_size(...) bytes (allocated here if None)."""
    import torch
    _check_f16_cuda("A", A)
    _check_f16_cuda("B", B)
    M, K = A.shape
    N, K2 = B.shape
    if K != K2:
        raise ValueError("A and B must share K")
    if out is None:
        out = torch.empty((M, N), dtype=torch.float16, device=A.device)
    _check_f16_cuda("out", out)
    with torch.cuda.device(A.device):
        need = lib().gemm_f16_splitk_workspace_size(M, N, K, splits)
        if need < 0:
            raise TmaGemmError(int(need), "gemm_f16_splitk_workspace_size")
        if workspace is None:
            workspace = torch.empty((max(int(need), 16),), dtype=torch.uint8, device=A.device)
        s = lib().gemm_f16_splitk(M, N, K, A.data_ptr(), B.data_ptr(), out.data_ptr(), splits,
                                  workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                                  _stream_handle(stream, A.device))
    if s != TMAGEMM_OK:
        raise TmaGemmError(s, "gemm_f16_splitk")
    return out


def gemv(x, W, out=None, stream=None):
    """y = x @ W.T for CUDA fp16 or bf16 tensors x (K,), W (N, K); returns y (N,)."""
    import torch
    dt = W.dtype if W.dtype in (torch.float16, torch.bfloat16) else torch.float16
    _check_f16_cuda("x", x, dt)
    _check_f16_cuda("W", W, dt)
    N, K = W.shape
    if tuple(x.shape) != (K,):
        raise ValueError("x must be (K,)")
    if out is None:
        out = torch.empty((N,), dtype=dt, device=W.device)
    _check_f16_cuda("out", out, dt)
    fn = lib().gemv_bf16 if dt == torch.bfloat16 else lib().gemv_f16
    with torch.cuda.device(W.device):
        s = fn(N, K, x.data_ptr(), W.data_ptr(), out.data_ptr(), _stream_handle(stream, W.device))
    if s != TMAGEMM_OK:
        raise TmaGemmError(s, "gemv_bf16" if dt == torch.bfloat16 else "gemv_f16")
    return out


def check(stream=None, device=None):
    """Synchronise and raise if a kernel recorded a device-side timeout."""
    import torch
    dev = device if device is not None else torch.cuda.current_device()
    with torch.cuda.device(dev):
        s = lib().tmagemm_check(_stream_handle(stream, dev))
    if s != TMAGEMM_OK:
        raise TmaGemmError(s, f"tmagemm_check (detail 0x{tmagemm_last_error_detail():x})")


def checked_unit_counts(n, stream=None):
    """Checked build: the first n work-unit counters (then zeroed), as a list."""
    import torch
    buf = (ctypes.c_uint32 * max(int(n), 1))()
    dev = torch.cuda.current_device()
    s = lib().tmagemm_checked_unit_counts(buf, int(n), _stream_handle(stream, torch.device("cuda", dev)))
    if s != TMAGEMM_OK:
        raise TmaGemmError(s, "tmagemm_checked_unit_counts")
    return list(buf)[: int(n)]
