"""CPU oracle for the FP16 TN GEMM ``D = A @ B.T`` and the M=1 GEMV ``y = x @ W.T``.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference leg of ``bench.py`` may import this package.  It shares
no code with the CUDA library in ``tma_pipelined_tensor_tn_gb300`` and imports
nothing from it.

The arithmetic lives in ``oracle.c`` (plain C, FP64 accumulation, k ascending,
one IEEE 754 round-to-nearest-even to binary16 at the end).  This module builds
that file with gcc and marshals numpy ``uint16`` (raw binary16 bits) arrays to it.

Definition followed (see the header of ``oracle.c`` for the passages):
"使用 TMA 为 GEMM 建立 Pipeline", step 4 "完整 Kernel" (A (M,K), B (N,K), D (M,N),
FP32 accumulate, FP16 out); "Learning TileLang with GEMV", §01 GEMV (y = x W^T,
W N x K row-major, FP32 accumulate).
"""
from __future__ import annotations

import ctypes
import hashlib
import os
import platform
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def _stamp() -> str:
    """This machine's architecture and the bytes of ``oracle.c``."""
    with open(_SRC, "rb") as f:
        return hashlib.sha256(platform.machine().encode() + f.read()).hexdigest()


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` into ``liboracle.so`` (gcc, -O2, OpenMP if available),
    unless a library built here from the same source exists."""
    stamp = _LIB + ".stamp"
    if not force and os.path.exists(_LIB) and os.path.exists(stamp):
        with open(stamp) as f:
            if f.read().strip() == _stamp():
                return _LIB
    base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", _SRC, "-o", _LIB + ".tmp", "-lm"]
    # -fno-fast-math keeps IEEE semantics; no -march flags so x86 and Arm agree.
    try:
        subprocess.run(base[:1] + ["-fopenmp", "-fno-fast-math"] + base[1:],
                       check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base[:1] + ["-fno-fast-math"] + base[1:], check=True,
                       capture_output=True)
    os.replace(_LIB + ".tmp", _LIB)
    with open(stamp, "w") as f:
        f.write(_stamp() + "\n")
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            i64, p = ctypes.c_int64, ctypes.c_void_p
            lib.oracle_half_to_double.argtypes = [ctypes.c_uint16]
            lib.oracle_half_to_double.restype = ctypes.c_double
            lib.oracle_double_to_half.argtypes = [ctypes.c_double]
            lib.oracle_double_to_half.restype = ctypes.c_uint16
            lib.oracle_max_threads.argtypes = []
            lib.oracle_max_threads.restype = ctypes.c_int
            lib.oracle_gemm_f16.argtypes = [i64, i64, i64, p, p, p, p, ctypes.c_int]
            lib.oracle_gemm_f16.restype = ctypes.c_int
            lib.oracle_gemm_f16_at.argtypes = [i64, i64, i64, p, p, i64, p, p, p, p,
                                               ctypes.c_int]
            lib.oracle_gemm_f16_at.restype = ctypes.c_int
            lib.oracle_gemv_f16.argtypes = [i64, i64, p, p, p, p, ctypes.c_int]
            lib.oracle_gemv_f16.restype = ctypes.c_int
            lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
            lib.oracle_bf16_to_double.restype = ctypes.c_double
            lib.oracle_double_to_bf16.argtypes = [ctypes.c_double]
            lib.oracle_double_to_bf16.restype = ctypes.c_uint16
            lib.oracle_gemm_bf16.argtypes = [i64, i64, i64, p, p, p, p, ctypes.c_int]
            lib.oracle_gemm_bf16.restype = ctypes.c_int
            lib.oracle_gemv_bf16.argtypes = [i64, i64, p, p, p, p, ctypes.c_int]
            lib.oracle_gemv_bf16.restype = ctypes.c_int
            _lib = lib
    return _lib


def _bits(a: np.ndarray) -> np.ndarray:
    """Accept float16 or uint16 arrays; return a C-contiguous uint16 view."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.float16:
        a = a.view(np.uint16)
    if a.dtype != np.uint16:
        raise TypeError(f"expected float16/uint16 bits, got {a.dtype}")
    return a


def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data)


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def half_to_double(h: int) -> float:
    """Decode one binary16 bit pattern."""
    return float(_load().oracle_half_to_double(int(h) & 0xFFFF))


def double_to_half(x: float) -> int:
    """Encode one double to binary16 bits, round to nearest, ties to even."""
    return int(_load().oracle_double_to_half(float(x)))


def gemm_f16(A, B, *, return_sum: bool = False, threads: int = 0):
    """D = fp16_rne(A @ B.T) with FP64 accumulation.

    A: (M, K) and B: (N, K) binary16 arrays (float16 or uint16 bits).
    Returns D as float16 (M, N); with ``return_sum`` also the FP64 sums.
    """
    A, B = _bits(A), _bits(B)
    M, K = A.shape
    N, K2 = B.shape
    if K != K2:
        raise ValueError("A and B must share K")
    D = np.empty((M, N), dtype=np.uint16)
    S = np.empty((M, N), dtype=np.float64) if return_sum else None
    _load().oracle_gemm_f16(M, N, K, _ptr(A), _ptr(B), _ptr(D),
                            _ptr(S) if S is not None else None, int(threads))
    D = D.view(np.float16)
    return (D, S) if return_sum else D


def gemm_f16_at(A, B, ms, ns, *, return_sum: bool = False, threads: int = 0):
    """D[ms[i], ns[i]] for sampled positions (same definition as ``gemm_f16``)."""
    A, B = _bits(A), _bits(B)
    M, K = A.shape
    N, _ = B.shape
    ms = np.ascontiguousarray(ms, dtype=np.int64)
    ns = np.ascontiguousarray(ns, dtype=np.int64)
    if ms.shape != ns.shape or ms.ndim != 1:
        raise ValueError("ms and ns must be 1-D and equally long")
    if ms.size and (ms.min() < 0 or ms.max() >= M or ns.min() < 0 or ns.max() >= N):
        raise IndexError("sample position out of range")
    out = np.empty(ms.shape, dtype=np.uint16)
    S = np.empty(ms.shape, dtype=np.float64) if return_sum else None
    _load().oracle_gemm_f16_at(M, N, K, _ptr(A), _ptr(B), ms.size, _ptr(ms), _ptr(ns),
                               _ptr(out), _ptr(S) if S is not None else None, int(threads))
    out = out.view(np.float16)
    return (out, S) if return_sum else out


def gemv_f16(x, W, *, return_sum: bool = False, threads: int = 0):
    """y = fp16_rne(x @ W.T) with FP64 accumulation; x: (K,), W: (N, K)."""
    x, W = _bits(x), _bits(W)
    N, K = W.shape
    if x.shape != (K,):
        raise ValueError("x must have length K")
    y = np.empty((N,), dtype=np.uint16)
    S = np.empty((N,), dtype=np.float64) if return_sum else None
    _load().oracle_gemv_f16(N, K, _ptr(x), _ptr(W), _ptr(y),
                            _ptr(S) if S is not None else None, int(threads))
    y = y.view(np.float16)
    return (y, S) if return_sum else y


# ---- bfloat16 forms (operands and results as raw uint16 bit patterns) --------

def _bits16(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError(f"expected uint16 bf16 bit patterns, got {a.dtype}")
    return a


def bf16_to_double(h: int) -> float:
    """Decode one bfloat16 bit pattern."""
    return float(_load().oracle_bf16_to_double(int(h) & 0xFFFF))


def double_to_bf16(x: float) -> int:
    """Encode one double to bfloat16 bits, round to nearest, ties to even."""
    return int(_load().oracle_double_to_bf16(float(x)))


def gemm_bf16(A, B, *, return_sum: bool = False, threads: int = 0):
    """D = bf16_rne(A @ B.T), FP64 accumulation; A (M, K), B (N, K) as uint16
    bf16 bit patterns.  Returns D as uint16 bit patterns (M, N)."""
    A, B = _bits16(A), _bits16(B)
    M, K = A.shape
    N, K2 = B.shape
    if K != K2:
        raise ValueError("A and B must share K")
    D = np.empty((M, N), dtype=np.uint16)
    S = np.empty((M, N), dtype=np.float64) if return_sum else None
    _load().oracle_gemm_bf16(M, N, K, _ptr(A), _ptr(B), _ptr(D),
                             _ptr(S) if S is not None else None, int(threads))
    return (D, S) if return_sum else D


def gemv_bf16(x, W, *, return_sum: bool = False, threads: int = 0):
    """y = bf16_rne(x @ W.T), FP64 accumulation; uint16 bf16 bit patterns."""
    x, W = _bits16(x), _bits16(W)
    N, K = W.shape
    if x.shape != (K,):
        raise ValueError("x must have length K")
    y = np.empty((N,), dtype=np.uint16)
    S = np.empty((N,), dtype=np.float64) if return_sum else None
    _load().oracle_gemv_bf16(N, K, _ptr(x), _ptr(W), _ptr(y),
                             _ptr(S) if S is not None else None, int(threads))
    return (y, S) if return_sum else y


def bf16_bits_to_float64(a) -> np.ndarray:
    """Decode an array of bf16 bit patterns through the oracle's codec table."""
    a = _bits16(a)
    lut = np.array([bf16_to_double(h) for h in range(65536)])
    return lut[a]


def gemm_f16_grouped(A, B, m_offsets, *, threads: int = 0):
    """Grouped GEMM: for each group g, rows [m_offsets[g], m_offsets[g+1]) of
    D are fp16_rne(A[rows] @ B[g].T) with FP64 accumulation.  A: (R, K),
    B: (G, N, K), m_offsets: G + 1 non-decreasing ints from 0 to R.  Each group
    is the plain GEMM definition on its window of A ("高级数据搬运：TMA、Swizzle
    与不规则访问", section "任意偏移窗口：view 与 from": the same computation at
    a run-time origin)."""
    A = _bits(A)
    B = np.ascontiguousarray(B)
    if B.dtype == np.float16:
        B = B.view(np.uint16)
    G, N, K = B.shape
    offs = [int(v) for v in m_offsets]
    if len(offs) != G + 1 or offs[0] != 0 or offs[-1] != A.shape[0]:
        raise ValueError("m_offsets must run from 0 to A.shape[0] with G + 1 entries")
    D = np.empty((A.shape[0], N), dtype=np.float16)
    for g in range(G):
        lo, hi = offs[g], offs[g + 1]
        if hi < lo:
            raise ValueError("m_offsets must be non-decreasing")
        if hi > lo:
            D[lo:hi] = gemm_f16(A[lo:hi], B[g], threads=threads)
    return D
