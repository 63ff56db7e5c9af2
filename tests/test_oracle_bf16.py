"""Pins for the oracle's bfloat16 forms (codec, GEMM, GEMV), checked against
things other than the oracle: float32 bit patterns (a bf16 value is the top
half of a binary32), the textbook float32 -> bf16 round-to-nearest-even on
bits, exact rational arithmetic, integer matmul and closed forms."""
from fractions import Fraction
import math

import numpy as np
import pytest

import oracle


def bf16_bits_from_f32(x):
    """Round float32 values to bf16 bits, nearest-even, on the bit pattern
    (finite inputs): add 0x7FFF plus the lowest kept bit, drop 16 bits."""
    u = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


def bf16_value(bits):
    with np.errstate(invalid="ignore"):   # NaN patterns
        return (np.asarray(bits, dtype=np.uint32) << 16).view(np.float32).astype(np.float64)


def frac_to_bf16(q: Fraction) -> float:
    if q == 0:
        return 0.0
    a = abs(q)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    e = max(e, -126)
    ulp = Fraction(2) ** (e - 7)
    v = round(a / ulp) * ulp
    out = math.inf if v >= Fraction(2) ** 128 else float(v)
    return out if q > 0 else -out


def test_bf16_decode_all_bit_patterns():
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bf16_value(pats)
    got = np.array([oracle.bf16_to_double(int(h)) for h in pats])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_bf16_encode_float32_representable_values():
    fin = np.arange(0, 0x7F80, dtype=np.uint32).astype(np.uint16)
    vals32 = (fin.astype(np.uint32) << 16).view(np.float32)
    nxt = (fin.astype(np.uint32) + 1 << 16).view(np.float32)
    mids = ((vals32.astype(np.float64) + nxt.astype(np.float64)) / 2).astype(np.float32)  # exact ties
    up = np.nextafter(mids, np.float32(np.inf))
    down = np.nextafter(mids, np.float32(0))
    rng = np.random.default_rng(5)
    rand = rng.standard_normal(20000).astype(np.float32) * np.float32(3.0)
    allv = np.concatenate([vals32, -vals32, mids, -mids, up, down, rand])
    allv = allv[np.isfinite(allv)]
    ref = bf16_bits_from_f32(allv)
    got = np.array([oracle.double_to_bf16(float(v)) for v in allv], dtype=np.uint16)
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, [(float(allv[i]), hex(got[i]), hex(ref[i])) for i in bad[:5]]


def test_bf16_encode_doubles_vs_rationals():
    rng = np.random.default_rng(6)
    vals = np.concatenate([rng.uniform(-1, 1, 1500),
                           np.ldexp(rng.uniform(0.5, 1, 500), rng.integers(-140, 130, 500))])
    for v in vals:
        assert oracle.bf16_to_double(oracle.double_to_bf16(float(v))) == frac_to_bf16(Fraction(float(v))), v
    assert oracle.double_to_bf16(float("inf")) == 0x7F80
    assert oracle.double_to_bf16(3.5e38) == 0x7F80          # rounds past the largest finite
    assert oracle.double_to_bf16(1.0 + 2.0 ** -8) == 0x3F80   # tie -> even


def bits_bf16(x):
    return bf16_bits_from_f32(np.asarray(x, dtype=np.float32))


@pytest.mark.parametrize("shape", [(1, 1, 1), (3, 5, 7), (6, 4, 32), (2, 7, 31)])
def test_gemm_bf16_exact_rational(shape):
    M, N, K = shape
    rng = np.random.default_rng(M * 100 + N * 10 + K)
    A = bits_bf16(rng.uniform(-1, 1, (M, K)))
    B = bits_bf16(rng.uniform(-1, 1, (N, K)))
    D = oracle.gemm_bf16(A, B)
    Av, Bv = bf16_value(A), bf16_value(B)
    for m in range(M):
        for n in range(N):
            s = sum(Fraction(float(Av[m, k])) * Fraction(float(Bv[n, k])) for k in range(K))
            assert float(bf16_value(D[m, n])) == frac_to_bf16(s), (m, n)


@pytest.mark.parametrize("M,N,K,lo,hi", [(40, 24, 600, -8, 8), (64, 48, 256, -2, 2)])
def test_gemm_bf16_integer_exact(M, N, K, lo, hi):
    rng = np.random.default_rng(M + N + K)
    Ai = rng.integers(lo, hi + 1, (M, K))
    Bi = rng.integers(lo, hi + 1, (N, K))
    exact = Ai @ Bi.T
    D = oracle.gemm_bf16(bits_bf16(Ai), bits_bf16(Bi))
    assert np.array_equal(D, bits_bf16(exact.astype(np.float32)))   # ints < 2^24: exact in f32


def test_gemm_bf16_closed_forms_and_gemv():
    rng = np.random.default_rng(9)
    K, N, M = 48, 40, 33
    B = bits_bf16(rng.uniform(-1, 1, (N, K)))
    A = bits_bf16(rng.uniform(-1, 1, (M, K)))
    I = bits_bf16(np.eye(K))
    assert np.array_equal(oracle.gemm_bf16(I, B), np.ascontiguousarray(B.T))
    assert np.array_equal(oracle.gemm_bf16(A, I), A)
    x = bits_bf16(rng.normal(0, 0.02, K))
    assert np.array_equal(oracle.gemv_bf16(x, B), oracle.gemm_bf16(x[None, :], B)[0])
    e = np.zeros(K)
    e[7] = 1.0
    assert np.array_equal(oracle.gemv_bf16(bits_bf16(e), B), np.ascontiguousarray(B[:, 7]))
