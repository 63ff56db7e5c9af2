"""Pins for the CPU oracle, checked against things other than the oracle itself.

* the binary16 codec against numpy's float16 over all 65536 bit patterns and a
  dense sweep of doubles including every exact tie;
* the GEMM/GEMV sum + rounding against exact rational arithmetic on tiny shapes;
* integer-valued inputs against an exact integer matmul;
* identity, rank-1 and unit-vector closed forms; transpose symmetry;
* the FP32-vs-FP16 accumulation point made in "Learning TileLang with GEMV",
  §5.2 block_split_k (an fp16 running sum stalls).
"""
from fractions import Fraction
import math

import numpy as np
import pytest

import oracle


def f16(x):
    return np.asarray(x, dtype=np.float16)


def bits(a):
    return np.ascontiguousarray(a).view(np.uint16)


# --------------------------------------------------------------------------
# binary16 codec
# --------------------------------------------------------------------------

def test_decode_all_bit_patterns():
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = pats.view(np.float16).astype(np.float64)
    got = np.array([oracle.half_to_double(int(h)) for h in pats])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    # sign of zero
    assert math.copysign(1.0, oracle.half_to_double(0x8000)) == -1.0


def _sweep_values():
    finite = np.arange(0, 0x7C00, dtype=np.uint32).astype(np.uint16).view(np.float16)
    fin = finite.astype(np.float64)
    mids = (fin[:-1] + fin[1:]) / 2.0            # exact ties between neighbours
    above = np.nextafter(mids, np.inf)
    below = np.nextafter(mids, -np.inf)
    rng = np.random.default_rng(1234)
    rand = np.concatenate([
        rng.uniform(-1, 1, 4000),
        np.ldexp(rng.uniform(0.5, 1.0, 4000), rng.integers(-30, 18, 4000)),
        rng.uniform(-7e-5, 7e-5, 2000),          # subnormal range
    ])
    edges = np.array([65504.0, 65519.999, 65520.0, 65536.0, 1e300, -65520.0,
                      2.0 ** -24, 2.0 ** -25, 2.0 ** -25 * 1.0000001, 3 * 2.0 ** -26,
                      2.0 ** -14, 2.0 ** -14 - 2.0 ** -25, 0.0, -0.0])
    return np.concatenate([fin, -fin, mids, -mids, above, below, rand, edges])


def test_encode_matches_numpy_including_ties():
    vals = _sweep_values()
    with np.errstate(over="ignore"):
        ref = vals.astype(np.float16).view(np.uint16)
    got = np.array([oracle.double_to_half(float(v)) for v in vals], dtype=np.uint16)
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, [(vals[i], hex(got[i]), hex(ref[i])) for i in bad[:10]]


def test_encode_special_values():
    assert oracle.double_to_half(float("inf")) == 0x7C00
    assert oracle.double_to_half(float("-inf")) == 0xFC00
    assert (oracle.double_to_half(float("nan")) & 0x7C00) == 0x7C00
    assert oracle.double_to_half(65520.0) == 0x7C00     # tie at max rounds to even -> inf
    assert oracle.double_to_half(65519.0) == 0x7BFF
    assert oracle.double_to_half(1.0 + 2.0 ** -11) == 0x3C00   # tie -> even (1.0)
    assert oracle.double_to_half(1.0 + 3 * 2.0 ** -11) == 0x3C02


# --------------------------------------------------------------------------
# sum + rounding vs exact rationals
# --------------------------------------------------------------------------

def frac_to_f16(q: Fraction) -> float:
    """Exact rational -> nearest binary16 value (ties to even), independent code."""
    if q == 0:
        return 0.0
    a = abs(q)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    e = max(e, -14)
    ulp = Fraction(2) ** (e - 10)
    n = round(a / ulp)               # Fraction rounding: half to even
    v = n * ulp
    if v > 65504:
        out = math.inf
    else:
        out = float(v)
    return out if q > 0 else -out


@pytest.mark.parametrize("shape", [(1, 1, 1), (3, 5, 7), (8, 8, 32), (5, 3, 16), (2, 7, 31)])
@pytest.mark.parametrize("scale", [1.0, 64.0, 1.0 / 256])
def test_gemm_exact_rational(shape, scale):
    M, N, K = shape
    rng = np.random.default_rng(M * 1000 + N * 10 + K)
    A = f16(rng.uniform(-1, 1, (M, K)) * scale)
    B = f16(rng.uniform(-1, 1, (N, K)))
    D = oracle.gemm_f16(A, B)
    for m in range(M):
        for n in range(N):
            s = sum(Fraction(float(A[m, k])) * Fraction(float(B[n, k])) for k in range(K))
            assert float(D[m, n]) == frac_to_f16(s), (m, n)


def test_gemv_exact_rational():
    rng = np.random.default_rng(7)
    N, K = 6, 40
    x = f16(rng.normal(0, 0.02, K))
    W = f16(rng.normal(0, 0.02, (N, K)))
    y = oracle.gemv_f16(x, W)
    for n in range(N):
        s = sum(Fraction(float(x[k])) * Fraction(float(W[n, k])) for k in range(K))
        assert float(y[n]) == frac_to_f16(s)


# --------------------------------------------------------------------------
# integer-valued inputs: exact against integer matmul
# --------------------------------------------------------------------------

@pytest.mark.parametrize("M,N,K,lo,hi", [(64, 48, 200, -2, 2), (129, 67, 256, -2, 2),
                                         (33, 20, 600, -8, 8), (1, 300, 72, -3, 3)])
def test_gemm_integer_exact(M, N, K, lo, hi):
    rng = np.random.default_rng(M + N + K)
    Ai = rng.integers(lo, hi + 1, (M, K))
    Bi = rng.integers(lo, hi + 1, (N, K))
    exact = Ai @ Bi.T                                     # int64, exact
    D = oracle.gemm_f16(f16(Ai), f16(Bi))
    assert np.array_equal(bits(D), bits(exact.astype(np.float64).astype(np.float16)))


def test_gemv_integer_exact():
    rng = np.random.default_rng(3)
    N, K = 100, 1024
    xi = rng.integers(-2, 3, K)
    Wi = rng.integers(-2, 3, (N, K))
    y = oracle.gemv_f16(f16(xi), f16(Wi))
    assert np.array_equal(bits(y), bits((Wi @ xi).astype(np.float64).astype(np.float16)))


# --------------------------------------------------------------------------
# closed forms and invariants
# --------------------------------------------------------------------------

def test_identity_left_gives_B_transpose():
    rng = np.random.default_rng(11)
    K, N = 48, 40
    A = np.eye(K, dtype=np.float16)
    B = f16(rng.uniform(-1, 1, (N, K)))
    D = oracle.gemm_f16(A, B)
    assert np.array_equal(bits(D), bits(np.ascontiguousarray(B.T)))


def test_identity_right_gives_A():
    rng = np.random.default_rng(12)
    M, K = 37, 56
    A = f16(rng.uniform(-1, 1, (M, K)))
    B = np.eye(K, dtype=np.float16)
    D = oracle.gemm_f16(A, B)
    assert np.array_equal(bits(D), bits(A))


def test_rank1_powers_of_two():
    rng = np.random.default_rng(13)
    M, N, K = 20, 24, 64
    a = rng.choice([-1, 1], M) * 2.0 ** rng.integers(-6, 3, M)
    b = rng.choice([-1, 1], N) * 2.0 ** rng.integers(-6, 3, N)
    A = f16(np.repeat(a[:, None], K, axis=1))
    B = f16(np.repeat(b[:, None], K, axis=1))
    D = oracle.gemm_f16(A, B)
    assert np.array_equal(D.astype(np.float64), K * np.outer(a, b))


def test_transpose_symmetry():
    rng = np.random.default_rng(14)
    A = f16(rng.uniform(-1, 1, (23, 96)))
    B = f16(rng.uniform(-1, 1, (31, 96)))
    assert np.array_equal(bits(oracle.gemm_f16(B, A)),
                          bits(np.ascontiguousarray(oracle.gemm_f16(A, B).T)))


def test_gemv_unit_vector_selects_column():
    rng = np.random.default_rng(15)
    N, K = 50, 64
    W = f16(rng.normal(0, 0.02, (N, K)))
    for j in (0, 17, K - 1):
        x = np.zeros(K, dtype=np.float16)
        x[j] = 1.0
        assert np.array_equal(bits(oracle.gemv_f16(x, W)), bits(np.ascontiguousarray(W[:, j])))


def test_gemv_equals_gemm_with_one_row():
    rng = np.random.default_rng(16)
    x = f16(rng.normal(0, 0.02, 200))
    W = f16(rng.normal(0, 0.02, (70, 200)))
    assert np.array_equal(bits(oracle.gemv_f16(x, W)), bits(oracle.gemm_f16(x[None, :], W)[0]))


def test_fp32_accumulation_matters():
    # An fp16 running sum of 4096 ones stalls at 2048 (2048 + 1 rounds back to 2048),
    # and 64 + 0.03 stays 64 in fp16.  The oracle must not accumulate in fp16.
    K = 4096
    x = np.ones(K, dtype=np.float16)
    W = np.ones((2, K), dtype=np.float16)
    assert np.all(oracle.gemv_f16(x, W).astype(np.float64) == 4096.0)
    assert np.float16(np.float16(64.0) + np.float16(0.03)) == np.float16(64.0)


def test_sampled_positions_match_full():
    rng = np.random.default_rng(17)
    A = f16(rng.uniform(-1, 1, (50, 72)))
    B = f16(rng.uniform(-1, 1, (45, 72)))
    D, S = oracle.gemm_f16(A, B, return_sum=True)
    ms = rng.integers(0, 50, 300)
    ns = rng.integers(0, 45, 300)
    d, s = oracle.gemm_f16_at(A, B, ms, ns, return_sum=True)
    assert np.array_equal(bits(d), bits(D[ms, ns]))
    assert np.array_equal(s, S[ms, ns])


def test_fp64_sums_close_to_float64_matmul():
    rng = np.random.default_rng(18)
    A = f16(rng.uniform(-1, 1, (64, 512)))
    B = f16(rng.uniform(-1, 1, (32, 512)))
    _, S = oracle.gemm_f16(A, B, return_sum=True)
    ref = A.astype(np.float64) @ B.astype(np.float64).T
    assert np.allclose(S, ref, rtol=0, atol=1e-12)


def test_threads_do_not_change_results():
    rng = np.random.default_rng(19)
    A = f16(rng.uniform(-1, 1, (40, 256)))
    B = f16(rng.uniform(-1, 1, (33, 256)))
    assert np.array_equal(bits(oracle.gemm_f16(A, B, threads=1)),
                          bits(oracle.gemm_f16(A, B, threads=4)))


# --------------------------------------------------------------------------
# grouped GEMM definition
# --------------------------------------------------------------------------

def test_grouped_integer_exact_per_group():
    rng = np.random.default_rng(30)
    offs = [0, 5, 5, 37, 40]            # includes an empty group
    G, N, K = 4, 24, 64
    Ai = rng.integers(-2, 3, (offs[-1], K))
    Bi = rng.integers(-2, 3, (G, N, K))
    D = oracle.gemm_f16_grouped(f16(Ai), f16(Bi), offs)
    for g in range(G):
        lo, hi = offs[g], offs[g + 1]
        exact = Ai[lo:hi] @ Bi[g].T
        assert np.array_equal(bits(D[lo:hi]), bits(exact.astype(np.float64).astype(np.float16)))


def test_grouped_rows_depend_only_on_their_group():
    rng = np.random.default_rng(31)
    offs = [0, 10, 30]
    A = f16(rng.uniform(-1, 1, (30, 48)))
    B = f16(rng.uniform(-1, 1, (2, 16, 48)))
    D1 = oracle.gemm_f16_grouped(A, B, offs)
    B2 = B.copy()
    B2[1] = f16(rng.uniform(-1, 1, (16, 48)))
    D2 = oracle.gemm_f16_grouped(A, B2, offs)
    assert np.array_equal(bits(D1[:10]), bits(D2[:10]))
    assert not np.array_equal(bits(D1[10:]), bits(D2[10:]))
    assert np.array_equal(bits(oracle.gemm_f16_grouped(A, B[:1], [0, 30])),
                          bits(oracle.gemm_f16(A, B[0])))
