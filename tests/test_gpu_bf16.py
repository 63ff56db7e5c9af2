"""GPU parity of the bf16 GEMM and GEMV (gemm_bf16 / gemv_bf16, through the C
ABI) against the oracle's bf16 definitions.

Tolerance: bf16 keeps 8 significant bits, so one rounding of the result moves
it by up to 2^-8 relative (half a step of 2^-7).  The fp16 rule's relative
term (2e-3) is below that, so the bf16 rule is |err| <= 1e-2 + 8e-3*|ref|
(one bf16 step relative), with the internal gate |err| <= 1 bf16 step of ref
+ 2^-11 as for fp16.  Integer-valued inputs must still match bit for bit."""
import numpy as np
import pytest

import oracle
from tma_pipelined_tensor_tn_gb300 import inputs
from tests.parity_util import compare_bf16

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

@pytest.fixture(scope="module")
def tg():
    import tma_pipelined_tensor_tn_gb300 as m
    m.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return m


def to_bits(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def uniform_bf16(shape, seed):
    g = torch.Generator().manual_seed(seed)
    return (torch.rand(shape, generator=g) * 2 - 1).to(torch.bfloat16)


def run(tg, A, B):
    D = tg.gemm(A.cuda(), B.cuda())
    tg.check()
    return to_bits(D)


@pytest.mark.parametrize("M,N,K", [(256, 256, 256), (4000, 3000, 4160), (4096, 4096, 4096)])
def test_gemm_bf16_parity(tg, M, N, K):
    A, B = uniform_bf16((M, K), M), uniform_bf16((N, K), N + 1)
    compare_bf16(run(tg, A, B), oracle.gemm_bf16(to_bits(A), to_bits(B)), f"bf16 {M}x{N}x{K}")


@pytest.mark.parametrize("bn", [256, 224, 192])
def test_gemm_bf16_each_tile_width(tg, bn):
    M, N, K = 1031, 1000, 1032
    A, B = uniform_bf16((M, K), bn), uniform_bf16((N, K), bn + 1)
    try:
        assert tg.tmagemm_set_tile_n(bn) == tg.TMAGEMM_OK
        D = run(tg, A, B)
    finally:
        tg.tmagemm_set_tile_n(0)
    compare_bf16(D, oracle.gemm_bf16(to_bits(A), to_bits(B)), f"bf16 BN={bn}")


def test_gemm_bf16_integer_bitexact(tg):
    M, N, K = 1000, 1024, 4160
    A = inputs.integer_f16((M, K), seed=70).to(torch.bfloat16)
    B = inputs.integer_f16((N, K), seed=71).to(torch.bfloat16)
    assert np.array_equal(run(tg, A, B), oracle.gemm_bf16(to_bits(A), to_bits(B)))


def test_gemm_bf16_identity(tg):
    K, N = 512, 264
    B = uniform_bf16((N, K), 72)
    I = torch.eye(K, dtype=torch.bfloat16)
    assert np.array_equal(run(tg, I, B), np.ascontiguousarray(to_bits(B).T))


def test_gemv_bf16_parity_and_m1_route(tg):
    N, K = 4096, 14336
    g = torch.Generator().manual_seed(73)
    x = (torch.randn(K, generator=g) * 0.02).to(torch.bfloat16)
    W = (torch.randn((N, K), generator=g) * 0.02).to(torch.bfloat16)
    y = tg.gemv(x.cuda(), W.cuda())
    tg.check()
    ref = oracle.gemv_bf16(to_bits(x), to_bits(W))
    compare_bf16(to_bits(y), ref, "gemv bf16")
    D = run(tg, x.reshape(1, -1), W)
    assert np.array_equal(D[0], to_bits(y))


def test_gemv_bf16_integer_bitexact(tg):
    N, K = 1000, 2056
    x = inputs.integer_f16((K,), seed=74).to(torch.bfloat16)
    W = inputs.integer_f16((N, K), seed=75).to(torch.bfloat16)
    y = tg.gemv(x.cuda(), W.cuda())
    tg.check()
    assert np.array_equal(to_bits(y), oracle.gemv_bf16(to_bits(x), to_bits(W)))


@pytest.mark.parametrize("M", [2, 8, 16, 17, 32, 33, 64])
def test_gemm_bf16_few_rows(tg, M):
    """gemm_bf16 with a few rows: the bf16 register-fragment kernel up to 16
    rows, the tile kernel with its cluster split above; route 3 forces the
    bf16 LSU-fed tcgen05 kernel (checked in test_gemm_bf16_lsu_forced)."""
    N, K = 4104, 4160
    A, B = uniform_bf16((M, K), 700 + M), uniform_bf16((N, K), 701 + M)
    compare_bf16(run(tg, A, B), oracle.gemm_bf16(to_bits(A), to_bits(B)), f"bf16 few rows M={M}")


@pytest.mark.parametrize("M", [8, 24, 64])
def test_gemm_bf16_few_rows_integer_bitexact(tg, M):
    N, K = 2056, 4160
    A = inputs.integer_f16((M, K), seed=710 + M).to(torch.bfloat16)
    B = inputs.integer_f16((N, K), seed=711 + M).to(torch.bfloat16)
    got = run(tg, A, B)
    ref = oracle.gemm_bf16(to_bits(A), to_bits(B))
    assert np.array_equal(np.ascontiguousarray(got).view(np.uint16), ref), f"M={M}"


@pytest.mark.parametrize("M", [2, 17, 40, 64])
def test_gemm_bf16_lsu_forced(tg, M):
    N, K = 1032, 4160
    A, B = uniform_bf16((M, K), 720 + M), uniform_bf16((N, K), 721 + M)
    try:
        assert tg.tmagemm_set_small_m_route(3) == tg.TMAGEMM_OK
        got = run(tg, A, B)
    finally:
        tg.tmagemm_set_small_m_route(0)
    compare_bf16(got, oracle.gemm_bf16(to_bits(A), to_bits(B)), f"bf16 LSU-fed M={M}")


@pytest.mark.parametrize("bn,ck", [(128, 4), (128, 8), (192, 2), (192, 4)])
def test_gemm_bf16_narrow_cluster_split(tg, bn, ck):
    """The bf16 forms of the 128- and 192-wide cluster-split tiles (forced):
    integer inputs bit for bit, uniform inputs within the bf16 rule."""
    M, N, K = 40, 1032, 4160
    Ai = inputs.integer_f16((M, K), seed=730 + bn + ck).to(torch.bfloat16)
    Bi = inputs.integer_f16((N, K), seed=731 + bn + ck).to(torch.bfloat16)
    Au, Bu = uniform_bf16((M, K), 732 + bn + ck), uniform_bf16((N, K), 733 + bn + ck)
    try:
        assert tg.tmagemm_set_tile_n(bn) == tg.TMAGEMM_OK
        assert tg.tmagemm_set_cluster_split(ck) == tg.TMAGEMM_OK
        p = tg.tmagemm_gemm_plan(M, N, K, 0)
        got_i, got_u = run(tg, Ai, Bi), run(tg, Au, Bu)
    finally:
        tg.tmagemm_set_cluster_split(0)
        tg.tmagemm_set_tile_n(0)
    assert (p["BN"], p["cluster_k"]) == (bn, ck), p
    ref_i = oracle.gemm_bf16(to_bits(Ai), to_bits(Bi))
    assert np.array_equal(np.ascontiguousarray(got_i).view(np.uint16), ref_i), (bn, ck)
    compare_bf16(got_u, oracle.gemm_bf16(to_bits(Au), to_bits(Bu)), f"bf16 split {bn}x{ck}")
