"""GPU parity of the skinny (2 <= M <= 64) GEMM, gemm_f16_small_m, through the
C ABI against the oracle's GEMM definition (D = fp16(X @ W.T)); the operand
swap and the K split change only the schedule."""
import numpy as np
import pytest

import oracle
from tma_pipelined_tensor_tn_gb300 import inputs
from tests.parity_util import assert_bitexact, compare

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tg():
    import tma_pipelined_tensor_tn_gb300 as m
    m.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return m


def run(tg, X, W):
    D = tg.gemm_small_m(X.cuda(), W.cuda())
    tg.check()
    return D.cpu().numpy()


# 1 = the tcgen05 swap-AB kernel, 2 = automatic (the register-fragment
# mma.sync kernel up to 16 rows, the tile kernel above), 3 = the LSU-fed
# tcgen05 kernel (every M).
@pytest.fixture(params=[1, 2, 3], ids=["swap_ab", "auto", "lsu"])
def route(tg, request):
    assert tg.tmagemm_set_small_m_route(request.param) == tg.TMAGEMM_OK
    yield request.param
    assert tg.tmagemm_set_small_m_route(0) == tg.TMAGEMM_OK


def decode_inputs(M, N, K, seed):
    g = torch.Generator().manual_seed(seed)
    X = (torch.randn((M, K), generator=g) * 0.02).half()
    W = (torch.randn((N, K), generator=g) * 0.02).half()
    return X, W


@pytest.mark.parametrize("M", [2, 3, 8, 16, 17, 32])
def test_small_m_parity_down_projection(tg, route, M):
    N, K = 4096, 14336
    X, W = decode_inputs(M, N, K, seed=M)
    compare(run(tg, X, W), oracle.gemm_f16(X.numpy(), W.numpy()), f"small-M M={M} route {route}", k=X.shape[1])


@pytest.mark.parametrize("M", [33, 64])
def test_small_m_parity_down_projection_wide(tg, route, M):
    N, K = 4096, 14336
    X, W = decode_inputs(M, N, K, seed=M)
    compare(run(tg, X, W), oracle.gemm_f16(X.numpy(), W.numpy()), f"small-M M={M} route {route}", k=X.shape[1])


# Ragged N (not a multiple of the 64 weight rows of a cluster), K shorter than
# the 8 slices, K not a multiple of the 32-k step, one row, one 16-byte chunk.
@pytest.mark.parametrize("M,N,K", [(5, 1000, 4160), (16, 136, 72), (2, 8, 1000), (9, 72, 8),
                                   (31, 520, 264), (4, 4104, 14344)])
def test_small_m_edge_shapes(tg, route, M, N, K):
    X, W = inputs.gemm_inputs(M, N, K, seed=M + N)
    compare(run(tg, X, W), oracle.gemm_f16(X.numpy(), W.numpy()),
            f"small-M {M}x{N}x{K} route {route}", k=X.shape[1])


@pytest.mark.parametrize("M,N,K", [(40, 264, 8), (64, 1000, 4160), (47, 136, 72), (33, 4104, 1000)])
def test_small_m_edge_shape_wide(tg, route, M, N, K):
    X, W = inputs.gemm_inputs(M, N, K, seed=M + N + K)
    compare(run(tg, X, W), oracle.gemm_f16(X.numpy(), W.numpy()), f"small-M {M}x{N}x{K} route {route}", k=X.shape[1])


@pytest.mark.parametrize("M", [12, 32, 64])
def test_small_m_integer_bitexact_and_deterministic(tg, route, M):
    N, K = 2056, 4160
    X = inputs.integer_f16((M, K), seed=80)
    W = inputs.integer_f16((N, K), seed=81)
    d1 = run(tg, X, W)
    assert_bitexact(d1, oracle.gemm_f16(X.numpy(), W.numpy()), f"small-M integer route {route}")
    assert_bitexact(run(tg, X, W), d1, "repeat")


def test_small_m_routes_agree_on_exact_sums(tg):
    """Integer inputs make every FP32 partial exact, so the two kernels must
    give the same bits although they add in different orders."""
    M, N, K = 16, 4096, 14336
    X = inputs.integer_f16((M, K), seed=82)
    W = inputs.integer_f16((N, K), seed=83)
    out = {}
    try:
        for r in (1, 2, 3):
            assert tg.tmagemm_set_small_m_route(r) == tg.TMAGEMM_OK
            out[r] = run(tg, X, W)
    finally:
        tg.tmagemm_set_small_m_route(0)
    assert_bitexact(out[2], out[1], "fragments vs tcgen05")
    assert_bitexact(out[3], out[1], "LSU-fed vs tcgen05")


@pytest.mark.parametrize("M", [2, 16, 17, 32, 33, 64])
def test_small_m_auto_route(tg, M):
    """The automatic route on each side of its threshold (16): no workspace,
    and the same bits as gemm_f16 (which routes the same way)."""
    N, K = 1032, 2056
    X, W = inputs.gemm_inputs(M, N, K, seed=400 + M)
    d = run(tg, X, W)
    compare(d, oracle.gemm_f16(X.numpy(), W.numpy()), f"small-M auto M={M}", k=X.shape[1])
    assert tg.gemm_f16_small_m_workspace_size(M, N, K) == 0
    assert_bitexact(d, tg.gemm(X.cuda(), W.cuda()).cpu().numpy(), f"small-M auto vs gemm_f16 M={M}")


def test_small_m_rejects_out_of_range_and_bad_workspace(tg):
    p = torch.zeros(1 << 20, dtype=torch.float16, device="cuda").data_ptr()
    assert tg.gemm_f16_small_m(1, 64, 64, p, p, p, p, 1 << 20, None) == tg.TMAGEMM_ERR_UNSUPPORTED
    assert tg.gemm_f16_small_m(65, 64, 64, p, p, p, p, 1 << 20, None) == tg.TMAGEMM_ERR_UNSUPPORTED
    # The automatic choices need no workspace.
    for M in (8, 40):
        assert tg.gemm_f16_small_m_workspace_size(M, 4096, 14336) == 0
        assert tg.gemm_f16_small_m(M, 64, 64, p, p, p, None, 0, None) == tg.TMAGEMM_OK
    # The swap-AB kernel (route 1) does.
    try:
        assert tg.tmagemm_set_small_m_route(1) == tg.TMAGEMM_OK
        assert tg.gemm_f16_small_m(40, 64, 64, p, p, p, None, 0, None) == tg.TMAGEMM_ERR_WORKSPACE
        need = tg.gemm_f16_small_m_workspace_size(40, 4096, 14336)
        assert need > 0
        assert tg.gemm_f16_small_m(40, 4096, 14336, p, p, p, p, need - 16, None) == \
            tg.TMAGEMM_ERR_WORKSPACE
        assert tg.gemm_f16_small_m_workspace_size(8, 4096, 14336) > 0
        assert tg.gemm_f16_small_m(8, 64, 64, p, p, p, None, 0, None) == tg.TMAGEMM_ERR_WORKSPACE
    finally:
        assert tg.tmagemm_set_small_m_route(0) == tg.TMAGEMM_OK
    torch.cuda.synchronize()


@pytest.mark.parametrize("M", [8, 16])
def test_fragments_wide_n_without_k_split(tg, M):
    """N = 28672: 448 groups of 64 weight rows; even two K slices per group
    would not fit in one wave of CTAs, so each CTA takes its 64 rows over the
    whole K (clusters of one CTA).  Parity, and integer inputs bit for bit."""
    N, K = 28672, 1032
    X, W = decode_inputs(M, N, K, seed=500 + M)
    compare(run(tg, X, W), oracle.gemm_f16(X.numpy(), W.numpy()), f"wide N M={M}", k=X.shape[1])
    Xi = inputs.integer_f16((M, K), seed=502 + M)
    Wi = inputs.integer_f16((N, K), seed=503 + M)
    assert_bitexact(run(tg, Xi, Wi), oracle.gemm_f16(Xi.numpy(), Wi.numpy()), f"wide N integer M={M}")
