"""GPU parity of gemm_f16's cluster split-K (few output tiles, long K): the
CTAs of a 2-, 4- or 8-CTA cluster compute one tile over separate K ranges and
add their FP32 accumulators through distributed shared memory before writing
D.  Splitting K changes only the schedule; D = fp16(A @ B.T) as for the plain
GEMM (same oracle)."""
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


def sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


def gemm_with(tg, A, B, mode):
    try:
        assert tg.tmagemm_set_cluster_split(mode) == tg.TMAGEMM_OK
        D = tg.gemm(A.cuda(), B.cuda())
        tg.check()
    finally:
        tg.tmagemm_set_cluster_split(0)
    return D.cpu().numpy()


def test_auto_plan_uses_cluster_split(tg):
    p = tg.tmagemm_gemm_plan(1024, 1024, 16384, sms(), 1, sms() // 2)
    assert p["cluster_k"] in (2, 4, 8) and p["splits"] == p["cluster_k"]


def test_auto_parity_1024x1024x16384(tg):
    M, N, K = 1024, 1024, 16384
    A, B = inputs.gemm_inputs(M, N, K, seed=600)
    compare(gemm_with(tg, A, B, 0), oracle.gemm_f16(A.numpy(), B.numpy()), "cluster split auto", k=A.shape[1])


@pytest.fixture(params=[0, 1], ids=["pairs_allowed", "single_ctas"])
def pair_mode(tg, request):
    """0: the plan may use CTA pairs inside the split clusters; 1: single CTAs."""
    assert tg.tmagemm_set_cta_pair(request.param) == tg.TMAGEMM_OK
    yield request.param
    assert tg.tmagemm_set_cta_pair(0) == tg.TMAGEMM_OK


# Ragged M and N (partial last tiles), K not a multiple of the slice.
@pytest.mark.parametrize("ck", [2, 4, 8])
@pytest.mark.parametrize("M,N,K", [(512, 1000, 4160), (300, 776, 8200), (128, 256, 1024)])
def test_forced_sizes_parity(tg, pair_mode, ck, M, N, K):
    p = None
    try:
        tg.tmagemm_set_cluster_split(ck)
        p = tg.tmagemm_gemm_plan(M, N, K, sms(), 1, 0 if pair_mode == 1 else sms() // 2)
    finally:
        tg.tmagemm_set_cluster_split(0)
    if ck == 8 and pair_mode == 0:
        assert p["cluster_k"] in (0, 8) and not (p["cluster_k"] == 8 and p["pair"]), p
    else:
        assert p["cluster_k"] == ck, p
    A, B = inputs.gemm_inputs(M, N, K, seed=M + N + ck)
    compare(gemm_with(tg, A, B, ck), oracle.gemm_f16(A.numpy(), B.numpy()),
            f"cluster split {ck} {M}x{N}x{K} pair mode {pair_mode}", k=A.shape[1])


@pytest.mark.parametrize("ck", [2, 4, 8])
def test_integer_bitexact_and_deterministic(tg, pair_mode, ck):
    M, N, K = 512, 1000, 4160
    A = inputs.integer_f16((M, K), seed=60)
    B = inputs.integer_f16((N, K), seed=61)
    d1 = gemm_with(tg, A, B, ck)
    assert_bitexact(d1, oracle.gemm_f16(A.numpy(), B.numpy()), f"cluster split {ck} integer")
    assert_bitexact(gemm_with(tg, A, B, ck), d1, "repeat")


def test_agrees_with_workspace_split_and_plain(tg):
    M, N, K = 1024, 1024, 16384
    A = inputs.integer_f16((M, K), seed=62)
    B = inputs.integer_f16((N, K), seed=63)
    ck = gemm_with(tg, A, B, 0)
    plain = gemm_with(tg, A, B, 1)
    ws = tg.gemm_splitk(A.cuda(), B.cuda(), splits=4).cpu().numpy()
    tg.check()
    assert_bitexact(ck, plain, "cluster split vs plain (exact integer sums)")
    assert_bitexact(ck, ws, "cluster split vs workspace split-K")


def test_output_guard(tg):
    """D inside a larger buffer: the direct stores of the cluster epilogue
    stay inside D and cover all of it."""
    M, N, K = 300, 776, 8200
    A, B = inputs.gemm_inputs(M, N, K, seed=64)
    guard = 4096
    sentinel = np.uint16(0x7E01)
    buf = torch.full((guard + M * N + guard,), int(sentinel.view(np.int16)), dtype=torch.int16)
    dbuf = buf.cuda()
    D = dbuf[guard:guard + M * N].view(torch.float16).view(M, N)
    try:
        assert tg.tmagemm_set_cluster_split(4) == tg.TMAGEMM_OK
        tg.gemm(A.cuda(), B.cuda(), out=D)
        tg.check()
    finally:
        tg.tmagemm_set_cluster_split(0)
    host = dbuf.cpu().numpy().view(np.uint16)
    assert np.all(host[:guard] == sentinel) and np.all(host[guard + M * N:] == sentinel)
    body = host[guard:guard + M * N]
    assert not np.any(body == sentinel)
    compare(body.view(np.float16).reshape(M, N), oracle.gemm_f16(A.numpy(), B.numpy()), "guarded", k=A.shape[1])


def forced_plan_and_gemm(tg, A, B, bn, ck):
    """gemm_f16 with the tile width and the cluster split forced; returns the
    device plan it ran and D."""
    M, K = A.shape
    N = B.shape[0]
    try:
        assert tg.tmagemm_set_tile_n(bn) == tg.TMAGEMM_OK
        assert tg.tmagemm_set_cluster_split(ck) == tg.TMAGEMM_OK
        p = tg.tmagemm_gemm_plan(M, N, K, 0)
        D = tg.gemm(A.cuda(), B.cuda())
        tg.check()
    finally:
        tg.tmagemm_set_cluster_split(0)
        tg.tmagemm_set_tile_n(0)
    return p, D.cpu().numpy()


# The narrower cluster-split tiles (128 x 128 and 128 x 192) that a few rows
# against a wide weight matrix get.  Shapes: ragged N (partial last tile), a
# row count that is not a multiple of anything (two tile rows at M = 130), K
# with an odd number of k-blocks or shorter than two k-blocks per CTA.
@pytest.mark.parametrize("bn,ck", [(128, 4), (128, 8), (192, 2), (192, 4)])
@pytest.mark.parametrize("M,N,K", [(40, 1032, 4160), (130, 776, 8200), (17, 1672, 1000)])
def test_narrow_tiles_parity(tg, bn, ck, M, N, K):
    A, B = inputs.gemm_inputs(M, N, K, seed=M + N + bn + ck)
    p, D = forced_plan_and_gemm(tg, A, B, bn, ck)
    assert (p["BN"], p["cluster_k"], p["pair"]) == (bn, ck, 0), p
    compare(D, oracle.gemm_f16(A.numpy(), B.numpy()), f"cluster split {bn}x{ck} {M}x{N}x{K}", k=A.shape[1])


@pytest.mark.parametrize("bn,ck", [(128, 4), (128, 8), (192, 2), (192, 4)])
def test_narrow_tiles_integer_bitexact(tg, bn, ck):
    M, N, K = 64, 1032, 4160
    A = inputs.integer_f16((M, K), seed=65)
    B = inputs.integer_f16((N, K), seed=66)
    p, D = forced_plan_and_gemm(tg, A, B, bn, ck)
    assert (p["BN"], p["cluster_k"]) == (bn, ck), p
    assert_bitexact(D, oracle.gemm_f16(A.numpy(), B.numpy()), f"cluster split {bn}x{ck} integer")


@pytest.mark.parametrize("M,N,K", [(32, 4096, 14336), (64, 14336, 4096)])
def test_decode_shapes_fill_the_sms(tg, M, N, K):
    """The automatic plan for a few tokens against a Llama-3-8B-sized weight
    splits K over clusters and keeps at least 80 % of the SMs streaming the
    weights; D matches the oracle on sampled rows."""
    p = tg.tmagemm_gemm_plan(M, N, K, 0)
    assert p["cluster_k"] in (2, 4, 8) and p["grid"] >= 0.8 * sms(), p
    g = torch.Generator().manual_seed(M + N)
    X = (torch.randn((M, K), generator=g) * 0.02).half()
    W = (torch.randn((N, K), generator=g) * 0.02).half()
    D = tg.gemm(X.cuda(), W.cuda()).cpu().numpy()
    tg.check()
    rows = np.arange(0, N, 97)
    compare(D[:, rows], oracle.gemm_f16(X.numpy(), W.numpy()[rows]), f"decode {M}x{N}x{K}", k=X.shape[1])


@pytest.mark.parametrize("M,N,K", [(17, 4096, 14336), (64, 4096, 14336), (40, 1000, 4160),
                                   (2, 520, 1032), (64, 4104, 200)])
def test_decode_cluster_split(tg, M, N, K):
    """The decode split (at most 64 rows; a stage holds a 64-row A box, so the
    128-row MMA's rows past it read the stage's own B box and reach only
    unstored accumulator rows; 9 stages): 4-CTA clusters of 128-wide tiles,
    forced per call, ragged N and K included.  The oracle's result; integer
    inputs bit-exact."""
    # small_m_route = 1 keeps every M on the tile kernel in gemm_f16_ex
    opts = tg.options(cluster_split=4, tile_n=128, small_m_route=1)
    A, B = inputs.gemm_inputs(M, N, K, seed=700 + M)
    D = tg.gemm(A.cuda(), B.cuda(), opts=opts)
    tg.check()
    compare(D.cpu().numpy(), oracle.gemm_f16(A.numpy(), B.numpy()), f"decode {M}x{N}x{K}", k=K)
    Ai = inputs.integer_f16((M, K), seed=M)
    Bi = inputs.integer_f16((N, K), seed=N)
    Di = tg.gemm(Ai.cuda(), Bi.cuda(), opts=opts)
    tg.check()
    assert_bitexact(Di.cpu().numpy(), oracle.gemm_f16(Ai.numpy(), Bi.numpy()), f"decode {M} int")
