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
    compare(gemm_with(tg, A, B, 0), oracle.gemm_f16(A.numpy(), B.numpy()), "cluster split auto")


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
            f"cluster split {ck} {M}x{N}x{K} pair mode {pair_mode}")


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
    compare(body.view(np.float16).reshape(M, N), oracle.gemm_f16(A.numpy(), B.numpy()), "guarded")
