"""Programmatic dependent launch: kernels queued back to back on one stream,
where each reads what the one before it wrote (read after write) or
overwrites what the one before it read (write after read), give the oracle's
results with the attribute on and off.  Every library kernel executes
griddepcontrol.wait before it touches an argument buffer, so an early-
scheduled kernel never sees a half-written input."""
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


@pytest.fixture(params=[1, 0], ids=["pdl", "plain"])
def pdl(tg, request):
    assert tg.tmagemm_set_pdl(request.param) == tg.TMAGEMM_OK
    yield request.param
    assert tg.tmagemm_set_pdl(1) == tg.TMAGEMM_OK


def _small_ints(shape, seed, lo=-2, hi=3):
    g = np.random.default_rng(seed)
    return g.integers(lo, hi, size=shape).astype(np.float16)


def test_gemm_chain_read_after_write(tg, pdl):
    """D1 = A B^T, then D2 = D1 C^T on the same stream, no sync between.
    Small integers keep every value exact, so the chain is bit-exact."""
    M, N1, K, N2 = 1000, 512, 768, 264
    A, B, C = _small_ints((M, K), 1), _small_ints((N1, K), 2), _small_ints((N2, N1), 3, -1, 2)
    ref1 = oracle.gemm_f16(A, B)
    ref2 = oracle.gemm_f16(ref1, C)
    assert np.all(np.isfinite(ref2.astype(np.float64)))
    a, b, c = (torch.from_numpy(t).cuda() for t in (A, B, C))
    for _ in range(3):
        d1 = tg.gemm(a, b)
        d2 = tg.gemm(d1, c)
        d3 = tg.gemm(d2, torch.eye(N2, dtype=torch.float16, device="cuda"))
    torch.cuda.synchronize()
    tg.check()
    assert_bitexact(d1.cpu().numpy(), ref1, "first GEMM")
    assert_bitexact(d2.cpu().numpy(), ref2, "second GEMM (reads the first's output)")
    assert_bitexact(d3.cpu().numpy(), ref2, "identity GEMM on the second's output")


def test_gemm_write_after_read(tg, pdl):
    """The second GEMM writes into the buffer the first one reads (A)."""
    M, N, K = 512, 512, 512
    A, B = _small_ints((M, K), 4), _small_ints((N, K), 5)
    ref1 = oracle.gemm_f16(A, B)
    a, b = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    d = torch.empty((M, N), dtype=torch.float16, device="cuda")
    ones = torch.ones((K, K), dtype=torch.float16, device="cuda")
    tg.gemm(a, b, out=d)
    tg.gemm(torch.zeros((M, K), dtype=torch.float16, device="cuda"), ones, out=a)   # a := 0
    torch.cuda.synchronize()
    tg.check()
    assert_bitexact(d.cpu().numpy(), ref1, "GEMM whose input is overwritten next")
    assert not a.any()


def test_gemv_chain(tg, pdl):
    """y1 = W1 x, y2 = W2 y1, then a split-K GEMM and a small-M GEMM on y2."""
    K = 4096
    x, W1 = inputs.gemv_inputs(K, K, seed=31)
    _, W2 = inputs.gemv_inputs(K, K, seed=32)
    y1_ref = oracle.gemv_f16(x.numpy(), W1.numpy())
    y2_ref = oracle.gemv_f16(y1_ref, W2.numpy())
    xd, w1, w2 = x.cuda(), W1.cuda(), W2.cuda()
    y1 = tg.gemv(xd, w1)
    y2 = tg.gemv(y1, w2)
    X = y2.reshape(1, K).repeat(8, 1)
    need = tg.gemm_f16_small_m_workspace_size(8, K, K)
    ws = torch.empty((max(need, 1),), dtype=torch.uint8, device="cuda")
    d_small = tg.gemm_small_m(X, w1, workspace=ws)
    torch.cuda.synchronize()
    tg.check()
    compare(y1.cpu().numpy(), y1_ref, "gemv 1")
    # y2 from the device's y1 (equal to the oracle's within tolerance): compare
    # against the oracle applied to the device's own y1, element for element.
    y2_dev_ref = oracle.gemv_f16(y1.cpu().numpy(), W2.numpy())
    compare(y2.cpu().numpy(), y2_dev_ref, "gemv 2 (input: gemv 1's output)")
    ref_small = oracle.gemm_f16(X.cpu().numpy(), W1.numpy())
    compare(d_small.cpu().numpy(), ref_small, "small-M GEMM after the GEMVs")


def test_splitk_chain(tg, pdl):
    """Split-K (GEMM + reduction kernel) twice in a row into the same output."""
    M, N, K = 256, 512, 8192
    A, B = inputs.gemm_inputs(M, N, K, seed=33)
    ref = oracle.gemm_f16(A.numpy(), B.numpy())
    a, b = A.cuda(), B.cuda()
    need = tg.gemm_f16_splitk_workspace_size(M, N, K, 4)
    ws = torch.empty((need,), dtype=torch.uint8, device="cuda")
    d = torch.empty((M, N), dtype=torch.float16, device="cuda")
    for _ in range(3):
        tg.gemm_splitk(a, b, workspace=ws, splits=4, out=d)
    torch.cuda.synchronize()
    tg.check()
    compare(d.cpu().numpy(), ref, "split-K, third of three back-to-back calls")
