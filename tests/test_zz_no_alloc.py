"""The split-K entry point for callers that cannot allocate device memory.

gemm_f16_splitk_noalloc runs split-K with the library's own fixed 32 MiB
device array as workspace, for callers that cannot hand the library a buffer
(no cudaMalloc allowed past their start-up, or all device memory owned by a
host framework's pool).  This checks it through the C ABI against the
existing entry point (gemm_f16_splitk with a caller workspace) on two calls in
a row, and that oversized problems are refused.  The file is collected last
on purpose and also passes on its own in a fresh process.
"""
import pytest

from tma_pipelined_tensor_tn_gb300 import inputs
from tests.parity_util import compare

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 32 << 20


@pytest.fixture(scope="module")
def tg():
    import tma_pipelined_tensor_tn_gb300 as m
    m.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return m


def with_caller_workspace(tg, A, B, splits):
    M, K = A.shape
    N = B.shape[0]
    need = tg.gemm_f16_splitk_workspace_size(M, N, K, splits)
    assert need >= 0
    ws = torch.empty((max(need, 16),), dtype=torch.uint8, device="cuda")
    D = torch.empty((M, N), dtype=torch.float16, device="cuda")
    s = tg.gemm_f16_splitk(M, N, K, A.data_ptr(), B.data_ptr(), D.data_ptr(), splits,
                           ws.data_ptr(), ws.numel(), None)
    assert s == tg.TMAGEMM_OK, tg.strerror(s)
    return D


def without_allocation(tg, A, B, splits, D):
    M, K = A.shape
    N = B.shape[0]
    return tg.gemm_f16_splitk_noalloc(M, N, K, A.data_ptr(), B.data_ptr(), D.data_ptr(), splits,
                                      None)


def test_noalloc_matches_caller_workspace_on_two_calls(tg):
    # Two calls in a row with different shapes and inputs: the second must not
    # depend on what the first left in the shared scratch.
    for (M, N, K, splits, seed) in ((1024, 1024, 16384, 0, 60), (777, 1000, 4160, 3, 61)):
        A, B = inputs.gemm_inputs(M, N, K, seed=seed)
        dA, dB = A.cuda(), B.cuda()
        assert tg.gemm_f16_splitk_workspace_size(M, N, K, splits) <= SCRATCH_BYTES
        D = torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda")
        assert without_allocation(tg, dA, dB, splits, D) == tg.TMAGEMM_OK
        ref = with_caller_workspace(tg, dA, dB, splits)
        tg.check()
        compare(D.cpu().numpy(), ref.cpu().numpy(), f"no-alloc split-K {M}x{N}x{K}")


def test_noalloc_refuses_problems_beyond_its_scratch(tg):
    M, N, K = 2048, 2048, 65536
    need = tg.gemm_f16_splitk_workspace_size(M, N, K, 4)
    assert need > SCRATCH_BYTES
    A = torch.zeros((M, K), dtype=torch.float16, device="cuda")
    B = torch.zeros((N, K), dtype=torch.float16, device="cuda")
    D = torch.zeros((M, N), dtype=torch.float16, device="cuda")
    assert without_allocation(tg, A, B, 4, D) == tg.TMAGEMM_ERR_SCRATCH_LIMIT
    assert "32 MiB" in tg.strerror(tg.TMAGEMM_ERR_SCRATCH_LIMIT)
    tg.check()
