"""The split-K entry point for callers that cannot allocate device memory.

gemm_f16_splitk_noalloc runs split-K with the library's own fixed 32 MiB
device array as workspace, for callers that cannot hand the library a buffer
(no cudaMalloc allowed past their start-up, or all device memory owned by a
host framework's pool).  This checks it through the C ABI against the CPU
oracle and against the existing entry point (gemm_f16_splitk with a caller
workspace) on two calls in a row, that repeated calls leave the device's free
memory unchanged, and that oversized problems are refused.  The file is
collected last on purpose and also passes on its own in a fresh process.
"""
import pytest

import oracle
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
        tg.check()
        got = D.cpu().numpy()
        compare(got, oracle.gemm_f16(A.numpy(), B.numpy()), f"no-alloc split-K {M}x{N}x{K} vs oracle")
        ref = with_caller_workspace(tg, dA, dB, splits)
        tg.check()
        compare(got, ref.cpu().numpy(), f"no-alloc split-K {M}x{N}x{K}")


def test_noalloc_calls_leave_free_device_memory_unchanged(tg):
    # After one call per shape (the first call on the device looks up the
    # array's address and may load kernels), further calls must not change the
    # device's free memory: nothing is allocated per call.
    cases = []
    for (M, N, K, splits, seed) in ((512, 768, 8192, 0, 62), (1000, 520, 4160, 4, 63)):
        A, B = inputs.gemm_inputs(M, N, K, seed=seed)
        D = torch.empty((M, N), dtype=torch.float16, device="cuda")
        cases.append((A.cuda(), B.cuda(), splits, D))
    for dA, dB, splits, D in cases:
        assert without_allocation(tg, dA, dB, splits, D) == tg.TMAGEMM_OK
    tg.check()
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        for dA, dB, splits, D in cases:
            assert without_allocation(tg, dA, dB, splits, D) == tg.TMAGEMM_OK
    tg.check()
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0, f"free device memory changed by {free0 - free1} bytes"


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
