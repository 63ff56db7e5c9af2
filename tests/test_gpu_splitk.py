"""GPU parity of the split-K GEMM (gemm_f16_splitk, through the C ABI) against
the same oracle definition as the plain GEMM: splitting K changes only the
schedule, D = fp16(A @ B.T) is unchanged."""
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


def run_splitk(tg, A, B, splits, ws=None):
    D = tg.gemm_splitk(A.cuda(), B.cuda(), workspace=ws, splits=splits)
    tg.check()
    return D.cpu().numpy()


@pytest.mark.parametrize("M,N,K,splits", [
    (1024, 1024, 16384, 0),     # automatic: 32 tiles -> 4 parts
    (1000, 1000, 4160, 3),      # ragged M, N; 65 k-blocks in parts of 22
    (256, 256, 256, 4),         # one k-block per part
    (129, 264, 1000, 5),        # 16 k-blocks: 5 requested, 4 non-empty parts of 4
    (4000, 3000, 4160, 2),      # the ragged workload in two parts
    (300, 520, 8, 3),           # one k-block in total: clamped to no split
])
def test_splitk_parity(tg, M, N, K, splits):
    A, B = inputs.gemm_inputs(M, N, K, seed=M + K)
    compare(run_splitk(tg, A, B, splits), oracle.gemm_f16(A.numpy(), B.numpy()),
            f"split-K {M}x{N}x{K} s={splits}", k=A.shape[1])


def test_splitk_integer_bitexact(tg):
    M, N, K = 777, 1000, 4160
    A = inputs.integer_f16((M, K), seed=40)
    B = inputs.integer_f16((N, K), seed=41)
    assert_bitexact(run_splitk(tg, A, B, 4), oracle.gemm_f16(A.numpy(), B.numpy()), "split-K int")


@pytest.mark.parametrize("bn", [256, 224, 192])
def test_splitk_each_tile_width(tg, bn):
    M, N, K = 520, 1000, 2056
    A, B = inputs.gemm_inputs(M, N, K, seed=bn + 7)
    try:
        assert tg.tmagemm_set_tile_n(bn) == tg.TMAGEMM_OK
        D = run_splitk(tg, A, B, 3)
    finally:
        tg.tmagemm_set_tile_n(0)
    compare(D, oracle.gemm_f16(A.numpy(), B.numpy()), f"split-K BN={bn}", k=A.shape[1])


def test_splitk_deterministic_and_one_part_equals_plain(tg):
    M, N, K = 640, 768, 8192
    A, B = inputs.gemm_inputs(M, N, K, seed=50)
    d1 = run_splitk(tg, A, B, 6)
    d2 = run_splitk(tg, A, B, 6)
    assert_bitexact(d1, d2, "split-K repeat")
    plain = tg.gemm(A.cuda(), B.cuda())
    tg.check()
    assert_bitexact(run_splitk(tg, A, B, 1), plain.cpu().numpy(), "splits=1 is the plain GEMM")
    compare(d1, oracle.gemm_f16(A.numpy(), B.numpy()), "split-K 6 parts", k=A.shape[1])


def test_splitk_workspace_rules(tg):
    M, N, K = 512, 512, 8192
    need = tg.gemm_f16_splitk_workspace_size(M, N, K, 4)
    assert need == 4 * M * N * 4
    A = torch.zeros((M, K), dtype=torch.float16, device="cuda")
    B = torch.zeros((N, K), dtype=torch.float16, device="cuda")
    D = torch.empty((M, N), dtype=torch.float16, device="cuda")
    ws = torch.empty((need + 64,), dtype=torch.uint8, device="cuda")
    a, b, d, w = A.data_ptr(), B.data_ptr(), D.data_ptr(), ws.data_ptr()
    assert tg.gemm_f16_splitk(M, N, K, a, b, d, 4, None, 0, None) == tg.TMAGEMM_ERR_WORKSPACE
    assert tg.gemm_f16_splitk(M, N, K, a, b, d, 4, w, need - 16, None) == tg.TMAGEMM_ERR_WORKSPACE
    assert tg.gemm_f16_splitk(M, N, K, a, b, d, 4, w + 8, need, None) == tg.TMAGEMM_ERR_WORKSPACE
    assert tg.gemm_f16_splitk(M, N, K, a, b, d, 4, w, need, None) == tg.TMAGEMM_OK
    # a plan without a split needs no workspace at all
    assert tg.gemm_f16_splitk_workspace_size(4096, 4096, 4096, 0) == 0
    assert tg.gemm_f16_splitk(M, N, 64, a, b, d, 0, None, 0, None) == tg.TMAGEMM_OK
    tg.check()
    assert torch.count_nonzero(D).item() == 0
