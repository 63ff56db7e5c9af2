"""GPU parity of the M=1 GEMV (through the C ABI) against the CPU oracle."""
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


def run_gemv(tg, x, W):
    y = tg.gemv(x.cuda(), W.cuda())
    tg.check()
    return y.cpu().numpy()


@pytest.mark.parametrize("seed", [0, 1])
def test_gemv_parity_llama_down_proj(tg, seed):
    w = inputs.WORKLOADS["gemv_4096x14336"]
    x, W = inputs.gemv_inputs(w["N"], w["K"], seed=seed)
    y = run_gemv(tg, x, W)
    ref = oracle.gemv_f16(x.numpy(), W.numpy())
    stats = compare(y, ref, f"gemv seed {seed}")
    # relative L2 error over the whole vector
    r = ref.astype(np.float64)
    rel = np.linalg.norm(y.astype(np.float64) - r) / np.linalg.norm(r)
    assert rel <= 1e-3, rel
    print("gemv", seed, stats, "relL2", rel)


def test_gemv_integer_bitexact(tg):
    N, K = 4096, 14336
    x = inputs.integer_f16((K,), seed=30)
    W = inputs.integer_f16((N, K), seed=31)
    assert_bitexact(run_gemv(tg, x, W), oracle.gemv_f16(x.numpy(), W.numpy()), "integer gemv")


def test_gemv_unit_vector(tg):
    N, K = 777, 2048
    _, W = inputs.gemv_inputs(N, K, seed=32)
    for j in (0, 5, 1031, K - 1):
        x = torch.zeros(K, dtype=torch.float16)
        x[j] = 1.0
        assert_bitexact(run_gemv(tg, x, W), W[:, j].numpy(), f"e_{j}")


@pytest.mark.parametrize("N,K", [(1, 8), (3, 72), (4097, 256), (100, 264), (513, 1000),
                                 (64, 14344), (5, 2048 * 8 + 8),
                                 # one row per CTA on 152 SMs; more rows per CTA than
                                 # the pieces kernel's table (one warp per row); many
                                 # pieces with a partial last one
                                 (152, 4096), (10000, 1024), (2048, 65536 + 8)])
def test_gemv_edge_shapes(tg, N, K):
    x, W = inputs.gemv_inputs(N, K, seed=N * 7 + K)
    compare(run_gemv(tg, x, W), oracle.gemv_f16(x.numpy(), W.numpy()), f"gemv {N}x{K}")


def test_gemv_pieces_table_limits(tg):
    # The pieces kernel holds up to 64 rows per CTA (one CTA per SM) and 64
    # slots per row (pieces of 224 16-byte chunks and a shorter last part):
    # exactly at each limit, and one past it (where the one-warp-per-row
    # kernel takes over).
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    for N, K in [(64 * sms, 1024), (64 * sms + 1, 1024), (256, 64 * 224 * 8),
                 (256, 63 * 224 * 8 + 8), (256, 64 * 224 * 8 + 8)]:
        x, W = inputs.gemv_inputs(N, K, seed=N + K)
        compare(run_gemv(tg, x, W), oracle.gemv_f16(x.numpy(), W.numpy()), f"gemv {N}x{K}")


def test_gemv_partial_piece_integer_bitexact(tg):
    # Rows of 375 16-byte chunks: one whole piece and a partial one per row.
    N, K = 1000, 3000
    x = inputs.integer_f16((K,), seed=32)
    W = inputs.integer_f16((N, K), seed=33)
    assert_bitexact(run_gemv(tg, x, W), oracle.gemv_f16(x.numpy(), W.numpy()),
                    "integer gemv, partial piece")


def test_gemv_fp32_accumulation(tg):
    # 14336 ones: an fp16 running sum would stall at 2048.
    K = 14336
    x = torch.ones(K, dtype=torch.float16)
    W = torch.ones((8, K), dtype=torch.float16)
    y = run_gemv(tg, x, W)
    assert np.all(y.astype(np.float64) == oracle.gemv_f16(x.numpy(), W.numpy()).astype(np.float64))
    assert np.all(y.astype(np.float64) == 14336.0)
