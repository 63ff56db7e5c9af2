"""The host-buffer executor (HostGemmPipeline, the end-to-end path the bench
times): every step's D, copied back to host memory, matches the CPU oracle on
that step's inputs, and overlapping the copies of neighbouring steps changes no
step's result (each equals the direct device call bit for bit)."""
import numpy as np
import pytest

import oracle
from tma_pipelined_tensor_tn_gb300 import inputs
from tests.parity_util import assert_bitexact, compare, compare_bf16

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tg():
    import tma_pipelined_tensor_tn_gb300 as m
    m.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return m


@pytest.mark.parametrize("depth", [1, 2, 3])
def test_pipeline_matches_direct_calls(tg, depth):
    from tma_pipelined_tensor_tn_gb300.pipeline import HostGemmPipeline
    M, N, K, steps = 640, 520, 1032, 7
    As, Bs = [], []
    for i in range(steps):
        a, b = inputs.gemm_inputs(M, N, K, seed=100 + i)
        As.append(a.pin_memory())
        Bs.append(b.pin_memory())
    Ds = [torch.empty((M, N), dtype=torch.float16).pin_memory() for _ in range(steps)]
    pipe = HostGemmPipeline(M, N, K, depth=depth)
    pipe.run(As, Bs, Ds)
    pipe.synchronize()
    tg.check()
    for i in range(steps):
        compare(Ds[i].numpy(), oracle.gemm_f16(As[i].numpy(), Bs[i].numpy()),
                f"pipeline step {i} vs oracle")
        ref = tg.gemm(As[i].cuda(), Bs[i].cuda())
        tg.check()
        assert_bitexact(Ds[i].numpy(), ref.cpu().numpy(), f"step {i}")
    assert pipe.h2d_bytes_per_step() == 2 * (M * K + N * K)
    assert pipe.d2h_bytes_per_step() == 2 * M * N


def test_pipeline_bf16_pageable_and_two_runs(tg):
    """bf16 steps from pageable host memory, enqueued by two run() calls
    before one synchronize: every step equals the direct call."""
    from tma_pipelined_tensor_tn_gb300.pipeline import HostGemmPipeline
    M, N, K = 256, 264, 520
    g = torch.Generator().manual_seed(130)
    As = [(torch.rand((M, K), generator=g) * 2 - 1).to(torch.bfloat16) for _ in range(5)]
    Bs = [(torch.rand((N, K), generator=g) * 2 - 1).to(torch.bfloat16) for _ in range(5)]
    Ds = [torch.empty((M, N), dtype=torch.bfloat16) for _ in range(5)]
    pipe = HostGemmPipeline(M, N, K, dtype=torch.bfloat16, depth=2)
    pipe.run(As[:2], Bs[:2], Ds[:2])
    pipe.run(As[2:], Bs[2:], Ds[2:])
    pipe.run([], [], [])
    pipe.synchronize()
    for i in range(5):
        ref_bits = oracle.gemm_bf16(As[i].view(torch.int16).numpy().view(np.uint16),
                                    Bs[i].view(torch.int16).numpy().view(np.uint16))
        compare_bf16(Ds[i].view(torch.int16).numpy().view(np.uint16), ref_bits,
                     f"bf16 pipeline step {i} vs oracle")
        ref = tg.gemm(As[i].cuda(), Bs[i].cuda())
        tg.check()
        assert torch.equal(Ds[i], ref.cpu()), f"step {i}"
    pipe.close()
    pipe.close()   # idempotent


def test_pipeline_rejects_bad_arguments(tg):
    from tma_pipelined_tensor_tn_gb300.pipeline import HostGemmPipeline
    pipe = HostGemmPipeline(64, 64, 64)
    with pytest.raises(ValueError):
        pipe.run([torch.zeros((64, 32), dtype=torch.float16)], [torch.zeros((64, 64), dtype=torch.float16)],
                 [torch.zeros((64, 64), dtype=torch.float16)])
    with pytest.raises(ValueError):
        pipe.run([torch.zeros((64, 64), dtype=torch.float16).cuda()],
                 [torch.zeros((64, 64), dtype=torch.float16)], [torch.zeros((64, 64), dtype=torch.float16)])
    pipe.close()
