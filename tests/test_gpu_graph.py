"""gemm_f16 / gemv_f16 / gemm_f16_splitk inside a captured CUDA graph: the C ABI
enqueues plain kernel launches (tensor maps are encoded on the host at capture
time and travel as kernel parameters), so replays give the same results as
direct calls."""
import numpy as np
import pytest

from tma_pipelined_tensor_tn_gb300 import inputs
from tests.parity_util import assert_bitexact

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tg():
    import tma_pipelined_tensor_tn_gb300 as m
    m.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return m


def test_graph_replay_matches_direct_calls(tg):
    M, N, K = 1024, 1032, 2056
    A, B = (t.cuda() for t in inputs.gemm_inputs(M, N, K, seed=200))
    x, W = (t.cuda() for t in inputs.gemv_inputs(4096, 14336, seed=201))
    A2, B2 = (t.cuda() for t in inputs.gemm_inputs(512, 512, 16384, seed=202))
    need = tg.gemm_f16_splitk_workspace_size(512, 512, 16384, 4)
    ws = torch.empty((need,), dtype=torch.uint8, device="cuda")
    D = torch.empty((M, N), dtype=torch.float16, device="cuda")
    y = torch.empty((4096,), dtype=torch.float16, device="cuda")
    D2 = torch.empty((512, 512), dtype=torch.float16, device="cuda")
    ref_D = tg.gemm(A, B).cpu().numpy()
    ref_y = tg.gemv(x, W).cpu().numpy()
    ref_D2 = tg.gemm_splitk(A2, B2, workspace=ws, splits=4).cpu().numpy()
    tg.check()

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        tg.gemm(A, B, out=D, stream=s)
        tg.gemv(x, W, out=y, stream=s)
        tg.gemm_splitk(A2, B2, workspace=ws, splits=4, out=D2, stream=s)
    for _ in range(3):
        D.zero_()
        y.zero_()
        D2.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert_bitexact(D.cpu().numpy(), ref_D, "graph gemm")
        assert_bitexact(y.cpu().numpy(), ref_y, "graph gemv")
        assert_bitexact(D2.cpu().numpy(), ref_D2, "graph split-K")
    tg.check()
