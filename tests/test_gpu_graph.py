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


def test_graph_replay_small_m_and_cluster_split(tg):
    """The register-fragment and LSU-fed small-M kernels and gemm_f16's cluster
    split (clusters of 4, distributed shared memory) replay from a graph with
    the direct calls' bits."""
    X8, W = (t.cuda() for t in inputs.gemv_inputs(4096, 4096, seed=210))
    X8 = X8.reshape(1, -1).repeat(8, 1).contiguous()
    X24 = torch.randn((24, 4096), generator=torch.Generator().manual_seed(211)).half().mul_(0.02).cuda()
    A, B = (t.cuda() for t in inputs.gemm_inputs(1024, 1024, 16384, seed=212))
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert tg.tmagemm_gemm_plan(1024, 1024, 16384, sms, 1, sms // 2)["cluster_k"] > 0
    ref8 = tg.gemm_small_m(X8, W).cpu().numpy()
    ref24 = tg.gemm_small_m(X24, W).cpu().numpy()
    refc = tg.gemm(A, B).cpu().numpy()
    tg.check()
    d8 = torch.empty((8, 4096), dtype=torch.float16, device="cuda")
    d24 = torch.empty((24, 4096), dtype=torch.float16, device="cuda")
    dc = torch.empty((1024, 1024), dtype=torch.float16, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        tg.gemm_small_m(X8, W, out=d8, stream=s)
        tg.gemm_small_m(X24, W, out=d24, stream=s)
        tg.gemm(A, B, out=dc, stream=s)
    for _ in range(2):
        for t in (d8, d24, dc):
            t.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert_bitexact(d8.cpu().numpy(), ref8, "graph small-M 8")
        assert_bitexact(d24.cpu().numpy(), ref24, "graph small-M 24")
        assert_bitexact(dc.cpu().numpy(), refc, "graph cluster split")
    tg.check()


def test_two_streams_concurrently(tg):
    """gemm_f16 and gemv_f16 keep no shared device state between calls: two
    streams running them at the same time give the sequential results."""
    shapes = [(2048, 2056, 1032), (1000, 3000, 4160)]
    ins = [tuple(t.cuda() for t in inputs.gemm_inputs(*sh, seed=220 + i)) for i, sh in enumerate(shapes)]
    refs = [tg.gemm(a, b).cpu().numpy() for a, b in ins]
    x, W = (t.cuda() for t in inputs.gemv_inputs(4096, 14336, seed=222))
    yref = tg.gemv(x, W).cpu().numpy()
    tg.check()
    streams = [torch.cuda.Stream() for _ in range(2)]
    outs = [torch.empty((sh[0], sh[1]), dtype=torch.float16, device="cuda") for sh in shapes]
    ys = [torch.empty((4096,), dtype=torch.float16, device="cuda") for _ in range(2)]
    for st in streams:
        st.wait_stream(torch.cuda.current_stream())
    for rep in range(5):
        for i, st in enumerate(streams):
            tg.gemm(*ins[i], out=outs[i], stream=st)
            tg.gemv(x, W, out=ys[i], stream=st)
    torch.cuda.synchronize()
    tg.check()
    for i in range(2):
        assert_bitexact(outs[i].cpu().numpy(), refs[i], f"stream {i} GEMM")
        assert_bitexact(ys[i].cpu().numpy(), yref, f"stream {i} GEMV")
