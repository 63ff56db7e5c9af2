"""GPU parity of the tcgen05 GEMM (through the C ABI) against the CPU oracle.

Sizes: the four GEMM workloads (256^3, 4096^3, ragged 4000x3000x4160 and
8192^3), each on seeds 0 and 1 and compared element by element over the whole
output, integer-valued inputs (bit-exact, 8192^3 included), the identity /
rank-1 closed forms, edge shapes next to the tile boundaries and an
out-of-bounds write guard.
"""
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


def run_gemm(tg, A, B, stream=None):
    """A, B: CPU fp16 tensors -> D (CPU fp16 numpy) computed by gemm_f16."""
    dA, dB = A.cuda(), B.cuda()
    D = tg.gemm(dA, dB, stream=stream)
    tg.check(stream)
    return D.cpu().numpy()


@pytest.mark.parametrize("name,seed", [
    ("gemm_256", 0), ("gemm_256", 1),
    ("gemm_ragged_4000x3000x4160", 0), ("gemm_ragged_4000x3000x4160", 1),
    ("gemm_4096", 0), ("gemm_4096", 1),
    ("gemm_8192", 0), ("gemm_8192", 1),
])
def test_gemm_parity_full(tg, name, seed):
    w = inputs.WORKLOADS[name]
    A, B = inputs.gemm_inputs(w["M"], w["N"], w["K"], seed=seed)
    D = run_gemm(tg, A, B)
    ref = oracle.gemm_f16(A.numpy(), B.numpy())
    stats = compare(D, ref, f"{name} seed {seed}", k=w["K"])
    print(name, seed, stats)


@pytest.mark.parametrize("M,N,K", [(256, 256, 256), (4000, 3000, 4160), (4096, 4096, 4096),
                                   (8192, 8192, 8192)])
def test_gemm_integer_bitexact(tg, M, N, K):
    # Entries in {-2..2}: every product and partial sum is an integer below 2^24,
    # so FP32 accumulation is exact and both sides round the same integer.
    A = inputs.integer_f16((M, K), seed=10)
    B = inputs.integer_f16((N, K), seed=11)
    D = run_gemm(tg, A, B)
    assert_bitexact(D, oracle.gemm_f16(A.numpy(), B.numpy()), f"integer {M}x{N}x{K}")


def test_gemm_identity_closed_forms(tg):
    g = torch.Generator().manual_seed(5)
    K, N, M = 512, 384, 640
    B = (torch.rand((N, K), generator=g) * 2 - 1).half()
    A = (torch.rand((M, K), generator=g) * 2 - 1).half()
    I = torch.eye(K, dtype=torch.float16)
    assert_bitexact(run_gemm(tg, I, B), B.numpy().T, "A = I gives B^T")
    assert_bitexact(run_gemm(tg, A, I), A.numpy(), "B = I gives A")


def test_gemm_rank1_powers_of_two(tg):
    rng = np.random.default_rng(21)
    M, N, K = 300, 264, 192
    a = rng.choice([-1, 1], M) * 2.0 ** rng.integers(-5, 3, M)
    b = rng.choice([-1, 1], N) * 2.0 ** rng.integers(-5, 3, N)
    A = torch.from_numpy(np.repeat(a[:, None], K, axis=1).astype(np.float16))
    B = torch.from_numpy(np.repeat(b[:, None], K, axis=1).astype(np.float16))
    D = run_gemm(tg, A, B)
    assert np.array_equal(D.astype(np.float64), K * np.outer(a, b))


@pytest.mark.parametrize("M,N,K", [
    (2, 8, 8), (127, 120, 64), (129, 136, 72), (200, 200, 24), (1000, 264, 296),
    (128, 256, 64), (129, 264, 8), (513, 1032, 1000), (3, 2056, 136),
])
@pytest.mark.parametrize("route", [0, 1], ids=["auto", "tile_kernel"])
def test_gemm_edge_shapes(tg, M, N, K, route):
    """route 1 (small-M swap-AB, which needs a workspace) keeps gemm_f16 on the
    tile kernel for the M <= 32 shapes too."""
    A, B = inputs.gemm_inputs(M, N, K, seed=M + N + K)
    try:
        assert tg.tmagemm_set_small_m_route(route) == tg.TMAGEMM_OK
        D = run_gemm(tg, A, B)
    finally:
        tg.tmagemm_set_small_m_route(0)
    compare(D, oracle.gemm_f16(A.numpy(), B.numpy()), f"edge {M}x{N}x{K} route {route}")


@pytest.mark.parametrize("pair", [1, 2])
@pytest.mark.parametrize("bn", [256, 224, 192])
@pytest.mark.parametrize("M,N,K", [(1031, 1000, 1032), (300, 2056, 4160)])
def test_gemm_each_tile_width(tg, bn, M, N, K, pair):
    """Every tile shape the plan can pick — single-CTA (pair=1) and CTA-pair
    (pair=2) tiles — on ragged shapes, real and integer inputs."""
    try:
        assert tg.tmagemm_set_cta_pair(pair) == tg.TMAGEMM_OK
        assert tg.tmagemm_set_tile_n(bn) == tg.TMAGEMM_OK
        A, B = inputs.gemm_inputs(M, N, K, seed=bn)
        compare(run_gemm(tg, A, B), oracle.gemm_f16(A.numpy(), B.numpy()), f"BN={bn} {M}x{N}x{K}")
        Ai = inputs.integer_f16((M, K), seed=bn + 1)
        Bi = inputs.integer_f16((N, K), seed=bn + 2)
        assert_bitexact(run_gemm(tg, Ai, Bi), oracle.gemm_f16(Ai.numpy(), Bi.numpy()), f"BN={bn} int")
    finally:
        tg.tmagemm_set_tile_n(0)
        tg.tmagemm_set_cta_pair(0)


@pytest.mark.parametrize("M,N,K", [(100, 520, 264), (129, 264, 64), (300, 136, 1000)])
def test_gemm_pair_with_half_tile_outside_m(tg, M, N, K):
    """CTA-pair tiles are 256 rows: for M <= 128 (or a last tile reaching
    less than 128 rows into the pair) the second CTA's rows are all outside D
    and its stores are skipped."""
    try:
        assert tg.tmagemm_set_cta_pair(2) == tg.TMAGEMM_OK
        A, B = inputs.gemm_inputs(M, N, K, seed=M)
        compare(run_gemm(tg, A, B), oracle.gemm_f16(A.numpy(), B.numpy()), f"pair {M}x{N}x{K}")
    finally:
        tg.tmagemm_set_cta_pair(0)


def test_gemm_pair_and_single_agree_on_4096(tg):
    A, B = inputs.gemm_inputs(4096, 4096, 4096, seed=2)
    out = {}
    try:
        for mode in (1, 2):
            assert tg.tmagemm_set_cta_pair(mode) == tg.TMAGEMM_OK
            out[mode] = run_gemm(tg, A, B)
    finally:
        tg.tmagemm_set_cta_pair(0)
    compare(out[2], out[1], "pair vs single 4096^3")


@pytest.mark.parametrize("g", [1, 2, 5, 8, 16])
def test_gemm_group_m_does_not_change_results(tg, g):
    """The tile order decides which CTA computes a tile, not how: every GROUP_M
    gives the same bits."""
    M, N, K = 1000, 3000, 520
    A, B = inputs.gemm_inputs(M, N, K, seed=70)
    ref = run_gemm(tg, A, B)
    try:
        assert tg.tmagemm_set_group_m(g) == tg.TMAGEMM_OK
        out = run_gemm(tg, A, B)
    finally:
        tg.tmagemm_set_group_m(0)
    assert_bitexact(out, ref, f"GROUP_M={g}")


def test_gemm_out_of_bounds_guard(tg):
    """D sits inside a larger buffer filled with a sentinel: after a ragged run
    the guard regions still hold it and every D element was written."""
    M, N, K = 4000, 3000, 4160
    A, B = inputs.gemm_inputs(M, N, K, seed=3)
    guard = 4096  # elements (8 KB) on each side, keeps D 16-byte aligned
    sentinel = np.uint16(0x7E01)  # a NaN pattern the kernel never produces
    buf = torch.full((guard + M * N + guard,), 0, dtype=torch.int16)
    buf.fill_(int(sentinel.view(np.int16)))
    dbuf = buf.cuda()
    D = dbuf[guard:guard + M * N].view(torch.float16).view(M, N)
    tg.gemm(A.cuda(), B.cuda(), out=D)
    tg.check()
    host = dbuf.cpu().numpy().view(np.uint16)
    assert np.all(host[:guard] == sentinel) and np.all(host[guard + M * N:] == sentinel)
    body = host[guard:guard + M * N]
    assert not np.any(body == sentinel), "some D elements were not written"
    compare(body.view(np.float16).reshape(M, N), oracle.gemm_f16(A.numpy(), B.numpy()), "guarded")


@pytest.mark.parametrize("M", [2, 8, 16, 17, 32, 33, 64, 65])
def test_gemm_few_rows_route(tg, M):
    """gemm_f16 with 2 <= M <= 16 runs the register-fragment kernel of
    gemm_f16_small_m (bit-identical); larger M the tile kernel (with its
    cluster split for these few-tile shapes)."""
    N, K = 4104, 4160
    A, B = inputs.gemm_inputs(M, N, K, seed=500 + M)
    a, b = A.cuda(), B.cuda()
    D = tg.gemm(a, b).cpu().numpy()
    tg.check()
    compare(D, oracle.gemm_f16(A.numpy(), B.numpy()), f"gemm_f16 M={M}")
    if M <= 16:
        assert_bitexact(D, tg.gemm_small_m(a, b).cpu().numpy(), f"gemm_f16 vs small-M M={M}")


def test_gemm_m1_routes_to_gemv(tg):
    x, W = inputs.gemv_inputs(1000, 1024, seed=4)
    A = x.reshape(1, -1)
    D = run_gemm(tg, A, W)
    y = tg.gemv(x.cuda(), W.cuda())
    tg.check()
    assert_bitexact(D[0], y.cpu().numpy(), "M=1 GEMM vs GEMV")
    compare(D, oracle.gemm_f16(A.numpy(), W.numpy()), "M=1")


@pytest.mark.parametrize("N,K", [(1000, 1024), (264, 8), (4096, 14336)])
def test_gemm_m1_through_tile_kernel(tg, N, K):
    """M = 1 forced through the tcgen05 tile kernel (per-call option m1_route = 1):
    equal to the oracle, and within tolerance of the GEMV path that gemm_f16
    takes for M = 1 by default ("Learning TileLang with GEMV", 01 GEMV: the
    decode step is the M = 1 case of the same GEMM)."""
    x, W = inputs.gemv_inputs(N, K, seed=N + K)
    A = x.reshape(1, -1)
    ref = oracle.gemm_f16(A.numpy(), W.numpy())
    dA, dW = A.cuda(), W.cuda()
    D_tile = tg.gemm(dA, dW, opts=tg.options(m1_route=1))
    D_gemv = tg.gemm(dA, dW)
    tg.check()
    D_tile, D_gemv = D_tile.cpu().numpy(), D_gemv.cpu().numpy()
    compare(D_tile, ref, f"M=1 tile kernel {N}x{K} vs oracle")
    compare(D_gemv, ref, f"M=1 GEMV {N}x{K} vs oracle")
    compare(D_tile, D_gemv, f"M=1 tile kernel vs GEMV {N}x{K}")
    # integer-valued inputs: both paths equal the oracle bit for bit
    xi = inputs.integer_f16((1, K), seed=N)
    Wi = inputs.integer_f16((N, K), seed=K)
    Di = tg.gemm(xi.cuda(), Wi.cuda(), opts=tg.options(m1_route=1))
    tg.check()
    assert_bitexact(Di.cpu().numpy(), oracle.gemm_f16(xi.numpy(), Wi.numpy()), "M=1 tile integer")


def test_gemm_m1_tile_kernel_needs_n_multiple_of_8(tg):
    x, W = inputs.gemv_inputs(1001, 64, seed=3)
    D = torch.empty((1, 1001), dtype=torch.float16, device="cuda")
    s = tg.gemm_f16_ex(1, 1001, 64, x.cuda().data_ptr(), W.cuda().data_ptr(), D.data_ptr(),
                       tg.options(m1_route=1))
    assert s == tg.TMAGEMM_ERR_ALIGN
    s = tg.gemm_f16_ex(1, 1001, 64, x.cuda().data_ptr(), W.cuda().data_ptr(), D.data_ptr(), None)
    assert s == tg.TMAGEMM_OK   # the GEMV takes any N
    tg.check()


@pytest.mark.parametrize("fields", [
    dict(), dict(tile_n=192, cta_pair=1), dict(tile_n=224, cta_pair=2), dict(tail_split=1),
    dict(group_m=3), dict(plain_launch=1), dict(cluster_split=1),
])
def test_gemm_per_call_options(tg, fields):
    """gemm_f16_ex under per-call options: the oracle's result, and the
    process-wide settings are untouched (a later gemm_f16 equals one made
    before)."""
    M, N, K = 1000, 1032, 1096
    A, B = inputs.gemm_inputs(M, N, K, seed=80)
    dA, dB = A.cuda(), B.cuda()
    before = tg.gemm(dA, dB)
    D = tg.gemm(dA, dB, opts=tg.options(**fields))
    after = tg.gemm(dA, dB)
    tg.check()
    compare(D.cpu().numpy(), oracle.gemm_f16(A.numpy(), B.numpy()), f"options {fields}")
    assert torch.equal(before, after)


def test_gemm_options_from_two_host_threads(tg):
    """Two host threads, each on its own stream, one with forced options and
    one with the defaults: every result equals the oracle's (per-call options
    change nothing for the other thread)."""
    import threading
    M, N, K = 512, 776, 1032
    A, B = inputs.gemm_inputs(M, N, K, seed=81)
    ref = oracle.gemm_f16(A.numpy(), B.numpy())
    dA, dB = A.cuda(), B.cuda()
    results, errors = {}, []

    def worker(name, opts):
        try:
            s = torch.cuda.Stream()
            outs = []
            with torch.cuda.stream(s):
                for _ in range(20):
                    outs.append(tg.gemm(dA, dB, stream=s, opts=opts))
            s.synchronize()
            results[name] = [o.cpu().numpy() for o in outs]
        except Exception as e:   # reported in the main thread
            errors.append(e)

    ts = [threading.Thread(target=worker, args=("forced", tg.options(tile_n=192, cta_pair=1))),
          threading.Thread(target=worker, args=("default", None))]
    for t in ts:
        t.start()
    for t in ts:
        t.join()
    assert not errors, errors
    tg.check()
    for name, outs in results.items():
        for i, D in enumerate(outs):
            compare(D, ref, f"{name} thread, call {i}")


def test_gemm_transpose_symmetry(tg):
    A, B = inputs.gemm_inputs(640, 512, 1024, seed=6)
    D1 = run_gemm(tg, A, B)
    D2 = run_gemm(tg, B, A)
    compare(D2, D1.T, "gemm(B, A) vs gemm(A, B)^T")
    print("transpose symmetry bit-exact:", np.array_equal(D2.view(np.uint16), D1.T.view(np.uint16)))


def test_gemm_side_stream_and_repeat(tg):
    A, B = inputs.gemm_inputs(1024, 768, 512, seed=8)
    s = torch.cuda.Stream()
    dA, dB = A.cuda(), B.cuda()
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        D1 = tg.gemm(dA, dB, stream=s)
        D2 = tg.gemm(dA, dB, stream=s)
    tg.check(s)
    assert_bitexact(D1.cpu().numpy(), D2.cpu().numpy(), "repeatable")
    compare(D1.cpu().numpy(), oracle.gemm_f16(A.numpy(), B.numpy()), "side stream")


def test_gemm_misaligned_device_pointer_rejected(tg):
    buf = torch.zeros(256 * 256 + 8, dtype=torch.float16, device="cuda")
    p = buf.data_ptr()
    assert tg.gemm_f16(256, 256, 256, p + 2, p, p, None) == tg.TMAGEMM_ERR_ALIGN
    assert tg.gemm_f16(256, 256, 260, p, p, p, None) == tg.TMAGEMM_ERR_ALIGN


def test_wait_timeout_is_reported_and_context_survives(tg):
    """A wait that nobody completes ends with a TIMEOUT status, not a hang; the
    next GEMM on the same context still works."""
    assert tg.tmagemm_check(None) == tg.TMAGEMM_OK
    assert tg.tmagemm_selftest_wait_timeout(200, None) == tg.TMAGEMM_OK
    assert tg.tmagemm_check(None) == tg.TMAGEMM_ERR_TIMEOUT
    assert tg.tmagemm_last_error_detail() & 0xFF == 7
    assert tg.tmagemm_check(None) == tg.TMAGEMM_OK          # cleared
    A, B = inputs.gemm_inputs(256, 256, 256, seed=9)
    compare(run_gemm(tg, A, B), oracle.gemm_f16(A.numpy(), B.numpy()), "after timeout")


def random_shapes(seed, count):
    """Seeded random shapes across the supported space: M any size >= 2,
    N and K multiples of 8, spanning one tile to several waves."""
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(count):
        M = int(rng.integers(2, 2600))
        N = 8 * int(rng.integers(1, 330))
        K = 8 * int(rng.integers(1, 600))
        out.append((M, N, K))
    return out


@pytest.mark.parametrize("M,N,K", random_shapes(2024, 12))
def test_gemm_random_shapes(tg, M, N, K):
    A, B = inputs.gemm_inputs(M, N, K, seed=M * 7 + N)
    compare(run_gemm(tg, A, B), oracle.gemm_f16(A.numpy(), B.numpy()), f"random {M}x{N}x{K}")


@pytest.mark.parametrize("M,N,K", random_shapes(77, 6))
def test_splitk_random_shapes(tg, M, N, K):
    A, B = inputs.gemm_inputs(M, N, K, seed=M + 3 * N)
    D = tg.gemm_splitk(A.cuda(), B.cuda(), splits=0)
    tg.check()
    compare(D.cpu().numpy(), oracle.gemm_f16(A.numpy(), B.numpy()), f"split-K random {M}x{N}x{K}")
