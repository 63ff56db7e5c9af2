"""GPU parity of gemm_f16's tail split.  When the last round of the
persistent tile schedule fills at most half of the resident CTAs (or CTA
pairs), each tile of that round runs as two work units over its column range
(128 columns, then the rest of the tile), so that round takes about half as
long.  Every output is still one unit's sum over all of K, so D = fp16(A @ B.T)
as for the plain GEMM (same oracle), and the result is bit-identical to the
schedule without the split."""
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


def ceil_div(a, b):
    return -(-a // b)


def set_knobs(tg, pair_mode, bn, tail=0):
    assert tg.tmagemm_set_cta_pair(pair_mode) == tg.TMAGEMM_OK
    assert tg.tmagemm_set_tile_n(bn) == tg.TMAGEMM_OK
    assert tg.tmagemm_set_tail_split(tail) == tg.TMAGEMM_OK


def reset(tg):
    tg.tmagemm_set_cta_pair(0)
    tg.tmagemm_set_tile_n(0)
    tg.tmagemm_set_tail_split(0)


def run(tg, A, B, pair_mode=0, bn=0, tail=0):
    """D from gemm_f16 (or gemm_bf16) with the given knobs, and the device plan."""
    try:
        set_knobs(tg, pair_mode, bn, tail)
        M, N, K = A.shape[0], B.shape[0], A.shape[1]
        tp = tg.tmagemm_gemm_tail_plan(M, N, K, 0)
        p = tg.tmagemm_gemm_plan(M, N, K, 0)
        D = tg.gemm(A.cuda(), B.cuda())
        tg.check()
    finally:
        reset(tg)
    return D.cpu(), p, tp


def slots(tg, pair_mode):
    """Resident work slots of the device's plan: CTA pairs or single CTAs."""
    try:
        set_knobs(tg, pair_mode, 256)
        p = tg.tmagemm_gemm_plan(256 * 64, 256 * 64, 64, 0)
    finally:
        reset(tg)
    return p["grid"] // (2 if p["pair"] else 1), p["pair"]


def tail_shape(tg, pair_mode, bn):
    """A ragged (M, N) whose tiles fill whole rounds plus a short last round:
    four tile columns (N = 4 bn - 40) and one more tile row than whole rounds
    need, so the last round holds 4 - slots % 4 tiles (4 when slots % 4 == 0)."""
    s, pair = slots(tg, pair_mode)
    tile_m = 256 if pair else 128
    grid_m = s // 4 + 1
    return grid_m * tile_m - 50, 4 * bn - 40


# Every tile width, in CTA pairs (2) and single CTAs (1); K ragged (2.1 k-blocks).
@pytest.mark.parametrize("bn", [256, 224, 192])
@pytest.mark.parametrize("pair_mode", [2, 1], ids=["pairs", "single"])
def test_tail_split_parity_and_bitexact(tg, pair_mode, bn):
    M, N = tail_shape(tg, pair_mode, bn)
    K = 136
    A, B = inputs.gemm_inputs(M, N, K, seed=bn + pair_mode)
    D, p, tp = run(tg, A, B, pair_mode, bn)
    assert p["BN"] == bn and p["cluster_k"] == 0, p
    assert tp["split_tiles"] > 0 and tp["full_units"] > 0, (tp, p)
    assert tp["narrow_cols"] == 128, tp
    assert p["units"] == tp["full_units"] + 2 * tp["split_tiles"], (tp, p)
    compare(D.numpy(), oracle.gemm_f16(A.numpy(), B.numpy()),
            f"tail split {M}x{N}x{K} BN={bn} pair mode {pair_mode}")
    # The same tiles without the split: the same bits.
    D0, p0, tp0 = run(tg, A, B, pair_mode, bn, tail=1)
    assert tp0["split_tiles"] == 0 and p0["units"] == p0["tiles"], (tp0, p0)
    assert_bitexact(D.numpy(), D0.numpy(), f"tail split on/off BN={bn} pair mode {pair_mode}")


def test_second_part_past_the_last_column(tg):
    """N = 3 * 256 + 64: the last tile column holds 64 columns, so its second
    part (columns 128..255) lies wholly outside D: its loads read zeros and it
    stores nothing."""
    M, N = tail_shape(tg, 2, 256)
    N, K = 3 * 256 + 64, 200
    A, B = inputs.gemm_inputs(M, N, K, seed=79)
    D, p, tp = run(tg, A, B, 2, 256)
    assert tp["split_tiles"] > 0 and p["BN"] == 256, (tp, p)
    compare(D.numpy(), oracle.gemm_f16(A.numpy(), B.numpy()), "empty second part")


def test_every_tile_split_when_one_round_is_half_full(tg):
    """Fewer tiles than half the slots: no whole rounds, every tile in two parts."""
    M, N, K = 1000, 1000, 520
    A, B = inputs.gemm_inputs(M, N, K, seed=77)
    D, p, tp = run(tg, A, B, 2, 256)
    assert tp["full_units"] == 0 and tp["split_tiles"] == p["tiles"] == 16, (tp, p)
    compare(D.numpy(), oracle.gemm_f16(A.numpy(), B.numpy()), "all tiles split")


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_integer_inputs_exact(tg, dtype):
    """Integer-valued inputs: FP32 sums are exact, so D is the oracle's rounding
    of the exact sum, bit for bit, in the split parts as in whole tiles."""
    bn = 224
    M, N = tail_shape(tg, 2, bn)
    K = 520
    A = inputs.integer_f16((M, K), seed=80)
    B = inputs.integer_f16((N, K), seed=81)
    if dtype == "bf16":
        A, B = A.to(torch.bfloat16), B.to(torch.bfloat16)
    D, p, tp = run(tg, A, B, 2, bn)
    assert tp["split_tiles"] > 0, tp
    if dtype == "bf16":
        bits = lambda t: t.contiguous().view(torch.int16).numpy().view(np.uint16)
        assert np.array_equal(bits(D), oracle.gemm_bf16(bits(A), bits(B)))
    else:
        assert_bitexact(D.numpy(), oracle.gemm_f16(A.numpy(), B.numpy()), "integer tail split")


def test_automatic_plan_8192(tg):
    """8192^3 on the device: 256 x 256 pair tiles with the last round split
    whenever it is at most half full (13.47 rounds of 76 pairs on GB300)."""
    tp = tg.tmagemm_gemm_tail_plan(8192, 8192, 8192, 0)
    p = tg.tmagemm_gemm_plan(8192, 8192, 8192, 0)
    s = p["grid"] // (2 if p["pair"] else 1)
    tail = p["tiles"] % s
    if 0 < tail <= s // 2 and p["BN"] in (256, 224, 192):
        assert tp["split_tiles"] == tail and tp["full_units"] == p["tiles"] - tail, (tp, p)
    assert p["units"] == tp["full_units"] + 2 * tp["split_tiles"], (tp, p)
