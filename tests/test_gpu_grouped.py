"""GPU parity of the grouped GEMM (gemm_f16_grouped, through the C ABI) against
the oracle's grouped definition: per group, the plain GEMM on its row window."""
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


def moe_offsets(G, tokens, seed):
    """Routed token counts per expert (a skewed draw), as row offsets."""
    rng = np.random.default_rng(seed)
    w = rng.dirichlet(np.full(G, 0.7))
    counts = np.floor(w * tokens).astype(np.int64)
    counts[0] += tokens - counts.sum()
    return np.concatenate([[0], np.cumsum(counts)]).tolist()


def run(tg, A, B, offs):
    D = tg.gemm_grouped(A.cuda(), B.cuda(), offs)
    tg.check()
    return D.cpu().numpy()


@pytest.mark.parametrize("G,tokens,N,K", [(8, 4096, 2048, 1024), (16, 3000, 1000, 4160),
                                          (64, 8192, 512, 256), (1, 1000, 1024, 512)])
def test_grouped_parity(tg, G, tokens, N, K):
    offs = moe_offsets(G, tokens, seed=G)
    g = torch.Generator().manual_seed(G + N)
    A = (torch.rand((tokens, K), generator=g) * 2 - 1).half()
    B = (torch.rand((G, N, K), generator=g) * 2 - 1).half()
    compare(run(tg, A, B, offs), oracle.gemm_f16_grouped(A.numpy(), B.numpy(), offs),
            f"grouped G={G}")


@pytest.mark.parametrize("pair", [1, 2])
def test_grouped_empty_and_tiny_groups_integer_bitexact(tg, pair):
    offs = [0, 0, 1, 130, 130, 257, 600]      # empty, 1-row, ragged groups
    G, N, K = 6, 264, 1000
    A = inputs.integer_f16((offs[-1], K), seed=90)
    B = inputs.integer_f16((G, N, K), seed=91)
    try:
        assert tg.tmagemm_set_cta_pair(pair) == tg.TMAGEMM_OK
        D = run(tg, A, B, offs)
    finally:
        tg.tmagemm_set_cta_pair(0)
    assert_bitexact(D, oracle.gemm_f16_grouped(A.numpy(), B.numpy(), offs), "grouped integer")


@pytest.mark.parametrize("pair", [1, 2])
@pytest.mark.parametrize("bn", [256, 224, 192])
def test_grouped_each_tile_width(tg, bn, pair):
    """Every tile width, single-CTA (pair=1) and CTA-pair (pair=2) tiles; a
    pair tile's second half often lies past its group's last row."""
    offs = moe_offsets(5, 1500, seed=bn)
    g = torch.Generator().manual_seed(bn)
    A = (torch.rand((1500, 520), generator=g) * 2 - 1).half()
    B = (torch.rand((5, 1000, 520), generator=g) * 2 - 1).half()
    try:
        assert tg.tmagemm_set_grouped_transposed(1) == tg.TMAGEMM_OK   # row tiles
        assert tg.tmagemm_set_tile_n(bn) == tg.TMAGEMM_OK
        assert tg.tmagemm_set_cta_pair(pair) == tg.TMAGEMM_OK
        D = run(tg, A, B, offs)
    finally:
        tg.tmagemm_set_grouped_transposed(0)
        tg.tmagemm_set_tile_n(0)
        tg.tmagemm_set_cta_pair(0)
    compare(D, oracle.gemm_f16_grouped(A.numpy(), B.numpy(), offs), f"grouped BN={bn} pair={pair}")


def test_grouped_rows_outside_groups_untouched_and_errors(tg):
    offs = [0, 100, 300]
    A = torch.zeros((300, 64), dtype=torch.float16, device="cuda")
    B = torch.zeros((2, 64, 64), dtype=torch.float16, device="cuda")
    buf = torch.full((400, 64), 7.0, dtype=torch.float16, device="cuda")
    D = buf[:300]
    assert tg.gemm_f16_grouped(2, offs, 64, 64, A.data_ptr(), B.data_ptr(), D.data_ptr(), None) == 0
    tg.check()
    assert torch.all(buf[:300] == 0) and torch.all(buf[300:] == 7.0)
    p = A.data_ptr()
    assert tg.gemm_f16_grouped(2, [0, 200, 100], 64, 64, p, p, p, None) == tg.TMAGEMM_ERR_INVALID
    assert tg.gemm_f16_grouped(2, [1, 2, 3], 64, 64, p, p, p, None) == tg.TMAGEMM_ERR_INVALID
    assert tg.gemm_f16_grouped(65, list(range(66)), 64, 64, p, p, p, None) == tg.TMAGEMM_ERR_UNSUPPORTED


@pytest.fixture(params=[(1, 1), (1, 2), (2, 1), (2, 2)],
                ids=["rows_single", "rows_pairs", "transposed_single", "transposed_pairs"])
def formulation(tg, request):
    """(grouped formulation: 1 row tiles, 2 transposed; CTA pairs: 1 never, 2 always)."""
    mode, pair = request.param
    assert tg.tmagemm_set_grouped_transposed(mode) == tg.TMAGEMM_OK
    assert tg.tmagemm_set_cta_pair(pair) == tg.TMAGEMM_OK
    yield request.param
    assert tg.tmagemm_set_grouped_transposed(0) == tg.TMAGEMM_OK
    assert tg.tmagemm_set_cta_pair(0) == tg.TMAGEMM_OK


@pytest.mark.parametrize("G,tokens,N,K", [(8, 8192, 4096, 2048), (16, 3000, 1000, 4160),
                                          (64, 8192, 512, 256), (3, 700, 1032, 72)])
def test_grouped_formulations_parity(tg, formulation, G, tokens, N, K):
    """Both formulations, single CTAs and pairs, against the oracle: the
    transposed one (a group's rows as the MMA's N in blocks of whole 16-row
    steps, the accumulator stored transposed through 16 x 128 boxes per
    group) and the row tiles.  8 x 8192 x 4096 x 2048 is the bench's shape
    (with its own routing here)."""
    offs = moe_offsets(G, tokens, seed=G + 7)
    g = torch.Generator().manual_seed(G + N + 1)
    A = (torch.rand((tokens, K), generator=g) * 2 - 1).half()
    B = (torch.rand((G, N, K), generator=g) * 2 - 1).half()
    compare(run(tg, A, B, offs), oracle.gemm_f16_grouped(A.numpy(), B.numpy(), offs),
            f"grouped {formulation} G={G}", k=K)


def test_grouped_transposed_tiny_groups_integer_bitexact(tg, formulation):
    """Empty, 1-row and ragged groups (and a group of exactly 16 rows, one of
    17): integer inputs match the oracle bit for bit in every formulation."""
    offs = [0, 0, 1, 130, 130, 257, 600, 616, 633]
    G, N, K = 8, 264, 1000
    A = inputs.integer_f16((offs[-1], K), seed=92)
    B = inputs.integer_f16((G, N, K), seed=93)
    assert_bitexact(run(tg, A, B, offs), oracle.gemm_f16_grouped(A.numpy(), B.numpy(), offs),
                    f"grouped integer {formulation}")


def test_grouped_every_block_width_integer_bitexact(tg, formulation):
    """Groups of 1..15 whole 16-row steps (each a single block of that width
    in the transposed form, which loads exactly a block's rows of A through
    the map for its width) and a 500-row group cut into blocks of two widths:
    integer inputs match the oracle bit for bit in every formulation."""
    counts = [16 * j - (j % 5) for j in range(1, 16)] + [500]
    offs = [0]
    for c in counts:
        offs.append(offs[-1] + c)
    G, N, K = len(counts), 264, 192
    A = inputs.integer_f16((offs[-1], K), seed=94)
    B = inputs.integer_f16((G, N, K), seed=95)
    assert_bitexact(run(tg, A, B, offs), oracle.gemm_f16_grouped(A.numpy(), B.numpy(), offs),
                    f"grouped widths {formulation}")


def test_grouped_full_width_blocks_integer_bitexact(tg, formulation):
    """Groups of exactly 256 rows (in the transposed form a block as wide as a
    tile, through the widest map of A), next to 250-, 17-, 512- and 1-row
    groups: integer inputs match the oracle bit for bit in every formulation."""
    counts = [256, 256, 256, 256, 250, 17, 512, 1]
    offs = [0]
    for c in counts:
        offs.append(offs[-1] + c)
    G, N, K = len(counts), 2048, 256
    A = inputs.integer_f16((offs[-1], K), seed=96)
    B = inputs.integer_f16((G, N, K), seed=97)
    assert_bitexact(run(tg, A, B, offs), oracle.gemm_f16_grouped(A.numpy(), B.numpy(), offs),
                    f"grouped 256-row blocks {formulation}")


def test_grouped_transposed_writes_only_group_rows(tg):
    """Transposed stores clip at each group's last row and at N: rows of D
    past the groups keep their contents, and every group row is written."""
    offs = [0, 37, 37, 200, 219]
    G, N, K = 4, 136, 192
    A, _ = inputs.gemm_inputs(offs[-1], 8, K, seed=94)
    _, Bf = inputs.gemm_inputs(8, G * N, K, seed=95)
    B = Bf.reshape(G, N, K)
    sentinel = torch.tensor(0x7E01, dtype=torch.int16).view(torch.float16)
    buf = torch.full((offs[-1] + 40, N), float("nan"), dtype=torch.float16, device="cuda")
    buf.view(torch.int16).fill_(0x7E01)
    try:
        assert tg.tmagemm_set_grouped_transposed(2) == tg.TMAGEMM_OK
        D = tg.gemm_grouped(A.cuda(), B.cuda(), offs, out=buf[:offs[-1]])
        tg.check()
    finally:
        tg.tmagemm_set_grouped_transposed(0)
    host = buf.cpu().view(torch.int16).numpy()
    assert np.all(host[offs[-1]:] == 0x7E01), "rows past the groups were written"
    assert not np.any(host[:offs[-1]] == 0x7E01), "some group rows were not written"
    compare(D.cpu().numpy(), oracle.gemm_f16_grouped(A.numpy(), B.numpy(), offs), "transposed guard")


def test_grouped_plan_for_the_bench_routing(tg):
    """At 8 experts x 8192 routed rows (N = 4096) on 152 SMs / 76 pairs the plan
    is transposed, in CTA pairs, with blocks of at most 240 rows; forced row
    tiles give the 224-wide pair tiles."""
    counts = [1697, 2233, 321, 376, 105, 1822, 706, 932]
    offs = [0]
    for c in counts:
        offs.append(offs[-1] + c)
    assert tg.tmagemm_grouped_plan(offs, 4096, 152, 76) == {
        "transposed": 1, "pair": 1, "bn": 256, "maxw": 240}
    try:
        assert tg.tmagemm_set_grouped_transposed(1) == tg.TMAGEMM_OK
        assert tg.tmagemm_grouped_plan(offs, 4096, 152, 76)["transposed"] == 0
    finally:
        tg.tmagemm_set_grouped_transposed(0)
