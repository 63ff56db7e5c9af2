"""Host-side tests of the CUDA library that need no GPU.

* the library loads and exports every symbol include/tmagemm.h declares;
* argument validation returns status codes before any CUDA call;
* the persistent schedule and the pipeline ring (the same functions the
  kernel runs, exported for introspection) against the pages' worked examples.
"""
import json
import os
import re

import pytest

import tma_pipelined_tensor_tn_gb300 as tg
from tma_pipelined_tensor_tn_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
GOLDEN = os.path.join(ROOT, "tests", "golden")


@pytest.fixture(scope="module", autouse=True)
def built():
    _build.build()
    return tg.lib()


def header_functions():
    text = open(os.path.join(ROOT, "include", "tmagemm.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\**\s+\**(\w+)\s*\(", text, flags=re.M)))


def test_header_is_plain_c(tmp_path):
    """include/tmagemm.h is a C ABI: it compiles as C99 and as C++17 with no
    warnings, with nothing but the standard headers it includes itself."""
    import shutil
    import subprocess
    src = tmp_path / "use_header.c"
    src.write_text('#include "tmagemm.h"\nint main(void) { return tmagemm_version() > 0 ? 0 : 1; }\n')
    inc = os.path.join(ROOT, "include")
    for cc, args in (("gcc", ["-std=c99"]), ("g++", ["-std=c++17", "-x", "c++"])):
        if shutil.which(cc) is None:
            pytest.skip(f"{cc} not available")
        r = subprocess.run([cc, *args, "-Wall", "-Wextra", "-Werror", "-I", inc, "-fsyntax-only",
                            str(src)], capture_output=True, text=True)
        assert r.returncode == 0, (cc, r.stderr)


def test_library_exports_every_header_symbol():
    names = header_functions()
    assert "gemm_f16" in names and "gemv_f16" in names
    L = tg.lib()
    for n in names:
        assert hasattr(L, n), n
        assert n in tg.SIGNATURES, n


def test_options_init_and_validation():
    """tmagemm_options_init zeroes every field; gemm_f16_ex / gemm_bf16_ex refuse
    a field outside its range before any CUDA call."""
    import ctypes
    o = tg.TmagemmOptions()
    for name, _ in tg.TmagemmOptions._fields_:
        setattr(o, name, 7)
    tg.lib().tmagemm_options_init(ctypes.byref(o))
    assert all(getattr(o, name) == 0 for name, _ in tg.TmagemmOptions._fields_)
    tg.lib().tmagemm_options_init(None)   # a no-op
    assert ctypes.sizeof(tg.TmagemmOptions) == 8 * 4
    bad = [dict(tile_n=100), dict(tile_n=-1), dict(cta_pair=3), dict(cluster_split=3),
           dict(cluster_split=16), dict(tail_split=2), dict(group_m=65), dict(small_m_route=4),
           dict(plain_launch=2), dict(m1_route=2), dict(m1_route=-1)]
    dummy = 1 << 20   # never dereferenced: validation fails first
    for fields in bad:
        opts = tg.options(**fields)
        for fn in (tg.gemm_f16_ex, tg.gemm_bf16_ex):
            assert fn(256, 256, 256, dummy, dummy, dummy, opts) == tg.TMAGEMM_ERR_INVALID, fields
    with pytest.raises(TypeError):
        tg.options(no_such_field=1)


def test_host_pipeline_argument_checks():
    """Checked before any CUDA call: bad sizes and NULL handles are refused."""
    import ctypes
    L = tg.lib()
    h = ctypes.c_void_p()
    for args in [(0, 64, 64, 2, 0), (64, -1, 64, 2, 0), (64, 64, 64, 0, 0), (64, 64, 64, 17, 0),
                 (64, 64, 64, 2, 2)]:
        assert L.tmagemm_host_pipeline_create(*args, ctypes.byref(h)) == tg.TMAGEMM_ERR_INVALID
        assert not h.value
    assert L.tmagemm_host_pipeline_create(64, 64, 64, 2, 0, None) == tg.TMAGEMM_ERR_INVALID
    assert L.tmagemm_host_pipeline_run(None, 1, None, None, None) == tg.TMAGEMM_ERR_INVALID
    assert L.tmagemm_host_pipeline_synchronize(None) == tg.TMAGEMM_ERR_INVALID
    L.tmagemm_host_pipeline_destroy(None)   # a no-op


def test_checked_api_in_the_normal_build():
    """The normal build exports the checked-build query and refuses it before
    any CUDA call; the check status has its own message."""
    assert not tg.CHECKED and tg.LIB_PATH.endswith("libtmagemm.so")
    assert tg.lib().tmagemm_checked_unit_counts(None, 0, None) == tg.TMAGEMM_ERR_UNSUPPORTED
    assert "self-check" in tg.strerror(tg.TMAGEMM_ERR_CHECK)


def test_strerror_covers_all_codes():
    for code in (0, -1, -2, -3, -4, -5, -6, -7, -8):
        assert tg.strerror(code) and tg.strerror(code) != "unknown status"
    assert tg.strerror(12345) == "unknown status"


@pytest.mark.parametrize("M,N,K,expect", [
    (0, 256, 256, tg.TMAGEMM_ERR_INVALID),
    (256, -1, 256, tg.TMAGEMM_ERR_INVALID),
    (256, 256, 0, tg.TMAGEMM_ERR_INVALID),
    (256, 256, 260, tg.TMAGEMM_ERR_ALIGN),      # K % 8
    (256, 250, 256, tg.TMAGEMM_ERR_ALIGN),      # N % 8 (M > 1)
    (1 << 31, 256, 256, tg.TMAGEMM_ERR_UNSUPPORTED),
])
def test_gemm_validation_codes(M, N, K, expect):
    p = 1 << 20   # aligned fake address: validation fails before it is touched
    assert tg.gemm_f16(M, N, K, p, p, p, None) == expect


def test_gemm_null_and_misaligned_pointers():
    p = 1 << 20
    assert tg.gemm_f16(256, 256, 256, None, p, p, None) == tg.TMAGEMM_ERR_INVALID
    assert tg.gemm_f16(256, 256, 256, p, p, None, None) == tg.TMAGEMM_ERR_INVALID
    assert tg.gemm_f16(256, 256, 256, p + 2, p, p, None) == tg.TMAGEMM_ERR_ALIGN
    assert tg.gemm_f16(256, 256, 256, p, p + 8, p, None) == tg.TMAGEMM_ERR_ALIGN
    # M == 1 goes to the GEMV rules: N need not be a multiple of 8, K must be.
    assert tg.gemm_f16(1, 250, 260, p, p, p, None) == tg.TMAGEMM_ERR_ALIGN
    assert tg.gemv_f16(4096, 14336, p, p, p + 4, None) == tg.TMAGEMM_ERR_ALIGN
    assert tg.gemv_f16(4096, 0, p, p, p, None) == tg.TMAGEMM_ERR_INVALID
    assert tg.gemm_f16_splitk(256, 256, 256, p, p, p, -1, p, 1 << 20, None) == tg.TMAGEMM_ERR_INVALID
    assert tg.gemm_f16_splitk(256, 256, 260, p, p, p, 2, p, 1 << 20, None) == tg.TMAGEMM_ERR_ALIGN


def test_group_m_order_golden():
    g = json.load(open(os.path.join(GOLDEN, "persistent_schedule.json")))
    for c in g["cases"]:
        assert tg.tmagemm_tile_coord(c["tile"], c["grid_m"], c["grid_n"], g["group_m"]) == (c["m"], c["n"]), c


@pytest.mark.parametrize("grid_m,grid_n", [(32, 32), (2, 2), (10, 3), (32, 12), (63, 17), (1, 5)])
def test_group_m_order_is_a_bijection(grid_m, grid_n):
    seen = set()
    for t in range(grid_m * grid_n):
        m, n = tg.tmagemm_tile_coord(t, grid_m, grid_n, 8)
        assert 0 <= m < grid_m and 0 <= n < grid_n
        seen.add((m, n))
    assert len(seen) == grid_m * grid_n


def test_tile_coord_rejects_out_of_range():
    with pytest.raises(tg.TmaGemmError):
        tg.tmagemm_tile_coord(4, 2, 2, 8)


def test_ring_reduces_to_pipeline_trace():
    g = json.load(open(os.path.join(GOLDEN, "pipeline_depth2_k5.json")))
    S, KT = g["pipe_depth"], g["k_tiles"]
    stages, tma_ph, mma_ph, refill = [], [], [], []
    for it in range(KT):
        s, ph = tg.tmagemm_ring_position(it, S)
        stages.append(s)
        tma_ph.append(ph)
        # one barrier reused every iteration (the page's single MMA barrier)
        mma_ph.append(tg.tmagemm_ring_position(it, 1)[1])
        # a producer refills a stage with load it + S once iteration it freed it
        refill.append(it + S if it + S < KT else None)
    assert stages == g["stage"]
    assert tma_ph == g["phase_tma"]
    assert mma_ph == g["phase_mma"]
    assert refill == g["refill_tile"]


class MBarrierModel:
    """Phase counter of an mbarrier with arrival count 1."""

    def __init__(self):
        self.completed = 0

    def arrive(self):
        self.completed += 1

    def wait_ok(self, parity):
        # try_wait.parity(P) succeeds once the phase with parity P completed,
        # i.e. when the current (incomplete) phase has the other parity.
        return (self.completed & 1) != parity


@pytest.mark.parametrize("k_tiles,stages", [(64, 2), (65, 4), (4, 4), (65, 2), (3, 5)])
def test_running_ring_counter_matches_barrier_phases(k_tiles, stages):
    """Consumer waits issued with the kernel's ring parity always match the
    barrier's state across tiles, for any K_TILES (odd ones included)."""
    full = [MBarrierModel() for _ in range(stages)]
    it = 0
    for _tile in range(3):
        for _kb in range(k_tiles):
            s, ph = tg.tmagemm_ring_position(it, stages)
            assert not full[s].wait_ok(ph)      # not complete before the load lands
            full[s].arrive()                    # TMA completes the phase
            assert full[s].wait_ok(ph)
            it += 1


def test_per_tile_phase_reset_breaks_with_odd_barrier_counts():
    """The page's per-tile reset of phases needs every barrier to be used an even
    number of times per tile; with 65 k-blocks the reset parity is wrong."""
    g = json.load(open(os.path.join(GOLDEN, "persistent_schedule.json")))
    kt, S = g["k_tiles"], g["pipe_depth"]
    uses = [0] * S
    for it in range(kt):
        uses[tg.tmagemm_ring_position(it, S)[0]] += 1
    assert uses == [g["tma_bar_uses_per_stage_per_tile"]] * S
    assert kt == g["mma_bar_uses_per_tile"]
    # odd count: after one tile of 65 uses the single MMA barrier has odd parity
    bar = MBarrierModel()
    for _ in range(65):
        bar.arrive()
    assert bar.completed & 1 == 1          # resetting the expected parity to 0 would be wrong
    assert tg.tmagemm_ring_position(65, 1)[1] == 1   # the running counter gets it right


def test_plan_for_the_workloads():
    g = json.load(open(os.path.join(GOLDEN, "persistent_schedule.json")))
    # The page's exercise: 4096^2 output, 128x128 tiles -> 1024 tiles.
    assert (4096 // 128) * (4096 // 128) == g["tiles_4096_128x128"]
    p = tg.tmagemm_gemm_plan(4096, 4096, 4096, 152)
    assert (p["BM"], p["BK"]) == (128, 64)
    assert p["tiles"] == -(-4096 // p["BM"]) * -(-4096 // p["BN"])
    assert p["grid"] == min(p["tiles"], 152)
    assert p["smem"] <= 232448
    r = tg.tmagemm_gemm_plan(4000, 3000, 4160, 152)
    assert r["tiles"] == -(-4000 // r["BM"]) * -(-3000 // r["BN"])
    s = tg.tmagemm_gemm_plan(256, 256, 256, 152)
    assert s["tiles"] <= 4
    # One short round: every tile runs as its two column parts.
    assert s["grid"] == s["units"] == 2 * s["tiles"]


def test_plan_balances_waves_on_gb300():
    # 4096^3 on 152 SMs: 128x224 tiles give 32 x 19 = 608 = 4 x 152 tiles, so
    # every SM runs exactly four tiles (128x256 would leave a partial 4th wave).
    p = tg.tmagemm_gemm_plan(4096, 4096, 4096, 152)
    assert p["BN"] == 224 and p["tiles"] == 4 * 152
    assert tg.tmagemm_gemm_plan(8192, 8192, 8192, 152)["BN"] == 256


def test_plan_with_cta_pairs_balances_waves():
    # With 76 co-resident CTA pairs, 256 x 224 pair tiles give 16 x 19 = 304 =
    # 4 x 76 tiles at 4096^3; 8192^3 takes 256 x 256 pair tiles.
    p = tg.tmagemm_gemm_plan(4096, 4096, 4096, 152, 1, 76)
    assert p["pair"] == 1 and p["BN"] == 224 and p["tiles"] == 4 * 76 and p["grid"] == 152
    q = tg.tmagemm_gemm_plan(8192, 8192, 8192, 152, 1, 76)
    assert q["pair"] == 1 and q["BN"] == 256
    # split-K plans never use pairs
    assert tg.tmagemm_gemm_plan(1024, 1024, 16384, 152, 0, 76)["pair"] == 0


def test_cluster_split_ranking():
    """Among cluster splits the plan weighs each CTA's B stream, the HBM
    floor and the distributed-shared-memory reduction, not k-blocks alone:
    a full 128-row tile makes a 4-way reduction of 256-wide tiles cost more
    than the 2-way reduction of 192-wide ones (measured on GB300: 31.5-32.1
    against 32.7-33.3 us at 128 x 8192 x 8192), and few tiles of a small
    problem favour 4-way 128-wide over 8-way 256-wide splits (11.9 against
    16.4 us at 128 x 3072 x 3072)."""
    p = tg.tmagemm_gemm_plan(128, 8192, 8192, 152, 1, 76)
    assert (p["cluster_k"], p["BN"], p["pair"], p["grid"]) == (2, 192, 0, 86), p
    q = tg.tmagemm_gemm_plan(128, 3072, 3072, 152, 1, 76)
    assert (q["cluster_k"], q["BN"], q["pair"]) == (4, 128, 0), q
    # A few tokens keep the 4-way 256-wide split: its reduction covers one warp of rows.
    r = tg.tmagemm_gemm_plan(32, 8192, 8192, 152, 1, 76)
    assert (r["cluster_k"], r["BN"], r["pair"]) == (4, 256, 0), r


def test_tail_split_plan():
    """A last round at most half full runs its tiles as two column parts: the
    whole rounds keep whole tiles, the parts fill the last round once."""
    t = tg.tmagemm_gemm_tail_plan(8192, 8192, 8192, 152, 76)
    p = tg.tmagemm_gemm_plan(8192, 8192, 8192, 152, 1, 76)
    # 32 x 32 = 1024 pair tiles = 13 rounds of 76 + 36
    assert (p["BN"], p["pair"], p["tiles"]) == (256, 1, 1024)
    assert t == {"full_units": 13 * 76, "split_tiles": 36, "narrow_cols": 128}
    assert p["units"] == 13 * 76 + 72 and p["grid"] == 152
    # 4096^3 fills four whole rounds of 256 x 224 pair tiles: nothing to split.
    assert tg.tmagemm_gemm_tail_plan(4096, 4096, 4096, 152, 76)["split_tiles"] == 0
    assert tg.tmagemm_gemm_plan(4096, 4096, 4096, 152, 1, 76)["BN"] == 224
    try:
        assert tg.tmagemm_set_tail_split(1) == tg.TMAGEMM_OK
        off = tg.tmagemm_gemm_tail_plan(8192, 8192, 8192, 152, 76)
        assert off == {"full_units": 1024, "split_tiles": 0, "narrow_cols": 0}
        assert tg.tmagemm_gemm_plan(8192, 8192, 8192, 152, 1, 76)["units"] == 1024
        assert tg.tmagemm_set_tail_split(2) == tg.TMAGEMM_ERR_INVALID
        assert tg.tmagemm_set_tail_split(-1) == tg.TMAGEMM_ERR_INVALID
    finally:
        assert tg.tmagemm_set_tail_split(0) == tg.TMAGEMM_OK
    with pytest.raises(tg.TmaGemmError):
        tg.tmagemm_gemm_tail_plan(0, 8, 8, 152, 76)


def test_tail_split_with_operands_in_l2():
    """Operands that fit in L2 (2(M+N)K + 2MN <= 96 MiB): a pair plan's parts
    run near their width, so 1024 x 6144 x 4096 takes 112 pair tiles of 224
    with the last 36 split (measured 36.4 us) over 128 tiles of 192 in two
    whole rounds (37.7 us).  Single CTAs' parts keep the full-round charge:
    384 x 14336 x 2048 stays on two rounds of 192-wide pair tiles."""
    p = tg.tmagemm_gemm_plan(1024, 6144, 4096, 152, 1, 76)
    t = tg.tmagemm_gemm_tail_plan(1024, 6144, 4096, 152, 76)
    assert (p["BN"], p["pair"], p["tiles"]) == (224, 1, 112), p
    assert t == {"full_units": 76, "split_tiles": 36, "narrow_cols": 128}
    q = tg.tmagemm_gemm_plan(384, 14336, 2048, 152, 1, 76)
    assert (q["BN"], q["pair"], q["tiles"], q["units"]) == (192, 1, 150, 150), q


@pytest.mark.parametrize("sms,pairs", [(152, 76), (152, 0), (132, 66), (148, 0)])
def test_tail_split_plan_invariants(sms, pairs):
    """Over many shapes: units = whole tiles + 2 x split tiles; a split happens
    only after whole rounds, on a last round at most half full, and each
    split tile's two parts are 128 columns and the rest of the tile."""
    import random
    rng = random.Random(sms + pairs)
    seen = 0
    for _ in range(400):
        M = rng.choice([rng.randint(1, 512), rng.randint(17, 9000)])
        N = 8 * rng.randint(1, 1200)
        K = 8 * rng.randint(1, 1200)
        p = tg.tmagemm_gemm_plan(M, N, K, sms, 1, pairs)
        t = tg.tmagemm_gemm_tail_plan(M, N, K, sms, pairs)
        assert p["units"] == t["full_units"] + 2 * t["split_tiles"], (M, N, K, p, t)
        if t["split_tiles"] == 0:
            assert t["narrow_cols"] == 0
            continue
        seen += 1
        slots = p["grid"] // (2 if p["pair"] else 1) if t["full_units"] else None
        assert p["cluster_k"] == 0 and p["splits"] == 1
        assert p["BN"] in (256, 224, 192) and t["narrow_cols"] == 128
        assert t["full_units"] + t["split_tiles"] == p["tiles"]
        s = pairs if p["pair"] else sms
        assert t["full_units"] % s == 0 and 2 * t["split_tiles"] <= s
        assert p["grid"] == min(p["units"], s) * (2 if p["pair"] else 1)
        if slots is not None:
            assert slots == s
    assert seen > 10


def test_cta_pair_override():
    try:
        assert tg.tmagemm_set_cta_pair(1) == tg.TMAGEMM_OK
        assert tg.tmagemm_gemm_plan(4096, 4096, 4096, 152, 1, 76)["pair"] == 0
        assert tg.tmagemm_set_cta_pair(2) == tg.TMAGEMM_OK
        assert tg.tmagemm_gemm_plan(256, 256, 256, 152, 1, 76)["pair"] == 1
        assert tg.tmagemm_set_cta_pair(3) == tg.TMAGEMM_ERR_INVALID
    finally:
        assert tg.tmagemm_set_cta_pair(0) == tg.TMAGEMM_OK


def test_pdl_switch():
    try:
        assert tg.tmagemm_set_pdl(0) == tg.TMAGEMM_OK
        assert tg.tmagemm_set_pdl(2) == tg.TMAGEMM_ERR_INVALID
        assert tg.tmagemm_set_pdl(-1) == tg.TMAGEMM_ERR_INVALID
    finally:
        assert tg.tmagemm_set_pdl(1) == tg.TMAGEMM_OK


def test_small_m_route_switch():
    try:
        assert tg.tmagemm_set_small_m_route(1) == tg.TMAGEMM_OK
        assert tg.tmagemm_set_small_m_route(2) == tg.TMAGEMM_OK
        assert tg.tmagemm_set_small_m_route(3) == tg.TMAGEMM_OK
        assert tg.tmagemm_set_small_m_route(4) == tg.TMAGEMM_ERR_INVALID
        assert tg.tmagemm_set_small_m_route(-1) == tg.TMAGEMM_ERR_INVALID
    finally:
        assert tg.tmagemm_set_small_m_route(0) == tg.TMAGEMM_OK


def test_cluster_split_plan():
    """Few tiles and a long K: gemm_f16's plan splits K over 4-CTA clusters
    (32 tiles x 4 = 128 CTAs <= 152); the headline shapes keep the tile plan."""
    # CTA pairs available: 16 pair tiles of 256 x 256, 4 pairs each (clusters of 8)
    p = tg.tmagemm_gemm_plan(1024, 1024, 16384, 152, 1, 76)
    assert (p["cluster_k"], p["splits"], p["grid"], p["BN"], p["pair"]) == (4, 4, 128, 256, 1)
    assert p["kb_per_unit"] == 64 and p["units"] == 64
    # without pairs: 32 single-CTA tiles x 4
    p = tg.tmagemm_gemm_plan(1024, 1024, 16384, 152, 1, 0)
    assert (p["cluster_k"], p["splits"], p["grid"], p["BN"], p["pair"]) == (4, 4, 128, 256, 0)
    assert p["kb_per_unit"] == 64 and p["units"] == 128
    for shape in [(4096, 4096, 4096), (8192, 8192, 8192), (4000, 3000, 4160), (256, 256, 256)]:
        assert tg.tmagemm_gemm_plan(*shape, 152, 1, 76)["cluster_k"] == 0, shape
    # explicit split-K requests never use it
    assert tg.tmagemm_gemm_plan(1024, 1024, 16384, 152, 0, 76)["cluster_k"] == 0


def test_group_m_choice():
    """Row order when A, B and D fit in L2 together; otherwise the GROUP_M that
    minimises the A and B panels a round of resident tiles touches."""
    assert tg.tmagemm_gemm_plan(4096, 4096, 4096, 152, 1, 76)["group_m"] == 1
    assert tg.tmagemm_gemm_plan(4000, 3000, 4160, 152, 1, 76)["group_m"] == 1
    assert tg.tmagemm_gemm_plan(8192, 8192, 8192, 152, 1, 76)["group_m"] == 8   # sqrt(76)
    try:
        assert tg.tmagemm_set_group_m(3) == tg.TMAGEMM_OK
        assert tg.tmagemm_gemm_plan(4096, 4096, 4096, 152, 1, 76)["group_m"] == 3
        assert tg.tmagemm_set_group_m(65) == tg.TMAGEMM_ERR_INVALID
    finally:
        assert tg.tmagemm_set_group_m(0) == tg.TMAGEMM_OK


def test_cluster_split_override():
    try:
        assert tg.tmagemm_set_cluster_split(1) == tg.TMAGEMM_OK
        assert tg.tmagemm_gemm_plan(1024, 1024, 16384, 152, 1, 76)["cluster_k"] == 0
        assert tg.tmagemm_set_cluster_split(8) == tg.TMAGEMM_OK
        p = tg.tmagemm_gemm_plan(512, 1000, 4160, 152, 1, 76)   # 16 tiles x 8 CTAs
        assert (p["cluster_k"], p["splits"], p["grid"], p["kb_per_unit"], p["pair"]) == (8, 8, 128, 9, 0)
        # 32 tiles x 8 would not fit one wave: the forced size does not apply
        assert tg.tmagemm_gemm_plan(1024, 1024, 16384, 152, 1, 76)["cluster_k"] != 8
        assert tg.tmagemm_set_cluster_split(2) == tg.TMAGEMM_OK
        assert tg.tmagemm_gemm_plan(1024, 1024, 16384, 152, 1, 76)["cluster_k"] == 2
        for bad in (3, 5, 16, -1):
            assert tg.tmagemm_set_cluster_split(bad) == tg.TMAGEMM_ERR_INVALID
    finally:
        assert tg.tmagemm_set_cluster_split(0) == tg.TMAGEMM_OK


def test_narrow_cluster_split_plans():
    """A few rows against a wide weight matrix: the narrower cluster-split
    tiles put more CTAs on the weight stream (14336 columns: 75 tiles of 192
    x 2 = 150 CTAs instead of 56 tiles of 256 x 2 = 112)."""
    p = tg.tmagemm_gemm_plan(32, 14336, 4096, 152, 1, 76)
    assert (p["cluster_k"], p["BN"], p["pair"], p["tiles"], p["grid"]) == (2, 192, 0, 75, 150)
    try:
        assert tg.tmagemm_set_tile_n(128) == tg.TMAGEMM_OK
        assert tg.tmagemm_set_cluster_split(4) == tg.TMAGEMM_OK
        p = tg.tmagemm_gemm_plan(32, 4096, 14336, 152, 1, 76)
        assert (p["cluster_k"], p["BN"], p["tiles"], p["grid"], p["kb_per_unit"]) == (4, 128, 32, 128, 56)
        # 128 only exists for cluster splits: a plain plan keeps its width
        assert tg.tmagemm_set_cluster_split(1) == tg.TMAGEMM_OK
        assert tg.tmagemm_gemm_plan(4096, 4096, 4096, 152)["BN"] != 128
    finally:
        assert tg.tmagemm_set_cluster_split(0) == tg.TMAGEMM_OK
        assert tg.tmagemm_set_tile_n(0) == tg.TMAGEMM_OK


def test_device_plan_needs_a_device():
    """num_sms == 0 asks for the current device's plan: an error without one."""
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a CUDA device is present")
    with pytest.raises(tg.TmaGemmError):
        tg.tmagemm_gemm_plan(32, 4096, 14336, 0)


def test_tile_width_override():
    try:
        assert tg.tmagemm_set_tile_n(256) == tg.TMAGEMM_OK
        assert tg.tmagemm_gemm_plan(4096, 4096, 4096, 152)["BN"] == 256
        assert tg.tmagemm_set_tile_n(192) == tg.TMAGEMM_OK
        assert tg.tmagemm_gemm_plan(4096, 4096, 4096, 152)["BN"] == 192
        assert tg.tmagemm_set_tile_n(100) == tg.TMAGEMM_ERR_INVALID
        assert tg.tmagemm_set_tile_n(64) == tg.TMAGEMM_ERR_INVALID
    finally:
        assert tg.tmagemm_set_tile_n(0) == tg.TMAGEMM_OK
    assert tg.tmagemm_gemm_plan(4096, 4096, 4096, 152)["BN"] == 224


@pytest.mark.parametrize("M,N,K,splits", [(1024, 1024, 16384, 0), (256, 256, 256, 8),
                                          (129, 264, 1000, 5), (4000, 3000, 4160, 2),
                                          (300, 520, 8, 3), (1000, 1000, 4160, 3)])
def test_splitk_plan_has_no_empty_part(M, N, K, splits):
    p = tg.tmagemm_gemm_plan(M, N, K, 152, splits)
    kb = -(-K // p["BK"])
    assert 1 <= p["splits"] <= kb
    assert (p["splits"] - 1) * p["kb_per_unit"] < kb <= p["splits"] * p["kb_per_unit"]
    assert p["units"] == p["tiles"] * p["splits"]
    assert p["grid"] == min(p["units"], 152)
    if splits > 1:
        assert p["splits"] == min(splits, -(-kb // p["kb_per_unit"]))


def test_splitk_auto_plan_fills_the_gpu():
    p = tg.tmagemm_gemm_plan(1024, 1024, 16384, 152, 0)
    assert p["splits"] > 1 and p["units"] <= 152 and p["units"] > 152 // 2
    assert tg.tmagemm_gemm_plan(4096, 4096, 4096, 152, 0)["splits"] == 1


def test_persistent_schedule_visits_every_tile_once():
    p = tg.tmagemm_gemm_plan(4000, 3000, 4160, 152)
    grid_m, grid_n = -(-4000 // p["BM"]), -(-3000 // p["BN"])
    visits = {}
    for cta in range(p["grid"]):
        for t in range(cta, p["tiles"], p["grid"]):
            mn = tg.tmagemm_tile_coord(t, grid_m, grid_n, 8)
            visits[mn] = visits.get(mn, 0) + 1
    assert len(visits) == grid_m * grid_n and set(visits.values()) == {1}


def test_no_gpu_returns_cuda_error_not_crash():
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    p = 1 << 20
    assert tg.gemm_f16(256, 256, 256, p, p, p, None) == tg.TMAGEMM_ERR_CUDA
