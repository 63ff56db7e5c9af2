"""Runs the library's work-split paths under the checked build
(libtmagemm_checked.so, loaded because TMAGEMM_CHECKED=1 is set by the test
that starts this script) and verifies, after each call, that no self-check
fired and that every work unit completed exactly once.  Prints one JSON line
per case and exits non-zero on the first failure."""
import json
import os
import sys

import torch

assert os.environ.get("TMAGEMM_CHECKED") == "1"
import tma_pipelined_tensor_tn_gb300 as tg  # noqa: E402

tg.build()
assert tg.CHECKED and tg.LIB_PATH.endswith("libtmagemm_checked.so")
dev = torch.device("cuda")


def ceil_div(a, b):
    return -(-a // b)


def rnd(shape, dtype=torch.float16, seed=0):
    g = torch.Generator(device="cuda").manual_seed(seed)
    return (torch.rand(shape, device=dev, generator=g) * 2 - 1).to(dtype)


def verify(name, counts, expected_units=None, ref=None, got=None):
    st = tg.lib().tmagemm_check(None)
    assert st == tg.TMAGEMM_OK, (name, tg.strerror(st), tg.tmagemm_last_error_detail())
    assert all(c <= 1 for c in counts), (name, "a unit ran twice", max(counts))
    done = sum(counts)
    assert all(c == 1 for c in counts[:done]), (name, "units done are not 0..U-1")
    if expected_units is not None:
        exp = expected_units if isinstance(expected_units, (list, tuple)) else [expected_units]
        assert done in exp, (name, "units done", done, "expected", exp)
    if ref is not None:
        err = (got.float() - ref.float()).abs().max().item()
        scale = ref.float().abs().max().item()
        assert err <= 1e-2 + 4e-3 * scale, (name, err)
    print(json.dumps({"case": name, "units": done}), flush=True)


def plain(name, M, N, K, dtype=torch.float16, knobs=()):
    for setter, value in knobs:
        assert setter(value) == tg.TMAGEMM_OK
    try:
        p = tg.tmagemm_gemm_plan(M, N, K, 0)
        a, b = rnd((M, K), dtype, 1), rnd((N, K), dtype, 2)
        d = tg.gemm(a, b)
        counts = tg.checked_unit_counts(min(p["units"] + 64, 65536))
        verify(name, counts, p["units"], torch.matmul(a, b.T), d)
    finally:
        for setter, _ in knobs:
            setter(0)


plain("pairs_4096", 4096, 4096, 4096)
plain("ragged", 4000, 3000, 4160)
plain("bf16_4096", 4096, 4096, 4096, torch.bfloat16)
for bn in (256, 224, 192):
    plain(f"single_{bn}", 1000, 1000, 1000, knobs=((tg.tmagemm_set_cta_pair, 1), (tg.tmagemm_set_tile_n, bn)))
    plain(f"pair_{bn}", 1000, 1000, 1000, knobs=((tg.tmagemm_set_cta_pair, 2), (tg.tmagemm_set_tile_n, bn)))
# Tail split: 80 pair tiles (156 single-CTA tiles) on 76 pairs (152 SMs),
# the last round's 4 tiles in two column parts each.
plain("tail_split_pairs", 5070, 984, 520, knobs=((tg.tmagemm_set_cta_pair, 2), (tg.tmagemm_set_tile_n, 256)))
plain("tail_split_single_224", 4942, 856, 520, knobs=((tg.tmagemm_set_cta_pair, 1), (tg.tmagemm_set_tile_n, 224)))
plain("tail_split_8192", 8192, 8192, 512)
plain("cluster_auto", 1024, 1024, 16384)
for ck in (2, 4, 8):
    plain(f"cluster_{ck}", 512, 1000, 4160, knobs=((tg.tmagemm_set_cluster_split, ck),))
plain("decode_32x4096x14336", 32, 4096, 14336)
plain("decode_48x4096x14336", 48, 4096, 14336)
plain("decode_64x14336x4096", 64, 14336, 4096)
plain("group_m_8", 8192, 8192, 1024)

# Split-K with a caller workspace: units are tiles x parts.
M, N, K, S = 1000, 1000, 4160, 3
p = tg.tmagemm_gemm_plan(M, N, K, 0, S)
a, b = rnd((M, K), seed=3), rnd((N, K), seed=4)
d = tg.gemm_splitk(a, b, splits=S)
verify("splitk_3", tg.checked_unit_counts(p["units"] + 64), p["units"], torch.matmul(a, b.T), d)

# Grouped: the groups' tiles, numbered one after the other.
counts_g = [1697, 2233, 321, 376, 105, 1822, 706, 932]
Ng, Kg = 4096, 2048
A = rnd((sum(counts_g), Kg), seed=5)
B = rnd((len(counts_g), Ng, Kg), seed=6)
offsets = [0]
for c in counts_g:
    offsets.append(offsets[-1] + c)
D = tg.gemm_grouped(A, B, offsets)
ref = torch.cat([torch.matmul(A[offsets[g]:offsets[g + 1]], B[g].T) for g in range(len(counts_g))])
exp = [sum(ceil_div(c, tm) for c in counts_g) * ceil_div(Ng, bn)
       for tm in (128, 256) for bn in (256, 224, 192)]


def transposed_units(counts, N, tile_m, maxw):
    """Units of the transposed grouped schedule: weight blocks x row blocks."""
    return ceil_div(N, tile_m) * sum(ceil_div(ceil_div(c, 16), maxw // 16) for c in counts if c)


exp_t = [transposed_units(counts_g, Ng, tm, w) for tm in (128, 256) for w in range(128, 257, 16)]
verify("grouped", tg.checked_unit_counts(4000), exp + exp_t, ref, D)
# Both formulations forced, single CTAs and pairs, with empty and 1-row groups.
counts_t = [0, 1, 129, 0, 16, 17, 700]
offs_t = [0]
for c in counts_t:
    offs_t.append(offs_t[-1] + c)
A_t = rnd((offs_t[-1], 520), seed=15)
B_t = rnd((len(counts_t), 1000, 520), seed=16)
ref_t = torch.cat([torch.matmul(A_t[offs_t[g]:offs_t[g + 1]], B_t[g].T) for g in range(len(counts_t))])
for mode in (1, 2):
    for pair in (1, 2):
        assert tg.tmagemm_set_grouped_transposed(mode) == tg.TMAGEMM_OK
        assert tg.tmagemm_set_cta_pair(pair) == tg.TMAGEMM_OK
        try:
            D_t = tg.gemm_grouped(A_t, B_t, offs_t)
            counts = tg.checked_unit_counts(4000)
        finally:
            tg.tmagemm_set_grouped_transposed(0)
            tg.tmagemm_set_cta_pair(0)
        tm = 256 if pair == 2 else 128
        if mode == 2:
            units = [transposed_units(counts_t, 1000, tm, w) for w in range(128, 257, 16)]
        else:
            units = [sum(ceil_div(c, tm) for c in counts_t) * ceil_div(1000, bn) for bn in (256, 224, 192)]
        verify(f"grouped_mode{mode}_pair{pair}", counts, units, ref_t, D_t)

# Swap-AB small-M (route 1): tile kernel units with FP32 partials.
assert tg.tmagemm_set_small_m_route(1) == tg.TMAGEMM_OK
try:
    X, W = rnd((24, 14336), seed=7), rnd((4096, 14336), seed=8)
    Y = tg.gemm_small_m(X, W)
    verify("swap_ab", tg.checked_unit_counts(4096), None, torch.matmul(X, W.T), Y)
finally:
    tg.tmagemm_set_small_m_route(0)
# Register-fragment small-M kernel (route 2: wherever it applies): one unit
# per CTA, clusters of S CTAs over 64-row groups (S = 8 at N = 4096, 2 at
# N = 14336, 1 at N = 28672 on 152 SMs).
sms = torch.cuda.get_device_properties(0).multi_processor_count
assert tg.tmagemm_set_small_m_route(2) == tg.TMAGEMM_OK
try:
    for Mx, Nw, Kw, dt in ((8, 4096, 14336, torch.float16), (16, 14336, 4096, torch.float16),
                           (8, 4096, 14336, torch.bfloat16), (12, 28672, 1024, torch.float16)):
        X, W = rnd((Mx, Kw), dt, 9), rnd((Nw, Kw), dt, 10)
        Y = tg.gemm(X, W)
        groups = ceil_div(Nw, 64)
        S = next((s for s in (8, 4, 2) if groups * s <= 4 * sms), 1)
        verify(f"fragments_{Mx}x{Nw}x{Kw}_{dt}", tg.checked_unit_counts(groups * S + 64),
               groups * S, torch.matmul(X, W.T), Y)
finally:
    tg.tmagemm_set_small_m_route(0)

# SM-load-fed tcgen05 small-M kernel (route 3): 128-row CTAs, 8 K slices.
assert tg.tmagemm_set_small_m_route(3) == tg.TMAGEMM_OK
try:
    X, W = rnd((40, 14336), seed=11), rnd((4096, 14336), seed=12)
    Y = tg.gemm_small_m(X, W)
    verify("lsu_40", tg.checked_unit_counts(256 + 64), 32 * 8, torch.matmul(X, W.T), Y)
finally:
    tg.tmagemm_set_small_m_route(0)

# GEMV: one unit per output row.
x, W = rnd((14336,), seed=13), rnd((4096, 14336), seed=14)
y = tg.gemv(x, W)
verify("gemv", tg.checked_unit_counts(4096 + 64), 4096, torch.matmul(W, x), y)
print("CHECKED OK", flush=True)
