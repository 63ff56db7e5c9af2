"""Comparison helpers for the GPU parity tests (CUDA path vs the CPU oracle)."""
import numpy as np

# Per-element pass rule for floating-point inputs: |gpu - ref| <= ATOL + RTOL * |ref|.
ATOL = 1e-2
RTOL = 2e-3
INNER_SLACK = 2.0 ** -11


def f16_ulp(x: np.ndarray) -> np.ndarray:
    """Spacing of binary16 numbers at |x| (subnormal spacing below 2^-14)."""
    a = np.abs(x.astype(np.float64))
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -14)))
    return 2.0 ** (e - 10)


def inner_slack(k=None):
    """Absolute slack of the internal gate for a K-term tensor-core sum.

    The FP32 accumulator's error is bounded by the number of accumulator
    additions (K/16 MMA steps) times the rounding of each, which scales with
    the magnitude of the partial sums (about sqrt(K) for the zero-mean inputs
    used here): it grows as K^1.5.  2^-11 held for every K <= 4160 measured
    (all seeds and shapes); above K = 4096 it is scaled by (K / 4096)^1.5
    (8192^3: max error 7.3e-4 against a slack of 1.4e-3).  Always far inside
    the pass rule's 1e-2 absolute term."""
    if k is None or k <= 4096:
        return INNER_SLACK
    return INNER_SLACK * (k / 4096.0) ** 1.5


def compare(gpu, ref, what="", k=None):
    """Assert the tolerance rule and the internal 1-ulp gate; return stats.
    `k`: the sum length, for the internal gate's slack (inner_slack)."""
    g = np.asarray(gpu).astype(np.float64)
    r = np.asarray(ref).astype(np.float64)
    assert g.shape == r.shape, (what, g.shape, r.shape)
    assert np.all(np.isfinite(g)), f"{what}: non-finite GPU outputs"
    err = np.abs(g - r)
    bound = ATOL + RTOL * np.abs(r)
    bad = np.nonzero(err > bound)
    assert bad[0].size == 0, (
        f"{what}: {bad[0].size} elements outside |err| <= {ATOL} + {RTOL}|ref|; first at "
        f"{tuple(int(b[0]) for b in bad)} gpu={g[tuple(b[0] for b in bad)]} ref={r[tuple(b[0] for b in bad)]}")
    ulps = err / f16_ulp(r)
    # Internal gate, tighter than the rule above: FP32 accumulation vs FP64 may
    # move the fp16 result by one step where the exact sum sits near a rounding
    # boundary, plus the FP32 rounding error itself (which dominates only for
    # outputs near zero, where the fp16 step is tiny).
    slack = inner_slack(k)
    excess = err - (f16_ulp(r) + slack)
    worst = np.max(excess, initial=-1.0)
    if worst > 0:
        at = np.unravel_index(np.argmax(excess), excess.shape)
        raise AssertionError(
            f"{what}: an element exceeds 1 fp16 ulp + {slack} (by {worst}) at {tuple(map(int, at))}: "
            f"gpu={g[at]} ref={r[at]} err={err[at]}")
    return {"max_abs": float(err.max(initial=0.0)), "max_ulp": float(ulps.max(initial=0.0)),
            "frac_ne": float(np.mean(err > 0)) if err.size else 0.0}


def assert_bitexact(gpu, ref, what=""):
    g = np.ascontiguousarray(np.asarray(gpu, dtype=np.float16)).view(np.uint16)
    r = np.ascontiguousarray(np.asarray(ref, dtype=np.float16)).view(np.uint16)
    assert g.shape == r.shape
    ne = np.nonzero(g != r)
    assert ne[0].size == 0, (f"{what}: {ne[0].size} elements differ; first at "
                             f"{tuple(int(x[0]) for x in ne)}")


# bf16 rule: one rounding to bf16 (8 significant bits) moves a result by up to
# half a step of 2^-7 relative, above the fp16 rule's relative term, so the
# bf16 rule is |err| <= 1e-2 + 8e-3 |ref| (one bf16 step), with the internal
# gate |err| <= 1 bf16 step of ref + 2^-11.
BF16_RTOL = 8e-3


def bf16_bits_value(b):
    """float64 values of bf16 bit patterns (uint16)."""
    with np.errstate(invalid="ignore"):
        return (np.asarray(b, dtype=np.uint32) << 16).view(np.float32).astype(np.float64)


def bf16_step(v):
    a = np.abs(v)
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -126)))
    return 2.0 ** (e - 7)


def compare_bf16(gpu_bits, ref_bits, what=""):
    """The bf16 rule on bit patterns (uint16) of the GPU result and the oracle's."""
    g, r = bf16_bits_value(gpu_bits), bf16_bits_value(ref_bits)
    assert g.shape == r.shape, (what, g.shape, r.shape)
    assert np.all(np.isfinite(g)), what
    err = np.abs(g - r)
    assert np.all(err <= ATOL + BF16_RTOL * np.abs(r)), (what, float(err.max(initial=0.0)))
    assert np.all(err <= bf16_step(r) + INNER_SLACK), (
        what, float((err - bf16_step(r)).max(initial=0.0)))
