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


def compare(gpu, ref, what=""):
    """Assert the tolerance rule and the internal 1-ulp gate; return stats."""
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
    inner = f16_ulp(r) + INNER_SLACK
    worst = np.max(err - inner, initial=-1.0)
    assert worst <= 0, f"{what}: an element exceeds 1 fp16 ulp + {INNER_SLACK} (by {worst})"
    return {"max_abs": float(err.max(initial=0.0)), "max_ulp": float(ulps.max(initial=0.0)),
            "frac_ne": float(np.mean(err > 0)) if err.size else 0.0}


def assert_bitexact(gpu, ref, what=""):
    g = np.ascontiguousarray(np.asarray(gpu, dtype=np.float16)).view(np.uint16)
    r = np.ascontiguousarray(np.asarray(ref, dtype=np.float16)).view(np.uint16)
    assert g.shape == r.shape
    ne = np.nonzero(g != r)
    assert ne[0].size == 0, (f"{what}: {ne[0].size} elements differ; first at "
                             f"{tuple(int(x[0]) for x in ne)}")
