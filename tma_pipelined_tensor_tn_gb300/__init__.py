"""FP16 TN GEMM (D = A @ B.T) and M=1 GEMV for GB300 (sm_103a).

The compute path is the CUDA library ``libtmagemm.so`` built from ``csrc/``;
this package only marshals arguments to its C ABI (``include/tmagemm.h``).
"""
from ._binding import (  # noqa: F401
    CHECKED,
    LIB_PATH,
    checked_unit_counts,
    SIGNATURES,
    TMAGEMM_ERR_ALIGN,
    TMAGEMM_ERR_CHECK,
    TMAGEMM_ERR_CUDA,
    TMAGEMM_ERR_INVALID,
    TMAGEMM_ERR_TIMEOUT,
    TMAGEMM_ERR_UNSUPPORTED,
    TMAGEMM_ERR_SCRATCH_LIMIT,
    TMAGEMM_ERR_WORKSPACE,
    TMAGEMM_OK,
    TmaGemmError,
    TmagemmOptions,
    check,
    gemm,
    gemm_bf16,
    gemm_f16,
    gemm_f16_ex,
    gemm_bf16_ex,
    gemm_f16_grouped,
    gemm_f16_small_m,
    gemm_f16_small_m_workspace_size,
    gemm_f16_splitk,
    gemm_f16_splitk_noalloc,
    gemm_f16_splitk_workspace_size,
    gemm_grouped,
    gemm_small_m,
    gemm_splitk,
    gemv,
    gemv_f16,
    gemv_bf16,
    lib,
    options,
    strerror,
    tmagemm_check,
    tmagemm_gemm_plan,
    tmagemm_gemm_tail_plan,
    tmagemm_last_error_detail,
    tmagemm_ring_position,
    tmagemm_selftest_wait_timeout,
    tmagemm_set_grouped_transposed,
    tmagemm_grouped_plan,
    tmagemm_set_cluster_split,
    tmagemm_set_cta_pair,
    tmagemm_set_group_m,
    tmagemm_set_pdl,
    tmagemm_set_small_m_route,
    tmagemm_set_tail_split,
    tmagemm_set_tile_n,
    tmagemm_tile_coord,
    tmagemm_version,
)


def build(force: bool = False) -> str:
    """Compile libtmagemm.so in-tree (nvcc, sm_103a); with TMAGEMM_CHECKED=1 in
    the environment, the checked build libtmagemm_checked.so instead."""
    from ._build import build as _b
    from ._binding import CHECKED
    return _b(force=force, checked=CHECKED)
