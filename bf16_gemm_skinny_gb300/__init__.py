"""Column-major FP16 GEMM and BF16 decode GEMV / prefill GEMM for GB300 (sm_103a).

The compute lives in a C-ABI shared library built from ``csrc/`` (hand-written
tcgen05/TMA and SIMT kernels); this package holds its thin ctypes binding
(``_native``), the build step (``build``) and the seeded input generators
(``inputs``).  Importing the package does not load the library: the first call
of a binding function does, and it raises if the library is missing.
"""
from ._native import (  # noqa: F401
    BIAS_COLUMN,
    BIAS_NONE,
    BIAS_ROW,
    COL_MAJOR,
    FP8_E4M3,
    FP8_E5M2,
    OUT_BF16,
    OUT_F32,
    ROW_MAJOR,
    BskError,
    decode_attention_bf16,
    gemm_f16,
    gemm_f16_colmajor,
    gemm_f16_colmajor_enqueue,
    gemm_f16_colmajor_noalloc,
    gemm_f16_enqueue,
    gemm_fp8,
    gemm_fp8_enqueue,
    gemv_bf16,
    gemv_bf16_enqueue,
    last_error,
    library_path,
    set_option,
    stream_check,
)
