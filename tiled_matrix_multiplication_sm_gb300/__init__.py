"""GB300-native tiled dense matrix multiplication, C = A x B.

The compute lives in ``libtgemm.so`` (CUDA for sm_103a, built from ``csrc/``
by :mod:`.build`); this package is its Python binding. See :mod:`.binding`
for the calls.
"""
from .binding import (  # noqa: F401
    TGEMM_TF32, TGEMM_BF16, TGEMM_TF32X3, TgemmError, load, library_path, gemm_f32, gemm_tc,
    gemm_f32_raw, gemm_tc_raw, device_status, status_string, matmul,
)

__all__ = ["TGEMM_TF32", "TGEMM_BF16", "TGEMM_TF32X3", "TgemmError", "load", "library_path",
           "gemm_f32", "gemm_tc", "gemm_f32_raw", "gemm_tc_raw",
           "device_status", "status_string", "matmul"]
