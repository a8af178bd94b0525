"""CPU oracle for dense C = A x B, accumulated in double precision.

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package. The CUDA library
never calls it and it never calls the CUDA library; the two share no code.

The arithmetic lives in ``gemm_oracle.c`` (the plain definition
C[i][j] = sum_k A[i][k] B[k][j] of "Tiled Matrix Multiplication in CUDA",
section 1, and "Tiled GEMM: Matrix Multiplication in CUDA", section 1, over
row-major matrices with leading dimensions as in section 7.1 of the latter).
This module only marshals arrays: it converts the fp32 or bf16 inputs to
float64 (exact) and passes pointers and leading dimensions.

Every function returns ``(C, absAB)`` as float64 numpy arrays, where
``absAB[i][j] = sum_k |A[i][k]| |B[k][j]|`` is the scale the parity
tolerances are written in.
"""
from __future__ import annotations

import ctypes
import os
from typing import Iterable, Tuple

import numpy as np

from . import build as _build

__all__ = ["Oracle", "default", "gemm", "gemm_rows", "gemm_ex", "set_threads",
           "max_threads", "to_float64"]

_c_double_p = ctypes.POINTER(ctypes.c_double)
_c_long_p = ctypes.POINTER(ctypes.c_long)


def to_float64(x) -> np.ndarray:
    """Exact conversion of a 2-D fp32/bf16/f64 torch tensor or array to float64.

    Keeps the row stride of a view whose columns are contiguous (so padded
    leading dimensions survive); otherwise returns a packed copy.
    """
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach()
            if x.device.type != "cpu":
                raise ValueError("the oracle takes host tensors only")
            x = x.to(torch.float64).numpy()
    except ImportError:  # numpy-only use
        pass
    x = np.asarray(x)
    if x.dtype != np.float64:
        x = x.astype(np.float64)
    if x.ndim != 2:
        raise ValueError("expected a 2-D matrix")
    return x


def _ld(x: np.ndarray) -> Tuple[np.ndarray, int]:
    """Return (base array, leading dimension) for a row-major 2-D view."""
    rows, cols = x.shape
    if cols > 0 and x.strides[1] != 8:
        x = np.ascontiguousarray(x)
    if rows > 1 and (x.strides[0] % 8 != 0 or x.strides[0] < 8 * cols):
        x = np.ascontiguousarray(x)
    ld = x.strides[0] // 8 if rows > 1 else max(cols, 1)
    return x, max(ld, cols, 1)


class Oracle:
    """Handle on one compiled copy of the oracle library."""

    def __init__(self, library_path: str):
        self.path = library_path
        lib = ctypes.CDLL(library_path)
        lib.oracle_gemm.restype = ctypes.c_int
        lib.oracle_gemm.argtypes = [
            ctypes.c_int, ctypes.c_int, ctypes.c_int,
            _c_double_p, ctypes.c_long, _c_double_p, ctypes.c_long,
            _c_double_p, ctypes.c_long, _c_double_p, ctypes.c_long]
        lib.oracle_gemm_rows.restype = ctypes.c_int
        lib.oracle_gemm_rows.argtypes = [
            ctypes.c_int, ctypes.c_int, ctypes.c_int,
            _c_double_p, ctypes.c_long, _c_double_p, ctypes.c_long,
            _c_long_p, ctypes.c_int,
            _c_double_p, ctypes.c_long, _c_double_p, ctypes.c_long]
        lib.oracle_gemm_ex.restype = ctypes.c_int
        lib.oracle_gemm_ex.argtypes = [
            ctypes.c_int, ctypes.c_int, ctypes.c_int,
            _c_double_p, ctypes.c_long, ctypes.c_int,
            _c_double_p, ctypes.c_long, ctypes.c_int,
            ctypes.c_double, ctypes.c_double,
            _c_double_p, ctypes.c_long, _c_double_p,
            _c_double_p, ctypes.c_long, _c_double_p, ctypes.c_long]
        lib.oracle_set_threads.restype = None
        lib.oracle_set_threads.argtypes = [ctypes.c_int]
        lib.oracle_max_threads.restype = ctypes.c_int
        lib.oracle_max_threads.argtypes = []
        self._lib = lib

    @staticmethod
    def _ptr(x: np.ndarray):
        if x.size == 0:
            return ctypes.cast(ctypes.pointer(ctypes.c_double(0.0)), _c_double_p)
        return x.ctypes.data_as(_c_double_p)

    def _operands(self, A, B):
        A = to_float64(A)
        B = to_float64(B)
        M, K = A.shape
        K2, N = B.shape
        if K != K2:
            raise ValueError(f"inner dimensions differ: {A.shape} x {B.shape}")
        A, lda = _ld(A)
        B, ldb = _ld(B)
        return A, lda, B, ldb, M, N, K

    def gemm(self, A, B) -> Tuple[np.ndarray, np.ndarray]:
        """Full product: returns (C, absAB), each M x N float64."""
        A, lda, B, ldb, M, N, K = self._operands(A, B)
        C = np.empty((M, N), dtype=np.float64)
        absAB = np.empty((M, N), dtype=np.float64)
        rc = self._lib.oracle_gemm(M, N, K, self._ptr(A), lda, self._ptr(B), ldb,
                                   self._ptr(C), max(N, 1), self._ptr(absAB), max(N, 1))
        if rc != 0:
            raise ValueError("oracle_gemm rejected its arguments")
        return C, absAB

    def gemm_rows(self, A, B, rows: Iterable[int]) -> Tuple[np.ndarray, np.ndarray]:
        """Rows ``rows`` of the product: returns (C_rows, absAB_rows)."""
        A, lda, B, ldb, M, N, K = self._operands(A, B)
        idx = np.ascontiguousarray(np.asarray(list(rows), dtype=np.int64))
        if idx.ndim != 1:
            raise ValueError("rows must be 1-D")
        n = int(idx.shape[0])
        C = np.empty((n, N), dtype=np.float64)
        absAB = np.empty((n, N), dtype=np.float64)
        idx_p = (idx.ctypes.data_as(_c_long_p) if n else
                 ctypes.cast(ctypes.pointer(ctypes.c_long(0)), _c_long_p))
        rc = self._lib.oracle_gemm_rows(M, N, K, self._ptr(A), lda, self._ptr(B), ldb,
                                        idx_p, n, self._ptr(C), max(N, 1),
                                        self._ptr(absAB), max(N, 1))
        if rc != 0:
            raise ValueError("oracle_gemm_rows rejected its arguments")
        return C, absAB

    def gemm_ex(self, A, B, trans_a=False, trans_b=False, alpha=1.0, beta=0.0, C0=None,
                bias=None) -> Tuple[np.ndarray, np.ndarray]:
        """alpha * op(A) op(B) + beta * C0 + bias; returns (C, scale).

        ``A`` and ``B`` are the STORED matrices: A is K x M when ``trans_a``
        (else M x K), B is N x K when ``trans_b`` (else K x N). ``bias`` has
        one entry per column of C. C0 is not read when ``beta == 0``.
        """
        A = to_float64(A)
        B = to_float64(B)
        M, K = (A.shape[1], A.shape[0]) if trans_a else A.shape
        K2, N = (B.shape[1], B.shape[0]) if trans_b else B.shape
        if K != K2:
            raise ValueError(f"inner dimensions differ: {A.shape} / {B.shape}")
        A, lda = _ld(A)
        B, ldb = _ld(B)
        if beta != 0.0:
            if C0 is None:
                raise ValueError("beta != 0 needs C0")
            C0 = to_float64(C0)
            if C0.shape != (M, N):
                raise ValueError("C0 must be M x N")
            C0, ldc0 = _ld(C0)
            c0_p = self._ptr(C0)
        else:
            ldc0, c0_p = max(N, 1), ctypes.cast(None, _c_double_p)
        if bias is not None:
            bias = np.ascontiguousarray(np.asarray(bias, dtype=np.float64).reshape(-1))
            if bias.shape[0] != N:
                raise ValueError("bias must have N entries")
            bias_p = self._ptr(bias)
        else:
            bias_p = ctypes.cast(None, _c_double_p)
        C = np.empty((M, N), dtype=np.float64)
        S = np.empty((M, N), dtype=np.float64)
        rc = self._lib.oracle_gemm_ex(M, N, K, self._ptr(A), lda, int(bool(trans_a)),
                                      self._ptr(B), ldb, int(bool(trans_b)), float(alpha),
                                      float(beta), c0_p, ldc0, bias_p, self._ptr(C), max(N, 1),
                                      self._ptr(S), max(N, 1))
        if rc != 0:
            raise ValueError("oracle_gemm_ex rejected its arguments")
        return C, S

    def set_threads(self, n: int) -> None:
        self._lib.oracle_set_threads(int(n))

    def max_threads(self) -> int:
        return int(self._lib.oracle_max_threads())


_default = None


def default() -> Oracle:
    """The oracle built from ``gemm_oracle.c`` (compiled on first use)."""
    global _default
    if _default is None:
        _default = Oracle(_build.ensure_built())
    return _default


def gemm(A, B):
    return default().gemm(A, B)


def gemm_rows(A, B, rows):
    return default().gemm_rows(A, B, rows)


def gemm_ex(A, B, **kw):
    return default().gemm_ex(A, B, **kw)


def set_threads(n: int) -> None:
    default().set_threads(n)


def max_threads() -> int:
    return default().max_threads()
