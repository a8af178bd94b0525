"""The C ABI of libtgemm.so, checked on the host (no compute calls, no GPU).

The library must load, export every entry point that include/tgemm.h
declares, and reject invalid arguments before it touches the CUDA runtime.
"""
import ctypes
import os
import re

import pytest
import torch

import tiled_matrix_multiplication_sm_gb300 as tg
from tiled_matrix_multiplication_sm_gb300 import binding

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "tgemm.h")


def declared_symbols():
    with open(HEADER) as f:
        text = f.read()
    return sorted(set(re.findall(r"^TGEMM_API\s+[\w\s\*]*?\b(\w+)\s*\(", text, re.M)))


@pytest.fixture(scope="module")
def lib():
    path = tg.library_path()
    if not os.path.exists(path):
        from tiled_matrix_multiplication_sm_gb300 import build
        build.build()
    return tg.load()


def test_header_declares_the_boundary():
    names = declared_symbols()
    for required in ["gemm_f32", "gemm_tc", "gemm_status_string", "gemm_device_status"]:
        assert required in names
    assert len(names) == 19


def test_library_exports_every_declared_symbol(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), name
    assert set(declared_symbols()) == set(binding._SIGNATURES)


def test_status_strings(lib):
    for code in range(6):
        s = tg.status_string(code)
        assert s and s != "unknown tgemm status"
    assert tg.status_string(99) == "unknown tgemm status"
    assert tg.status_string(-7) == "unknown tgemm status"


FAKE = 0x10000           # never dereferenced: every call below is rejected first


@pytest.mark.parametrize("args", [
    (-1, 4, 4, FAKE, 4, FAKE, 4, FAKE, 4),        # negative M
    (4, -1, 4, FAKE, 4, FAKE, 4, FAKE, 4),        # negative N
    (4, 4, -1, FAKE, 4, FAKE, 4, FAKE, 4),        # negative K
    (4, 4, 8, FAKE, 7, FAKE, 4, FAKE, 4),         # lda < K
    (4, 8, 4, FAKE, 4, FAKE, 7, FAKE, 8),         # ldb < N
    (4, 8, 4, FAKE, 4, FAKE, 8, FAKE, 7),         # ldc < N
    (4, 4, 4, 0, 4, FAKE, 4, FAKE, 4),            # null A
    (4, 4, 4, FAKE, 4, 0, 4, FAKE, 4),            # null B
    (4, 4, 4, FAKE, 4, FAKE, 4, 0, 4),            # null C
    (4, 4, 4, FAKE + 2, 4, FAKE, 4, FAKE, 4),     # A not 4-byte aligned
    (4, 4, 4, FAKE, 4, FAKE, 4, FAKE + 1, 4),     # C not 4-byte aligned
])
def test_f32_invalid_arguments(lib, args):
    assert tg.gemm_f32_raw(*args, 0) == binding.TGEMM_ERR_INVALID_ARG


@pytest.mark.parametrize("args,code", [
    ((4, 4, 4, FAKE, 4, FAKE, 4, FAKE, 4, 4), binding.TGEMM_ERR_INVALID_ARG),     # bad in_type
    ((4, 4, 4, FAKE, 4, FAKE, 4, FAKE, 4, -1), binding.TGEMM_ERR_INVALID_ARG),
    ((4, 4, 4, FAKE, 4, FAKE, 4, FAKE, 4, 0), binding.TGEMM_ERR_INVALID_ARG),
    ((-1, 4, 4, FAKE, 4, FAKE, 4, FAKE, 4, 2), binding.TGEMM_ERR_INVALID_ARG),
    ((4, 4, 8, FAKE, 4, FAKE, 4, FAKE, 4, 2), binding.TGEMM_ERR_INVALID_ARG),     # lda < K
    ((4, 8, 8, FAKE + 1, 8, FAKE, 8, FAKE, 8, 2), binding.TGEMM_ERR_INVALID_ARG), # bf16 A odd byte
    ((4, 8, 8, FAKE, 8, FAKE + 3, 8, FAKE, 8, 2), binding.TGEMM_ERR_INVALID_ARG), # bf16 B odd byte
    ((4, 8, 8, FAKE + 2, 8, FAKE, 8, FAKE, 8, 1), binding.TGEMM_ERR_INVALID_ARG), # tf32 A not 4-B
    ((4, 8, 8, FAKE, 8, FAKE + 6, 8, FAKE, 8, 1), binding.TGEMM_ERR_INVALID_ARG), # tf32 B not 4-B
    ((4, 8, 8, FAKE, 8, FAKE, 8, FAKE + 2, 8, 1), binding.TGEMM_ERR_INVALID_ARG), # C misaligned
])
def test_tc_invalid_arguments(lib, args, code):
    assert tg.gemm_tc_raw(*args, 0) == code


def test_tc_peak_rejects_bad_arguments(lib):
    """Argument checks of the tensor-rate probe come before any device work."""
    import ctypes
    d = ctypes.c_double(0.0)
    ref = ctypes.byref(d)
    bad = binding.TGEMM_ERR_INVALID_ARG
    assert lib.gemm_tc_peak(4, 1, 1000, ref, ref, None) == bad          # unknown in_type
    assert lib.gemm_tc_peak(binding.TGEMM_TF32X3, 1, 1000, ref, ref, None) == bad
    assert lib.gemm_tc_peak(binding.TGEMM_BF16, 2, 1000, ref, ref, None) == bad   # pair not 0/1
    assert lib.gemm_tc_peak(binding.TGEMM_BF16, 1, 0, ref, ref, None) == bad      # no MMAs
    assert lib.gemm_tc_peak(binding.TGEMM_BF16, 1, 10 ** 9, ref, ref, None) == bad
    assert lib.gemm_tc_peak(binding.TGEMM_BF16, 1, 1000, None, ref, None) == bad  # null output


def test_ex_entry_rejects_bad_arguments(lib):
    ok = (4, 4, 4, FAKE, 4, FAKE, 4, FAKE, 4)
    bad = binding.TGEMM_ERR_INVALID_ARG
    assert lib.gemm_ex(*ok, 4, 0, 1.0, 0.0, None, 0) == bad            # unknown path
    assert lib.gemm_ex(*ok, 0, 4, 1.0, 0.0, None, 0) == bad            # unknown flag
    assert lib.gemm_ex(*ok, 0, 0, 1.0, 0.0, FAKE + 2, 0) == bad        # bias not 4-B aligned
    # trans_a: A stored K x M needs lda >= M
    assert lib.gemm_ex(6, 4, 4, FAKE, 5, FAKE, 4, FAKE, 4, 0, 1, 1.0, 0.0, None, 0) == bad
    # trans_b: B stored N x K needs ldb >= K
    assert lib.gemm_ex(4, 4, 6, FAKE, 6, FAKE, 5, FAKE, 4, 0, 2, 1.0, 0.0, None, 0) == bad
    assert lib.gemm_ex(0, 4, 4, 0, 4, 0, 4, 0, 4, 0, 3, 2.0, 1.0, None, 0) == binding.TGEMM_OK


def test_host_entry_rejects_bad_arguments(lib):
    assert lib.gemm_host(4, 4, 4, FAKE, 4, FAKE, 4, FAKE, 4, 7, 0) == binding.TGEMM_ERR_INVALID_ARG
    assert lib.gemm_host(4, 4, 4, FAKE, 3, FAKE, 4, FAKE, 4, 0, 0) == binding.TGEMM_ERR_INVALID_ARG
    assert lib.gemm_host(4, 4, 4, FAKE + 2, 4, FAKE, 4, FAKE, 4, 0, 0) == binding.TGEMM_ERR_INVALID_ARG
    assert lib.gemm_host(0, 4, 4, 0, 4, 0, 4, 0, 4, 0, 0) == binding.TGEMM_OK


def test_scratch_query_rejects_bad_arguments(lib):
    """gemm_scratch_bytes checks its arguments like gemm_ex, before any CUDA
    call, and answers 0 for an empty product."""
    bad = -binding.TGEMM_ERR_INVALID_ARG
    q = lib.gemm_scratch_bytes
    assert q(4, 4, 4, FAKE, 4, FAKE, 4, FAKE, 4, 4, 0) == bad          # unknown path
    assert q(4, 4, 4, FAKE, 4, FAKE, 4, FAKE, 4, 0, 8) == bad          # unknown flag
    assert q(-1, 4, 4, FAKE, 4, FAKE, 4, FAKE, 4, 0, 0) == bad         # negative M
    assert q(4, 4, 8, FAKE, 7, FAKE, 4, FAKE, 4, 1, 0) == bad          # lda < K
    assert q(4, 4, 4, FAKE, 4, FAKE, 4, 0, 4, 2, 0) == bad             # null C
    assert q(4, 8, 8, FAKE + 1, 8, FAKE, 8, FAKE, 8, 2, 0) == bad      # bf16 A odd byte
    assert q(0, 4, 4, 0, 4, 0, 4, 0, 4, 1, 0) == 0                     # nothing to compute
    assert q(4, 0, 4, 0, 4, 0, 4, 0, 4, 3, 3) == 0


@pytest.mark.parametrize("M,N", [(0, 5), (5, 0), (0, 0)])
def test_empty_output_is_noop(lib, M, N):
    """Nothing to compute: OK without any CUDA call (null pointers allowed)."""
    assert tg.gemm_f32_raw(M, N, 3, 0, 3, 0, max(N, 1), 0, max(N, 1), 0) == binding.TGEMM_OK
    assert tg.gemm_tc_raw(M, N, 8, 0, 8, 0, 8, 0, 8, 2, 0) == binding.TGEMM_OK


def test_setters_validate(lib):
    assert binding.set_wait_limit_ns(0) == binding.TGEMM_ERR_INVALID_ARG
    assert binding.set_wait_limit_ns(-5) == binding.TGEMM_ERR_INVALID_ARG
    assert binding.set_wait_limit_ns(2_000_000_000) == binding.TGEMM_OK
    n = lib.gemm_f32_kernel_count()
    assert n >= 2
    assert binding.set_f32_kernel(n) == binding.TGEMM_ERR_INVALID_ARG
    assert binding.set_f32_kernel(-2) == binding.TGEMM_ERR_INVALID_ARG
    assert binding.set_f32_kernel(-1) == binding.TGEMM_OK
    assert binding.set_tc_kernel(5) == binding.TGEMM_ERR_INVALID_ARG
    assert binding.set_tc_kernel(-2) == binding.TGEMM_ERR_INVALID_ARG
    assert binding.set_tc_kernel(-1) == binding.TGEMM_OK
    assert binding.set_tc_streamk(-65) == binding.TGEMM_ERR_INVALID_ARG
    assert binding.set_tc_streamk(40) == binding.TGEMM_OK
    assert binding.set_tc_streamk(-1) == binding.TGEMM_OK
    assert binding.set_tc_a_loader(2) == binding.TGEMM_ERR_INVALID_ARG
    assert binding.set_tc_a_loader(-2) == binding.TGEMM_ERR_INVALID_ARG
    assert binding.set_tc_a_loader(-1) == binding.TGEMM_OK
    assert lib.gemm_f32_kernel_name(n) == b""
    names = binding.f32_kernel_names()
    assert len(set(names)) == n and all(names)


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-GPU failure path")
def test_valid_call_without_gpu_fails_loudly(lib):
    """A valid call on a host with no usable GPU returns an error, never falls back."""
    st = tg.gemm_f32_raw(4, 4, 4, FAKE, 4, FAKE, 4, FAKE, 4, 0)
    assert st in (binding.TGEMM_ERR_CUDA, binding.TGEMM_ERR_UNSUPPORTED)
    with pytest.raises((ValueError, RuntimeError)):
        tg.gemm_f32(torch.ones(4, 4), torch.ones(4, 4))


def test_binding_rejects_bad_tensors(lib):
    with pytest.raises(ValueError):
        tg.gemm_f32(torch.ones(4), torch.ones(4, 4))
    with pytest.raises(ValueError):
        tg.gemm_f32(torch.ones(4, 4), torch.ones(4, 4))   # host tensors need matmul()
