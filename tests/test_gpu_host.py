"""gemm_host: the product for operands in host memory, with the transfers
overlapped with the multiplication (row panels of A and C), checked against
the CPU oracle through the C ABI on every path."""
import pytest
import torch

import oracle
from tests.parity import (F32_ABS, F32_REL, TC_ABS, TC_REL, assert_bit_exact,
                          assert_within)
from tiled_matrix_multiplication_sm_gb300 import inputs

pytestmark = pytest.mark.gpu

DTYPE = {"f32": torch.float32, "tf32": torch.float32, "bf16": torch.bfloat16,
         "tf32x3": torch.float32}


def host_padded(x, ld, pinned=True, pad=float("nan")):
    rows, cols = x.shape
    store = torch.full((rows, ld), pad, dtype=x.dtype, pin_memory=pinned)
    store[:, :cols] = x
    return store[:, :cols]


@pytest.mark.parametrize("path", ["f32", "tf32", "bf16", "tf32x3"])
@pytest.mark.parametrize("shape", [(1, 1, 1), (7, 9, 3), (300, 520, 200), (1024, 264, 136),
                                   (2100, 300, 64), (513, 1000, 1)])
def test_integer_bit_exact(tgemm, path, shape):
    M, N, K = shape
    g = inputs.generator(M + 7 * N + 13 * K)
    A = inputs.draw(M, K, "int4", g).to(DTYPE[path]).pin_memory()
    B = inputs.draw(K, N, "int4", g).to(DTYPE[path]).pin_memory()
    C = tgemm.matmul(A, B, path)
    assert C.device.type == "cpu"
    assert tgemm.binding.last_kernel().startswith("host_pipeline")
    assert tgemm.device_status() == 0
    C_ref, _ = oracle.gemm(A, B)
    assert_bit_exact(C, C_ref, f"host {path} {shape}")


@pytest.mark.parametrize("path", ["f32", "tf32", "bf16", "tf32x3"])
def test_padded_host_layouts_and_canaries(tgemm, path):
    """Host leading dimensions with NaN padding (never read) and a C whose
    padding columns must stay untouched."""
    M, N, K = 1100, 333, 97
    g = inputs.generator(55)
    A = host_padded(inputs.draw(M, K, "int4", g).to(DTYPE[path]), 101)
    B = host_padded(inputs.draw(K, N, "int4", g).to(DTYPE[path]), 350)
    Cstore = torch.full((M, 341), 4321.0, pin_memory=True)
    C = Cstore[:, :N]
    tgemm.binding.gemm_host(A, B, path, out=C)
    C_ref, _ = oracle.gemm(A, B)
    assert_bit_exact(C, C_ref, f"padded host {path}")
    assert (Cstore[:, N:] == 4321.0).all()


@pytest.mark.parametrize("path", ["f32", "tf32", "bf16", "tf32x3"])
def test_float_tolerance_pageable(tgemm, path):
    M, N, K = 700, 640, 300
    g = inputs.generator(66)
    dist = "normal002" if path == "bf16" else "normal"
    A = inputs.draw(M, K, dist, g).to(DTYPE[path])          # pageable host memory
    B = inputs.draw(K, N, dist, g).to(DTYPE[path])
    C = tgemm.binding.gemm_host(A, B, path)
    C_ref, absAB = oracle.gemm(A, B)
    rel, abs_ = (F32_REL, F32_ABS) if path in ("f32", "tf32x3") else (TC_REL, TC_ABS)
    assert_within(C, C_ref, absAB, rel, abs_, f"pageable {path}")


def test_k_zero_and_empty(tgemm):
    C = tgemm.binding.gemm_host(torch.empty(5, 0), torch.empty(0, 7), "f32")
    assert (C == 0).all()
    C = tgemm.binding.gemm_host(torch.empty(0, 4), torch.ones(4, 7), "f32")
    assert C.shape == (0, 7)


@pytest.mark.parametrize("path", ["f32", "tf32"])
def test_workload_n4096_host_full(tgemm, workload_reference, path):
    """The benchmark's end-to-end calls on its full workload (both paths of
    the step), every output checked against the oracle."""
    A, B, C_ref, absAB = workload_reference("n4096")
    C = tgemm.matmul(A.pin_memory(), B.pin_memory(), path)
    rel, abs_ = (F32_REL, F32_ABS) if path == "f32" else (TC_REL, TC_ABS)
    assert_within(C, C_ref, absAB, rel, abs_, f"n4096 host {path}")


def test_invalid_path_and_misaligned_host_operand(tgemm):
    b = tgemm.binding
    A = torch.ones(4, 4, dtype=torch.bfloat16)
    B = torch.ones(4, 4, dtype=torch.bfloat16)
    C = torch.empty(4, 4)
    assert b.load().gemm_host(4, 4, 4, A.data_ptr(), 4, B.data_ptr(), 4, C.data_ptr(), 4, 7,
                              0) == b.TGEMM_ERR_INVALID_ARG
    assert b.load().gemm_host(4, 4, 4, A.data_ptr() + 1, 4, B.data_ptr(), 4, C.data_ptr(), 4, 2,
                              0) == b.TGEMM_ERR_INVALID_ARG


def test_calls_in_flight_together_on_two_streams(tgemm):
    """Six gemm_host calls enqueued on two streams before either is
    synchronised (the result copy streams are taken in turn): every result is
    the oracle's, bit for bit."""
    s = [torch.cuda.Stream(), torch.cuda.Stream()]
    jobs = []
    for i, path in enumerate(["f32", "tf32", "bf16", "tf32x3", "f32", "tf32"]):
        M, N, K = 2100 + 64 * i, 264 + 8 * i, 136
        g = inputs.generator(900 + i)
        A = inputs.draw(M, K, "int4", g).to(DTYPE[path]).pin_memory()
        B = inputs.draw(K, N, "int4", g).to(DTYPE[path]).pin_memory()
        C = tgemm.binding.gemm_host(A, B, path, stream=s[i % 2], synchronize=False)
        jobs.append((A, B, C, path))
    for st in s:
        st.synchronize()
    assert tgemm.device_status() == 0
    for A, B, C, path in jobs:
        C_ref, _ = oracle.gemm(A, B)
        assert_bit_exact(C, C_ref, f"async host {path} {tuple(A.shape)}")


@pytest.mark.parametrize("path,M,panels", [("f32", 512, 1), ("f32", 1024, 3), ("f32", 1300, 3),
                                           ("f32", 2048, 4), ("f32", 2333, 4), ("tf32", 1024, 2),
                                           ("tf32", 2333, 4), ("bf16", 2048, 4)])
def test_row_panels(tgemm, path, M, panels):
    """The row-panel schedule: FP32 (compute-bound) takes a 256-row first
    panel, a 256-511-row last panel and one or two panels between; the
    tensor paths (bound by the CPU-GPU link) take 2 or 4 equal panels. Every
    boundary row and every panel's first and last rows come out bit-exact."""
    N, K = 136, 72
    g = inputs.generator(M + N + K)
    A = inputs.draw(M, K, "int4", g).to(DTYPE[path]).pin_memory()
    B = inputs.draw(K, N, "int4", g).to(DTYPE[path]).pin_memory()
    C = tgemm.matmul(A, B, path)
    assert tgemm.binding.last_kernel().startswith(f"host_pipeline(panels={panels})"), \
        tgemm.binding.last_kernel()
    assert tgemm.device_status() == 0
    C_ref, _ = oracle.gemm(A, B)
    assert_bit_exact(C, C_ref, f"host panels {path} M={M}")


@pytest.mark.parametrize("M,N,K", [(1100, 777, 150), (2300, 1536, 96)])
def test_fp32_first_panel_in_column_halves(tgemm, M, N, K):
    """On the FP32 path B goes up in two column halves and the first row
    panel is multiplied in the same halves (the left one as soon as it has
    arrived). Padded host layouts; every output bit-exact; C's padding
    columns untouched."""
    g = inputs.generator(M * 7 + N + K)
    A = host_padded(inputs.draw(M, K, "int4", g), K + 3)
    B = host_padded(inputs.draw(K, N, "int4", g), N + 5)
    Cstore = torch.full((M, N + 7), 999.0, pin_memory=True)
    C = Cstore[:, :N]
    tgemm.binding.gemm_host(A, B, "f32", out=C)
    assert tgemm.device_status() == 0
    C_ref, _ = oracle.gemm(A, B)
    assert_bit_exact(C, C_ref, f"host halves {M}x{N}x{K}")
    assert (Cstore[:, N:] == 999.0).all()
