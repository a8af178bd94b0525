"""Parity of the FP32 CUDA-core path (gemm_f32) with the CPU oracle.

Tolerance (FP32 path): |C - C_ref| <= 1e-5 * absAB + 1e-6 element by element,
absAB = sum_k |A[i][k]| |B[k][j]|; integer-valued inputs whose partial sums
stay below 2^24 must match bit for bit. All calls go through the C ABI.
"""
import numpy as np
import pytest
import torch

import oracle
from tests.parity import F32_ABS, F32_REL, assert_bit_exact, assert_within
from tiled_matrix_multiplication_sm_gb300 import inputs

pytestmark = pytest.mark.gpu


def run_f32(tg, A, B, out=None):
    C = tg.gemm_f32(A.cuda() if A.device.type == "cpu" else A,
                    B.cuda() if B.device.type == "cpu" else B, out=out)
    assert tg.device_status() == 0
    return C


def padded_cuda(x, ld, pad=float("nan")):
    """Device copy of ``x`` as a view with leading dimension ``ld``; the
    columns past x's width hold ``pad``."""
    rows, cols = x.shape
    store = torch.full((rows, ld), pad, dtype=x.dtype, device="cuda")
    store[:, :cols] = x.cuda()
    return store[:, :cols]


# ---------------------------------------------------------------- workloads

def test_workload_int128_bit_exact(tgemm):
    w = inputs.WORKLOADS["int128"]
    A, B = inputs.operands(w)
    C = run_f32(tgemm, A, B)
    C_ref, _ = oracle.gemm(A, B)
    assert_bit_exact(C, C_ref, "int128")


def test_workload_u1024_full(tgemm):
    w = inputs.WORKLOADS["u1024"]
    A, B = inputs.operands(w)
    C = run_f32(tgemm, A, B)
    C_ref, absAB = oracle.gemm(A, B)
    assert_within(C, C_ref, absAB, F32_REL, F32_ABS, "u1024")


def test_workload_n4096_full(tgemm, workload_reference):
    """Full-size launch, every output checked against the oracle's full
    product (every split-K tail tile and every raster group)."""
    A, B, C_ref, absAB = workload_reference("n4096")
    C = run_f32(tgemm, A, B)
    assert_within(C, C_ref, absAB, F32_REL, F32_ABS, "n4096")


def test_workload_ragged_full(tgemm, workload_reference):
    """3000 x 5001 x 1537 with packed (16-byte-unaligned) leading dimensions,
    every output checked."""
    A, B, C_ref, absAB = workload_reference("ragged")
    C = run_f32(tgemm, A, B)
    # Large and unaligned: both operands are repacked to 16-byte rows first
    # (one launch copies both).
    assert "repack_ab+" in tgemm.binding.last_kernel()
    assert_within(C, C_ref, absAB, F32_REL, F32_ABS, "ragged")


def test_workload_skinny_f32_full(tgemm, workload_reference):
    """16 x 14336 x 4096 (bound by reading B), every output checked."""
    A, B, C_ref, absAB = workload_reference("skinny_f32")
    C = run_f32(tgemm, A, B)
    assert_within(C, C_ref, absAB, F32_REL, F32_ABS, "skinny f32")


def test_repacked_and_four_byte_loaders_agree_with_oracle(tgemm):
    """The same unaligned operands through the 4-byte loaders (forced kernel)
    and through the repack + 16-byte loader route."""
    g = inputs.generator(41)
    A = inputs.draw(300, 257, "int4", g)        # lda = 257, ldb = 301: rows off 16 bytes
    B = inputs.draw(257, 301, "int4", g)
    C_ref, _ = oracle.gemm(A, B)
    C = run_f32(tgemm, A, B)
    assert "repack_ab+" in tgemm.binding.last_kernel()
    assert_bit_exact(C, C_ref, "repacked")
    names = tgemm.binding.f32_kernel_names()
    try:
        assert tgemm.binding.set_f32_kernel(names.index("f32_128x256x32_s3_ffma2_a4_b4")) == 0
        C = run_f32(tgemm, A, B)
        assert "repack" not in tgemm.binding.last_kernel()
        assert_bit_exact(C, C_ref, "4-byte loaders")
    finally:
        tgemm.binding.set_f32_kernel(-1)


def test_ragged_reduced_full(tgemm):
    """The ragged workload's shape class, small enough for a full oracle check."""
    g = inputs.generator(31)
    A = inputs.draw(300, 501, "uniform", g)
    B = inputs.draw(501, 437, "uniform", g)
    C = run_f32(tgemm, A, B)
    C_ref, absAB = oracle.gemm(A, B)
    assert_within(C, C_ref, absAB, F32_REL, F32_ABS, "ragged-small")


# ---------------------------------------------------------------- every kernel

SHAPES = [(1, 1, 1), (1, 37, 1), (37, 1, 5), (7, 9, 3), (64, 64, 16), (65, 63, 17),
          (128, 128, 15), (129, 257, 33), (200, 130, 1), (300, 77, 250), (17, 300, 64)]


def kernel_ids(tg):
    return range(len(tg.binding.f32_kernel_names()))


@pytest.mark.parametrize("shape", SHAPES)
def test_every_kernel_integer_bit_exact(tgemm, shape):
    M, N, K = shape
    g = inputs.generator(M * 1000 + N * 10 + K)
    A = inputs.draw(M, K, "int4", g)
    B = inputs.draw(K, N, "int4", g)
    C_ref, _ = oracle.gemm(A, B)
    names = tgemm.binding.f32_kernel_names()
    # Leading dimensions rounded up to 4 floats (NaN in the padding) so that
    # the 16-byte loaders may read the operands too.
    Ad, Bd = padded_cuda(A, -(-K // 4) * 4), padded_cuda(B, -(-N // 4) * 4)
    try:
        for kid in kernel_ids(tgemm):
            assert tgemm.binding.set_f32_kernel(kid) == 0
            C = run_f32(tgemm, Ad, Bd)
            assert names[kid] in tgemm.binding.last_kernel().split("+")
            assert_bit_exact(C, C_ref, f"{names[kid]} {shape}")
    finally:
        tgemm.binding.set_f32_kernel(-1)


@pytest.mark.parametrize("shape", [(130, 260, 77), (33, 129, 1025)])
def test_every_kernel_float_tolerance(tgemm, shape):
    M, N, K = shape
    g = inputs.generator(sum(shape))
    A = inputs.draw(M, K, "normal", g)
    B = inputs.draw(K, N, "normal", g)
    C_ref, absAB = oracle.gemm(A, B)
    Ad, Bd = padded_cuda(A, -(-K // 4) * 4), padded_cuda(B, -(-N // 4) * 4)
    try:
        for kid in kernel_ids(tgemm):
            assert tgemm.binding.set_f32_kernel(kid) == 0
            assert_within(run_f32(tgemm, Ad, Bd), C_ref, absAB, F32_REL, F32_ABS, f"kernel {kid}")
    finally:
        tgemm.binding.set_f32_kernel(-1)


def test_forced_vector_kernel_rejects_unaligned_operands(tgemm):
    A = torch.ones(8, 5, device="cuda")     # lda = 5: not a multiple of 4
    B = torch.ones(5, 8, device="cuda")
    try:
        assert tgemm.binding.set_f32_kernel(0) == 0     # 16-byte loaders for A and B
        with pytest.raises(tgemm.TgemmError) as e:
            tgemm.gemm_f32(A, B)
        assert e.value.status == 2
    finally:
        tgemm.binding.set_f32_kernel(-1)


def test_integer_bit_exact_larger(tgemm):
    """Partial sums stay below 2^24 (|sum| <= 16 K), so every order is exact."""
    g = inputs.generator(12345)
    A = inputs.draw(257, 1031, "int4", g)
    B = inputs.draw(1031, 263, "int4", g)
    C_ref, _ = oracle.gemm(A, B)
    assert_bit_exact(run_f32(tgemm, A, B), C_ref, "int 257x263x1031")


# ---------------------------------------------------------------- memory safety

def test_padding_never_read_and_canaries_intact(tgemm):
    """NaN in the ld padding of A and B must not reach C; C's padding and the
    guard bands around it must be untouched."""
    M, N, K = 70, 90, 45
    A = padded_cuda(inputs.matrix(M, K, "uniform", seed=1), 52)    # 16-B aligned ld
    B = padded_cuda(inputs.matrix(K, N, "uniform", seed=2), 97)    # unaligned ld
    ldc, guard = 101, 64
    store = torch.full((guard + M * ldc + guard,), 12345.0, device="cuda")
    C = store[guard:guard + M * ldc].view(M, ldc)[:, :N]
    tgemm.gemm_f32(A, B, out=C)
    assert tgemm.device_status() == 0
    C_ref, absAB = oracle.gemm(A.cpu(), B.cpu())
    assert_within(C, C_ref, absAB, F32_REL, F32_ABS, "padded")
    host = store.cpu()
    assert (host[:guard] == 12345.0).all() and (host[guard + M * ldc:] == 12345.0).all()
    assert (host[guard:guard + M * ldc].view(M, ldc)[:, N:] == 12345.0).all()


def test_unaligned_pointers(tgemm):
    """Operands that start 4 bytes past a 16-byte boundary take the 4-byte loaders."""
    M, N, K = 50, 60, 70
    baseA = inputs.matrix(1, M * K + 1, "uniform", seed=3).cuda()
    baseB = inputs.matrix(1, K * N + 1, "uniform", seed=4).cuda()
    A = baseA[0, 1:].view(M, K)
    B = baseB[0, 1:].view(K, N)
    C = run_f32(tgemm, A, B)
    assert "a4_b4" in tgemm.binding.last_kernel()
    C_ref, absAB = oracle.gemm(A.cpu(), B.cpu())
    assert_within(C, C_ref, absAB, F32_REL, F32_ABS, "unaligned")


def test_k_zero_writes_zeros(tgemm):
    C = torch.full((5, 7), 3.0, device="cuda")
    tgemm.gemm_f32(torch.empty(5, 0, device="cuda"), torch.empty(0, 7, device="cuda"), out=C)
    assert tgemm.device_status() == 0
    assert (C == 0).all()


def test_empty_output_untouched(tgemm):
    C = torch.full((0, 7), 3.0, device="cuda")
    tgemm.gemm_f32(torch.ones(0, 4, device="cuda"), torch.ones(4, 7, device="cuda"), out=C)
    assert C.shape == (0, 7)


def test_runs_on_caller_stream(tgemm):
    g = inputs.generator(9)
    A = inputs.draw(256, 256, "int4", g).cuda()
    B = inputs.draw(256, 256, "int4", g).cuda()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        C = tgemm.gemm_f32(A, B)
    s.synchronize()
    C_ref, _ = oracle.gemm(A.cpu(), B.cpu())
    assert_bit_exact(C, C_ref, "stream")


def test_matmul_host_round_trip(tgemm):
    g = inputs.generator(10)
    A = inputs.draw(100, 80, "int4", g).pin_memory()
    B = inputs.draw(80, 60, "int4", g).pin_memory()
    C = tgemm.matmul(A, B, "f32")
    assert C.device.type == "cpu"
    C_ref, _ = oracle.gemm(A, B)
    assert_bit_exact(C, C_ref, "matmul")


@pytest.mark.parametrize("M,tile", [(1, "16x256"), (16, "16x256"), (40, "32x256"), (96, "32x256"),
                                    (128, "128x128"), (192, "32x256"), (256, "128x128")])
def test_few_rows_take_short_tiles(tgemm, M, tile):
    """By shape, products with few rows take 16- or 32-row tiles (no FMAs on
    rows far past M); results stay bit-exact on integer data."""
    N, K = 2048, 700
    g = inputs.generator(4000 + M)
    A = inputs.draw(M, K, "int4", g)
    B = inputs.draw(K, N, "int4", g)
    C = run_f32(tgemm, A.cuda(), B.cuda())
    assert tgemm.binding.last_kernel().startswith("f32_" + tile), tgemm.binding.last_kernel()
    C_ref, _ = oracle.gemm(A, B)
    assert_bit_exact(C, C_ref, f"few rows M={M}")


@pytest.mark.parametrize("shape,tile", [((128, 128, 128), "64x64"), ((384, 384, 384), "64x64"),
                                        ((512, 512, 512), "64x64"), ((256, 256, 4096), "64x64"),
                                        ((640, 640, 640), "128x128"), ((1024, 256, 1024), "128x128"),
                                        ((2048, 2048, 256), "128x128"), ((1024, 1024, 1024), "128x256"),
                                        ((4096, 4096, 8), "128x256")])
def test_small_products_take_smaller_tiles(tgemm, shape, tile):
    """Products whose 128 x 256 tiles would not fill one wave of the GPU take
    64 x 64 or 128 x 128 tiles by a rule fitted to measurements; results stay
    bit-exact on integer data."""
    M, N, K = shape
    g = inputs.generator(M + 5 * N + 11 * K)
    A = inputs.draw(M, K, "int4", g)
    B = inputs.draw(K, N, "int4", g)
    C = run_f32(tgemm, A.cuda(), B.cuda())
    assert tgemm.binding.last_kernel().startswith("f32_" + tile), tgemm.binding.last_kernel()
    rows = sorted(set([0, M - 1] + torch.randint(0, M, (40,), generator=g).tolist()))
    C_ref, _ = oracle.gemm_rows(A, B, rows)
    assert_bit_exact(C.cpu()[rows], C_ref, f"small product {shape}")
