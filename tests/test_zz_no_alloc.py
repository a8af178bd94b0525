"""The allocation-free TF32 entry point, gemm_tc_tf32_noalloc.

It serves callers that cannot allocate device memory (an application that
reserves all of its memory up front, code that must not touch the device
allocator while it runs): its scratch is a fixed array inside the library.
Each case calls it through the C ABI twice in a row, on different operands
and shapes, and checks both results against the CPU oracle: with the
tensor-path tolerance |C - C_ref| <= 1e-2 * absAB on random data, bit for
bit on integer data (small integers and their sums are exact in TF32 and
FP32). A B whose rows are 16-byte aligned is read as stored and the array is
not touched ("large", and a problem larger than the array); a B with
ldb = N + 1 is transposed into the array, which covers both of its row
pitches (128-byte rows when they fit, else 16-byte rows: K = 1001 with
N = 4150). The cases also cover a K that is not a multiple of 4 (A then
comes as a padded view with lda a multiple of 4) and a C whose rows are not
16-byte aligned (ldc = N + 1), which takes the register-store epilogue. A
problem whose transposed B would not fit the array is refused without
launching.

The file is named so that pytest collects it last.
"""
import pytest
import torch

import oracle
from tests.parity import TC_ABS, TC_REL, assert_bit_exact, assert_within
from tiled_matrix_multiplication_sm_gb300 import inputs

pytestmark = pytest.mark.gpu

SCRATCH_FLOATS = 4194304


def noalloc(tg, A, B, C):
    return tg.binding.gemm_tc_tf32_noalloc_raw(
        A.shape[0], B.shape[1], A.shape[1], A.data_ptr(), A.stride(0), B.data_ptr(),
        B.stride(0), C.data_ptr(), C.stride(0), torch.cuda.current_stream().cuda_stream)


def device_view(x, ld, pad=float("nan")):
    """Device copy of ``x`` as a view with leading dimension ``ld`` (padding
    columns hold ``pad``)."""
    rows, cols = x.shape
    store = torch.full((rows, ld), pad, dtype=x.dtype, device="cuda")
    store[:, :cols] = x.cuda()
    return store[:, :cols]


# (M, N, K, dist, lda, ldb, ldc): None = packed.
CASES = {
    # B transposed into the array at the 128-byte pitch (1000 x 800 floats
    # fit); then integers.
    "pitch128": [(300, 1000, 772, "normal", None, 1001, None),
                 (640, 768, 1024, "int4", None, 769, None)],
    # B read as stored. The first problem takes the 256 x 512 CTA-pair tiles
    # (64 of them: one round, no split tail).
    "large": [(8192, 1024, 4096, "normal", None, None, None),
              (256, 512, 8192, "normal", None, None, None)],
    # 16-byte pitch (4150 x 1024 floats would not fit, 4150 x 1004 do), K not
    # a multiple of 4 (lda = 1004), C rows off 16 bytes (ldc = 4151).
    "pitch16": [(300, 4150, 1001, "normal", 1004, 4151, 4151),
                (129, 4150, 1001, "int4", 1004, 4151, 4151)],
}


@pytest.mark.parametrize("case", sorted(CASES))
def test_noalloc_matches_oracle_on_two_calls(tgemm, case):
    for call, (M, N, K, dist, lda, ldb, ldc) in enumerate(CASES[case]):
        g = inputs.generator(900 + 10 * sorted(CASES).index(case) + call)
        A = inputs.draw(M, K, dist, g)
        B = inputs.draw(K, N, dist, g)
        Ad = device_view(A, lda) if lda else A.cuda()
        Bd = device_view(B, ldb) if ldb else B.cuda()
        C = device_view(torch.empty(M, N), ldc or N)
        C.fill_(float("nan"))
        assert noalloc(tgemm, Ad, Bd, C) == 0
        assert tgemm.device_status() == 0
        C_ref, absAB = oracle.gemm(A, B)
        what = f"no-alloc {case} call {call + 1} ({M}x{N}x{K}, {dist})"
        if dist == "int4":
            assert_bit_exact(C, C_ref, what)
        else:
            assert_within(C, C_ref, absAB, TC_REL, TC_ABS, what)


def test_noalloc_refuses_problems_beyond_its_scratch(tgemm):
    N, K = 4096, 1028                     # 4096 x 1028 floats > 4 Mi floats
    assert N * K > SCRATCH_FLOATS
    A = torch.ones(8, K, device="cuda")
    B = device_view(torch.ones(K, N), N + 1)      # rows off 16 bytes: must be transposed
    C = torch.full((8, N), 7.0, device="cuda")
    assert noalloc(tgemm, A, B, C) == tgemm.binding.TGEMM_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert (C == 7.0).all()


def test_noalloc_reads_aligned_b_beyond_the_array_size(tgemm):
    """The same sizes with B's rows 16-byte aligned: read as stored, exact."""
    M, N, K = 8, 4096, 1028
    g = inputs.generator(77)
    A = inputs.draw(M, K, "int4", g)
    B = inputs.draw(K, N, "int4", g)
    C = torch.full((M, N), float("nan"), device="cuda")
    assert noalloc(tgemm, A.cuda(), B.cuda(), C) == 0
    assert tgemm.device_status() == 0
    assert_bit_exact(C, oracle.gemm(A, B)[0], "no-alloc, B read as stored")
