"""The allocation-free TF32 entry point, gemm_tc_tf32_noalloc.

It serves callers that cannot allocate device memory (an application that
reserves all of its memory up front, code that must not touch the device
allocator while it runs): its scratch is a fixed array inside the library.
This test calls it through the C ABI twice in a row, on different operands
and shapes, and checks each result against gemm_tc's TF32 result on the same
operands with the tensor-path tolerance |C - C_ref| <= 1e-2 * absAB. It also
checks that a problem too large for the fixed scratch is refused.

The file is named so that pytest collects it last.
"""
import pytest
import torch

import oracle
from tests.parity import TC_ABS, TC_REL, assert_within
from tiled_matrix_multiplication_sm_gb300 import inputs

pytestmark = pytest.mark.gpu

SCRATCH_FLOATS = 4194304


def noalloc(tg, A, B, C):
    return tg.binding.gemm_tc_tf32_noalloc_raw(
        A.shape[0], B.shape[1], A.shape[1], A.data_ptr(), A.stride(0), B.data_ptr(),
        B.stride(0), C.data_ptr(), C.stride(0), torch.cuda.current_stream().cuda_stream)


# The second pair's first problem takes the 256 x 512 CTA-pair tiles (64 of
# them: one round, no split of a tail).
@pytest.mark.parametrize("first,second", [((300, 1000, 772), (513, 264, 2048)),
                                          ((8192, 1024, 4096), (256, 512, 8192))])
def test_noalloc_matches_gemm_tc_on_two_calls(tgemm, first, second):
    for call, (M, N, K) in enumerate([first, second]):
        g = inputs.generator(900 + call)
        A = inputs.draw(M, K, "normal", g)
        B = inputs.draw(K, N, "normal", g)
        Ad, Bd = A.cuda(), B.cuda()
        C_ref = tgemm.gemm_tc(Ad, Bd, "tf32")
        C = torch.full((M, N), float("nan"), device="cuda")
        assert noalloc(tgemm, Ad, Bd, C) == 0
        assert tgemm.device_status() == 0
        _, absAB = oracle.gemm(A, B)
        assert_within(C, C_ref.cpu().double().numpy(), absAB, TC_REL, TC_ABS,
                      f"no-alloc call {call + 1}")


def test_noalloc_refuses_problems_beyond_its_scratch(tgemm):
    N, K = 4096, 1028                     # 4096 x 1028 floats > 4 Mi floats
    assert N * K > SCRATCH_FLOATS
    A = torch.ones(8, K, device="cuda")
    B = torch.ones(K, N, device="cuda")
    C = torch.full((8, N), 7.0, device="cuda")
    assert noalloc(tgemm, A, B, C) == tgemm.binding.TGEMM_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert (C == 7.0).all()
