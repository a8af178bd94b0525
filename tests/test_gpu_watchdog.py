"""Failure detection on the tensor-core path, without a GPU fault.

With the library's stall hook on, the producer never marks the first
pipeline stage as loaded, so the MMA warp's bounded wait runs out. The kernel
must record TGEMM_ERR_DEVICE_TIMEOUT, free its tensor memory and exit; the
host reads the status and the context stays usable for a correct launch
right after.
"""
import time

import pytest
import torch

import oracle
from tests.parity import assert_bit_exact
from tiled_matrix_multiplication_sm_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("mode", [0, 1, 2], ids=["one_sm", "sm_pair", "sm_pair_wide"])
def test_stalled_pipeline_reports_timeout_and_recovers(tgemm, mode):
    b = tgemm.binding
    assert b.set_tc_kernel(mode) == 0
    g = inputs.generator(4)
    A = inputs.draw(256, 128, "int4", g).to(torch.bfloat16).cuda()
    B = inputs.draw(128, 512, "int4", g).to(torch.bfloat16).cuda()
    assert tgemm.device_status() == 0
    try:
        assert b.set_wait_limit_ns(50_000_000) == 0        # 50 ms
        b.set_debug_stall(True)
        t0 = time.time()
        tgemm.gemm_tc(A, B, "bf16")
        st = tgemm.device_status()
        elapsed = time.time() - t0
    finally:
        b.set_debug_stall(False)
        b.set_wait_limit_ns(2_000_000_000)
        b.set_tc_kernel(-1)
    assert st == b.TGEMM_ERR_DEVICE_TIMEOUT
    assert elapsed < 10.0
    # The status word is cleared by the read ...
    assert tgemm.device_status() == 0
    # ... and the next launch is correct.
    b.set_tc_kernel(mode)
    try:
        C = tgemm.gemm_tc(A, B, "bf16")
    finally:
        b.set_tc_kernel(-1)
    assert tgemm.device_status() == 0
    C_ref, _ = oracle.gemm(A.cpu(), B.cpu())
    assert_bit_exact(C, C_ref, "after timeout")
