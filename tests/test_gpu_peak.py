"""The tensor-rate probe (gemm_tc_peak): back-to-back MMAs from resident
shared memory. Checks that it runs to completion on every form and that its
figures are self-consistent: TF32 retires half the FLOP per clock of BF16 on
the same MMA shape, and the SM-pair and one-SM forms agree per SM."""
import pytest

pytestmark = pytest.mark.gpu


def test_peak_rates_are_consistent(tgemm):
    b = tgemm.binding
    rate = {}
    for kind in ("bf16", "tf32"):
        for pair in (False, True):
            per_clk, tflops = b.tc_peak(kind, pair, iters=20000)
            assert per_clk > 0 and tflops > 0
            rate[kind, pair] = per_clk
    assert tgemm.device_status() == 0
    # 2*M*N*K FLOP per MMA; the pipe's rate per clock does not depend on the form
    assert rate["bf16", True] == pytest.approx(rate["bf16", False], rel=0.1)
    assert rate["tf32", True] / rate["bf16", True] == pytest.approx(0.5, rel=0.1)
