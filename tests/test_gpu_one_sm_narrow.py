"""The one-SM tensor-core kernel with 128 x 128 tiles.

Products with at most 128 rows take 128 x 128 tiles where the timing model
expects them to finish first: twice the tiles of the 128 x 256 shape, so a
row of them fills more SMs without sharing tiles along K. Tensor-core mode 4
forces the shape at any M. Every result is checked against the oracle: bit
for bit on integer data, within the path's tolerance on random data.
"""
import re
import time

import pytest
import torch

import oracle
from tests.parity import TC_ABS, TC_REL, assert_bit_exact, assert_within
from tiled_matrix_multiplication_sm_gb300 import inputs

pytestmark = pytest.mark.gpu

DTYPES = {"tf32": torch.float32, "bf16": torch.bfloat16}
NAMES = {"tf32": "tc_tf32_128x128x32_s6_persistent", "bf16": "tc_bf16_128x128x64_s6_persistent"}


def operands(M, N, K, dist, kind, seed):
    g = inputs.generator(seed)
    return inputs.draw(M, K, dist, g).to(DTYPES[kind]), inputs.draw(K, N, dist, g).to(DTYPES[kind])


def padded_cuda(x, ld, pad=float("nan")):
    rows, cols = x.shape
    store = torch.full((rows, ld), pad, dtype=x.dtype, device="cuda")
    store[:, :cols] = x.cuda()
    return store[:, :cols]


def run(tg, fn, mode=-1, slots=-1):
    assert tg.binding.set_tc_kernel(mode) == 0
    assert tg.binding.set_tc_streamk(slots) == 0
    try:
        out = fn()
        name = tg.binding.last_kernel()
    finally:
        tg.binding.set_tc_kernel(-1)
        tg.binding.set_tc_streamk(-1)
    assert tg.device_status() == 0
    return out, name


def test_few_rows_bf16_take_narrow_tiles(tgemm):
    """By default a 16-row BF16 product with many columns takes 128 x 128
    tiles, one per SM, with no stream-K tail."""
    A, B = operands(16, 14336, 512, "int4", "bf16", seed=16)
    C, name = run(tgemm, lambda: tgemm.gemm_tc(A.cuda(), B.cuda(), "bf16"))
    assert name == NAMES["bf16"], name
    assert_bit_exact(C, oracle.gemm(A, B)[0], "16 x 14336 x 512")


@pytest.mark.parametrize("kind", ["bf16", "tf32"])
@pytest.mark.parametrize("shape", [(1, 8, 8), (128, 256, 64), (129, 264, 72), (127, 248, 40),
                                   (300, 520, 200), (64, 1000, 8), (5, 16, 4104), (256, 512, 1024)])
def test_forced_integer_bit_exact(tgemm, kind, shape):
    M, N, K = shape
    A, B = operands(M, N, K, "int4", kind, seed=M + 3 * N + K)
    C, name = run(tgemm, lambda: tgemm.gemm_tc(A.cuda(), B.cuda(), kind), mode=4)
    assert NAMES[kind] in name, name
    assert_bit_exact(C, oracle.gemm(A, B)[0], f"{kind} {shape}")


@pytest.mark.parametrize("kind", ["bf16", "tf32"])
def test_b_stored_transposed(tgemm, kind):
    """B stored N x K (read K-major), with NaN padding in both operands."""
    M, N, K = 100, 300, 96
    A, B = operands(M, N, K, "int4", kind, seed=7)
    Bt = padded_cuda(B.t().contiguous(), K + 8)
    C, name = run(tgemm, lambda: tgemm.binding.gemm_ex(padded_cuda(A, K + 8), Bt, kind, trans_b=True),
                  mode=4)
    assert NAMES[kind] in name, name
    assert_bit_exact(C, oracle.gemm(A, B)[0], f"{kind} B transposed")


@pytest.mark.parametrize("kind", ["bf16", "tf32"])
def test_ragged_nan_padding_and_guard_bands(tgemm, kind):
    M, N, K = 120, 301, 97
    A, B = operands(M, N, K, "int4", kind, seed=9)
    ldc, guard = 307, 32
    store = torch.full((guard + M * ldc + guard,), -777.0, device="cuda")
    C = store[guard:guard + M * ldc].view(M, ldc)[:, :N]
    _, name = run(tgemm, lambda: tgemm.gemm_tc(padded_cuda(A, 104), padded_cuda(B, 312), kind, out=C),
                  mode=4)
    assert NAMES[kind] in name, name
    assert_bit_exact(C, oracle.gemm(A, B)[0], f"{kind} ragged")
    host = store.cpu()
    assert (host[:guard] == -777.0).all() and (host[guard + M * ldc:] == -777.0).all()
    assert (host[guard:guard + M * ldc].view(M, ldc)[:, N:] == -777.0).all()


@pytest.mark.parametrize("kind", ["bf16", "tf32"])
@pytest.mark.parametrize("slots", [40, 152])
def test_stream_k_integer_bit_exact(tgemm, kind, slots):
    M, N, K = 16, 2000, 4096
    A, B = operands(M, N, K, "int4", kind, seed=slots)
    C, name = run(tgemm, lambda: tgemm.gemm_tc(A.cuda(), B.cuda(), kind), mode=4, slots=slots)
    m = re.search(r"streamk:slots=(\d+)", name)
    assert NAMES[kind] in name and m is not None, name
    assert_bit_exact(C, oracle.gemm(A, B)[0], f"{kind} slots={slots}")


@pytest.mark.parametrize("kind", ["bf16", "tf32"])
def test_full_output_rule(tgemm, kind):
    M, N, K = 96, 700, 300
    g = inputs.generator(71)
    A = inputs.draw(M, K, "int4", g).to(DTYPES[kind])
    B = inputs.draw(K, N, "int4", g).to(DTYPES[kind])
    C0 = inputs.draw(M, N, "int4", g)
    bias = inputs.draw(1, N, "int4", g)[0]
    C = C0.clone().cuda()
    _, name = run(tgemm, lambda: tgemm.binding.gemm_ex(A.cuda(), B.cuda(), kind, alpha=2.0, beta=-1.0,
                                                       bias=bias.cuda(), out=C), mode=4)
    assert NAMES[kind] in name, name
    ref, _ = oracle.gemm_ex(A, B, alpha=2.0, beta=-1.0, C0=C0, bias=bias)
    assert_bit_exact(C, ref, f"{kind} rule")


def test_float_tolerance(tgemm):
    M, N, K = 64, 1100, 1531
    A, B = operands(M, N, K, "normal002", "bf16", seed=1531)
    C, name = run(tgemm, lambda: tgemm.gemm_tc(A.cuda(), B.cuda(), "bf16"), mode=4)
    C_ref, absAB = oracle.gemm(A, B)
    assert_within(C, C_ref, absAB, TC_REL, TC_ABS, "bf16 float")


def test_stalled_pipeline_reports_timeout_and_recovers(tgemm):
    b = tgemm.binding
    A, B = operands(64, 512, 128, "int4", "bf16", seed=4)
    Ad, Bd = A.cuda(), B.cuda()
    assert b.set_tc_kernel(4) == 0
    try:
        assert b.set_wait_limit_ns(50_000_000) == 0
        b.set_debug_stall(True)
        t0 = time.time()
        tgemm.gemm_tc(Ad, Bd, "bf16")
        st = tgemm.device_status()
        elapsed = time.time() - t0
        name = b.last_kernel()
    finally:
        b.set_debug_stall(False)
        b.set_wait_limit_ns(2_000_000_000)
        b.set_tc_kernel(-1)
    assert NAMES["bf16"] in name, name
    assert st == b.TGEMM_ERR_DEVICE_TIMEOUT
    assert elapsed < 10.0
    assert tgemm.device_status() == 0
    C = tgemm.gemm_tc(Ad, Bd, "bf16")
    assert tgemm.device_status() == 0
    assert_bit_exact(C, oracle.gemm(A, B)[0], "after timeout")
