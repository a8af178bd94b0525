"""The tensor paths' in-place loader for an A whose rows are 4-byte but not
16-byte aligned (gemm_set_tc_a_loader(1)): two extra warps of the GEMM
kernel copy A with 4-byte asynchronous copies into the layout a TMA copy
would write, instead of a repack pre-pass.

Every tile shape (one SM, SM pair, wide SM pair) and both input types, with
ragged M, N and K (an odd K on BF16 leaves half a word at the end of each
row), A's leading-dimension padding filled with NaN (any read of it poisons
the product) and integer data: bit for bit against the oracle. Plus a
stream-K tail, random data within tolerance, and the bounded-wait path.
"""
import pytest
import torch

import oracle
from tests.parity import TC_ABS, TC_REL, assert_bit_exact, assert_within
from tiled_matrix_multiplication_sm_gb300 import inputs

pytestmark = pytest.mark.gpu

DTYPES = {"tf32": torch.float32, "bf16": torch.bfloat16}


def nan_padded(x, ld):
    rows, cols = x.shape
    store = torch.full((rows, ld), float("nan"), dtype=x.dtype, device="cuda")
    store[:, :cols] = x.cuda()
    return store[:, :cols]


def pick_lda(K, esz):
    """The first leading dimension past K whose rows are 4- but not 16-byte aligned."""
    ld = K + 1
    while (ld * esz) % 4 != 0 or (ld * esz) % 16 == 0:
        ld += 1
    return ld


def run(tg, mode, A, B, kind, streamk=-1, out=None):
    assert tg.binding.set_tc_a_loader(1) == 0
    assert tg.binding.set_tc_kernel(mode) == 0
    assert tg.binding.set_tc_streamk(streamk) == 0
    try:
        C = tg.gemm_tc(A, B, kind, out=out)
        name = tg.binding.last_kernel()
    finally:
        tg.binding.set_tc_a_loader(-1)
        tg.binding.set_tc_kernel(-1)
        tg.binding.set_tc_streamk(-1)
    assert tg.device_status() == 0
    return C, name


# (M, N, K): K = 1 word short of a block, K past a block, odd K (bf16 half words).
SHAPES = [(100, 300, 70), (300, 520, 517), (513, 1000, 129), (257, 264, 1031)]


@pytest.mark.parametrize("mode", [0, 1, 2])
@pytest.mark.parametrize("kind", ["tf32", "bf16"])
@pytest.mark.parametrize("shape", SHAPES)
def test_integer_bit_exact_nan_padding(tgemm, mode, kind, shape):
    M, N, K = shape
    g = inputs.generator(M + 3 * N + 5 * K + mode)
    A = inputs.draw(M, K, "int4", g).to(DTYPES[kind])
    B = inputs.draw(K, N, "int4", g).to(DTYPES[kind])
    lda = pick_lda(K, A.element_size())
    C, name = run(tgemm, mode, nan_padded(A, lda), B.cuda(), kind)
    assert "(a_loader)" in name and "repack_a" not in name, name
    assert_bit_exact(C, oracle.gemm(A, B)[0], f"{kind} {shape} mode {mode}")


@pytest.mark.parametrize("kind", ["tf32", "bf16"])
def test_stream_k_tail_and_random_data(tgemm, kind):
    M, N, K = 600, 1100, 1027
    g = inputs.generator(99)
    dist = "normal002" if kind == "bf16" else "normal"
    A = inputs.draw(M, K, dist, g).to(DTYPES[kind])
    B = inputs.draw(K, N, dist, g).to(DTYPES[kind])
    lda = pick_lda(K, A.element_size())
    C, name = run(tgemm, 1, nan_padded(A, lda), B.cuda(), kind, streamk=40)
    assert "(a_loader)" in name and "streamk" in name, name
    C_ref, absAB = oracle.gemm(A, B)
    assert_within(C, C_ref, absAB, TC_REL, TC_ABS, f"{kind} loader + stream-K")


def test_bounded_wait_with_loader(tgemm):
    """The stall hook leaves stage 0 empty: the kernel reports the timeout,
    its loader warps finish their copies and the next launch is correct."""
    g = inputs.generator(5)
    A = inputs.draw(300, 301, "int4", g)
    B = inputs.draw(301, 520, "int4", g)
    Ad = nan_padded(A, 302)
    assert tgemm.binding.set_wait_limit_ns(50_000_000) == 0
    assert tgemm.binding.set_debug_stall(True) == 0
    assert tgemm.binding.set_tc_a_loader(1) == 0
    try:
        tgemm.gemm_tc(Ad, B.cuda(), "tf32")
        assert tgemm.device_status() == tgemm.binding.TGEMM_ERR_DEVICE_TIMEOUT
    finally:
        tgemm.binding.set_debug_stall(False)
        tgemm.binding.set_wait_limit_ns(2_000_000_000)
        tgemm.binding.set_tc_a_loader(-1)
    C, name = run(tgemm, -1, Ad, B.cuda(), "tf32")
    assert_bit_exact(C, oracle.gemm(A, B)[0], "after the timeout")


@pytest.mark.parametrize("mode", [0, 1, 2])
def test_tf32_b_stored_transposed(tgemm, mode):
    """TF32 with B stored N x K (read K-major, rows 16-byte aligned: K a
    multiple of 4) beside the loader's A (lda = K + 1)."""
    M, N, K = 300, 520, 516
    g = inputs.generator(7 + mode)
    A = inputs.draw(M, K, "int4", g)
    B = inputs.draw(K, N, "int4", g)
    lda = pick_lda(K, 4)
    assert tgemm.binding.set_tc_a_loader(1) == 0
    assert tgemm.binding.set_tc_kernel(mode) == 0
    try:
        C = tgemm.binding.gemm_ex(nan_padded(A, lda), B.t().contiguous().cuda(), "tf32",
                                  trans_b=True)
        name = tgemm.binding.last_kernel()
    finally:
        tgemm.binding.set_tc_a_loader(-1)
        tgemm.binding.set_tc_kernel(-1)
    assert tgemm.device_status() == 0
    assert "(a_loader)" in name and "repack" not in name and "transpose" not in name, name
    assert_bit_exact(C, oracle.gemm(A, B)[0], f"tf32 B^T mode {mode}")
