"""The TF32 kernel that transposes B in shared memory (128 x 128 tiles).

TMA lands each 32 x 128 block of a B stored K x N (N contiguous) in its
MN-major layout and two warps of the kernel rewrite it K-major in place
before the MMAs read it. The other kernels now read such a B MN-major
directly (faster), so this one runs only when tensor-core mode 3 forces it,
at any M. Every result is checked against the oracle: bit for bit on
integer data, within the TF32 tolerance on random data.
"""
import re
import time

import pytest
import torch

import oracle
from tests.parity import TC_ABS, TC_REL, assert_bit_exact, assert_within
from tiled_matrix_multiplication_sm_gb300 import inputs

pytestmark = pytest.mark.gpu

KERNEL = "tc_tf32_128x128x32_s6_btrans_persistent"


def operands(M, N, K, dist, seed):
    g = inputs.generator(seed)
    return inputs.draw(M, K, dist, g), inputs.draw(K, N, dist, g)


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


@pytest.mark.parametrize("M", [1, 16, 100, 128, 129])
def test_default_reads_b_as_stored_without_this_kernel(tgemm, M):
    """By default (mode -1) TF32 reads B MN-major as stored with the other
    kernels at any M: neither this kernel nor a transpose pre-pass."""
    N, K = 1000, 264
    A, B = operands(M, N, K, "int4", seed=M)
    C, name = run(tgemm, lambda: tgemm.gemm_tc(A.cuda(), B.cuda(), "tf32"))
    assert KERNEL not in name and "transpose_b" not in name, name
    assert_bit_exact(C, oracle.gemm(A, B)[0], f"M={M}")


@pytest.mark.parametrize("shape", [(1, 8, 8), (8, 8, 8), (127, 248, 40), (129, 264, 72),
                                   (300, 520, 200), (64, 1000, 8), (1000, 136, 16),
                                   (256, 512, 1024), (5, 16, 4104), (513, 1000, 136)])
def test_forced_integer_bit_exact(tgemm, shape):
    """Mode 3 at any M: several tiles in both dimensions, ragged edges, K of
    one block and of many."""
    M, N, K = shape
    A, B = operands(M, N, K, "int4", seed=M + 5 * N + 3 * K)
    C, name = run(tgemm, lambda: tgemm.gemm_tc(A.cuda(), B.cuda(), "tf32"), mode=3)
    assert KERNEL in name, name
    assert_bit_exact(C, oracle.gemm(A, B)[0], f"{shape}")


def test_ragged_nan_padding_never_read(tgemm):
    """N not a multiple of 4 and K not a multiple of the block: the copies
    fill columns past N and rows past K with zeros, never the NaN padding."""
    M, N, K = 389, 301, 97
    A, B = operands(M, N, K, "int4", seed=6)
    C = torch.full((M, N), -1.0, device="cuda")
    run(tgemm, lambda: tgemm.gemm_tc(padded_cuda(A, 104), padded_cuda(B, 312), "tf32", out=C),
        mode=3)
    assert_bit_exact(C, oracle.gemm(A, B)[0], "ragged")


def test_unaligned_rows_are_repacked(tgemm):
    """Packed operands whose rows are not 16-byte aligned: A and B are
    repacked (B as K x N, 128-byte rows), then read as stored."""
    M, N, K = 100, 261, 77
    A, B = operands(M, N, K, "int4", seed=261)
    C, name = run(tgemm, lambda: tgemm.gemm_tc(A.cuda(), B.cuda(), "tf32"), mode=3)
    assert KERNEL in name and "repack_ab+" in name, name
    assert_bit_exact(C, oracle.gemm(A, B)[0], "unaligned")


@pytest.mark.parametrize("ldc,offset", [(523, 3), (524, 1), (520, 0)])
def test_output_rows_and_guard_bands(tgemm, ldc, offset):
    """C rows off 16-byte boundaries (row copies), or aligned (TMA stores);
    padding columns and guard bands untouched."""
    M, N, K = 120, 517, 64
    A, B = operands(M, N, K, "int4", seed=ldc)
    guard = 64
    store = torch.full((guard + offset + M * ldc + guard,), -555.0, device="cuda")
    base = guard + offset
    C = store[base:base + M * ldc].view(M, ldc)[:, :N]
    _, name = run(tgemm, lambda: tgemm.gemm_tc(A.cuda(), B.cuda(), "tf32", out=C), mode=3)
    assert KERNEL in name, name
    assert_bit_exact(C, oracle.gemm(A, B)[0], f"ldc={ldc} offset={offset}")
    host = store.cpu()
    assert (host[:base] == -555.0).all() and (host[base + M * ldc:] == -555.0).all()
    assert (host[base:base + M * ldc].view(M, ldc)[:, N:] == -555.0).all()


@pytest.mark.parametrize("ta", [False, True])
def test_full_output_rule_bit_exact(tgemm, ta):
    """C = alpha A B + beta C + bias, with A stored transposed or not."""
    M, N, K = 96, 700, 300
    g = inputs.generator(70 + ta)
    A = inputs.draw(M, K, "int4", g)
    B = inputs.draw(K, N, "int4", g)
    C0 = inputs.draw(M, N, "int4", g)
    bias = inputs.draw(1, N, "int4", g)[0]
    As = A.t().contiguous() if ta else A
    C = C0.clone().cuda()
    _, name = run(tgemm, lambda: tgemm.binding.gemm_ex(As.cuda(), B.cuda(), "tf32", trans_a=ta,
                                                       alpha=2.0, beta=-1.0, bias=bias.cuda(),
                                                       out=C), mode=3)
    assert KERNEL in name, name
    ref, _ = oracle.gemm_ex(As, B, trans_a=ta, alpha=2.0, beta=-1.0, C0=C0, bias=bias)
    assert_bit_exact(C, ref, f"rule ta={ta}")


@pytest.mark.parametrize("shape,slots", [((100, 1000, 2048), 33), ((16, 2000, 4096), 40),
                                         ((16, 2000, 4096), 152), ((300, 2100, 1032), 100)])
def test_stream_k_integer_bit_exact(tgemm, shape, slots):
    """The tail's K blocks shared by `slots` SMs: partial tiles handed on
    and added by the owner in a fixed order."""
    M, N, K = shape
    A, B = operands(M, N, K, "int4", seed=slots + N)
    C, name = run(tgemm, lambda: tgemm.gemm_tc(A.cuda(), B.cuda(), "tf32"), mode=3, slots=slots)
    m = re.search(r"streamk:slots=(\d+)", name)
    assert KERNEL in name and m is not None and int(m.group(1)) > 0, name
    assert_bit_exact(C, oracle.gemm(A, B)[0], f"{shape} slots={slots}")


@pytest.mark.parametrize("slots", [-1, 0, 152])
def test_float_tolerance(tgemm, slots):
    M, N, K = 100, 1100, 1531
    A, B = operands(M, N, K, "normal", seed=1531)
    C, name = run(tgemm, lambda: tgemm.gemm_tc(A.cuda(), B.cuda(), "tf32"), mode=3, slots=slots)
    assert KERNEL in name, name
    C_ref, absAB = oracle.gemm(A, B)
    assert_within(C, C_ref, absAB, TC_REL, TC_ABS, f"float slots={slots}")


def test_stalled_pipeline_reports_timeout_and_recovers(tgemm):
    """With the stall hook the first stage never lands: the transposer warps'
    and the MMA warp's bounded waits run out, the kernel records the timeout
    and exits, and the next launch is correct."""
    b = tgemm.binding
    A, B = operands(64, 512, 128, "int4", seed=4)
    Ad, Bd = A.cuda(), B.cuda()
    assert tgemm.device_status() == 0
    try:
        assert b.set_wait_limit_ns(50_000_000) == 0
        assert b.set_tc_kernel(3) == 0
        b.set_debug_stall(True)
        t0 = time.time()
        tgemm.gemm_tc(Ad, Bd, "tf32")
        st = tgemm.device_status()
        elapsed = time.time() - t0
        name = b.last_kernel()
    finally:
        b.set_debug_stall(False)
        b.set_tc_kernel(-1)
        b.set_wait_limit_ns(2_000_000_000)
    assert KERNEL in name, name
    assert st == b.TGEMM_ERR_DEVICE_TIMEOUT
    assert elapsed < 10.0
    assert tgemm.device_status() == 0
    C = tgemm.gemm_tc(Ad, Bd, "tf32")
    assert tgemm.device_status() == 0
    assert_bit_exact(C, oracle.gemm(A, B)[0], "after timeout")


@pytest.mark.parametrize("M,N,K", [(16, 32, 64), (100, 96, 300), (7, 160, 33), (128, 640, 96),
                                   (33, 4128, 200)])
def test_whole_chunk_widths_nan_padding(tgemm, M, N, K):
    """N a multiple of 32: each 32 x 128 block of B lands as one 3-D box of
    32-column chunks; the chunks past N and the rows past K read as zeros,
    and the NaN padding of ldb (past N) is never read."""
    A, B = operands(M, N, K, "int4", seed=N + K)
    C, name = run(tgemm, lambda: tgemm.gemm_tc(padded_cuda(A, K + 4), padded_cuda(B, N + 12), "tf32"),
                  mode=3)
    assert KERNEL in name, name
    assert_bit_exact(C, oracle.gemm(A, B)[0], f"{M}x{N}x{K}")
