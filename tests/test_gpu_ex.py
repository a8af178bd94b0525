"""gemm_ex: transposed storage (column-major operands) and the output rule
C = alpha * op(A) op(B) + beta * C + bias, on every path, against the
oracle's extended form. Integer data makes every step exact (products, sums
below 2^24, the epilogue's scaling by small integers), so those cases must
match bit for bit; float data is checked at each path's tolerance against
scale = |alpha| absAB + |beta C_old| + |bias|."""
import numpy as np
import pytest
import torch

import oracle
from tests.parity import (F32_ABS, F32_REL, TC_ABS, TC_REL, assert_bit_exact,
                          assert_within)
from tiled_matrix_multiplication_sm_gb300 import inputs

pytestmark = pytest.mark.gpu

DTYPE = {"f32": torch.float32, "tf32": torch.float32, "bf16": torch.bfloat16,
         "tf32x3": torch.float32}
TOL = {"f32": (F32_REL, F32_ABS), "tf32": (TC_REL, TC_ABS), "bf16": (TC_REL, TC_ABS),
       "tf32x3": (F32_REL, F32_ABS)}
PATHS = ["f32", "tf32", "bf16", "tf32x3"]


def stored(x, trans):
    return x.t().contiguous() if trans else x


def case(M, N, K, dist, path, seed, ta, tb):
    g = inputs.generator(seed)
    A = inputs.draw(M, K, dist, g).to(DTYPE[path])
    B = inputs.draw(K, N, dist, g).to(DTYPE[path])
    C0 = inputs.draw(M, N, dist, g)
    bias = inputs.draw(1, N, dist, g)[0]
    return stored(A, ta), stored(B, tb), C0, bias


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("ta,tb", [(False, False), (True, False), (False, True), (True, True)])
@pytest.mark.parametrize("shape", [(67, 130, 45), (300, 264, 200)])
def test_integer_full_rule_bit_exact(tgemm, path, ta, tb, shape):
    M, N, K = shape
    As, Bs, C0, bias = case(M, N, K, "int4", path, M + N + K + 7 * ta + 3 * tb, ta, tb)
    C = C0.clone().cuda()
    tgemm.binding.gemm_ex(As.cuda(), Bs.cuda(), path, trans_a=ta, trans_b=tb, alpha=2.0,
                          beta=-1.0, bias=bias.cuda(), out=C)
    assert tgemm.device_status() == 0
    ref, _ = oracle.gemm_ex(As, Bs, trans_a=ta, trans_b=tb, alpha=2.0, beta=-1.0, C0=C0,
                            bias=bias)
    assert_bit_exact(C, ref, f"{path} ta={ta} tb={tb} {shape}")


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("ta,tb", [(True, False), (False, True)])
def test_float_full_rule_tolerance(tgemm, path, ta, tb):
    M, N, K = 513, 380, 777
    dist = "normal002" if path == "bf16" else "normal"
    As, Bs, C0, bias = case(M, N, K, dist, path, 99 + ta, ta, tb)
    C = C0.clone().cuda()
    tgemm.binding.gemm_ex(As.cuda(), Bs.cuda(), path, trans_a=ta, trans_b=tb, alpha=0.75,
                          beta=0.5, bias=bias.cuda(), out=C)
    ref, scale = oracle.gemm_ex(As, Bs, trans_a=ta, trans_b=tb, alpha=0.75, beta=0.5, C0=C0,
                                bias=bias)
    rel, abs_ = TOL[path]
    assert_within(C, ref, scale, rel, abs_, f"{path} float rule")


@pytest.mark.parametrize("path", PATHS)
def test_transposed_storage_with_nan_padding(tgemm, path):
    """Column-major operands inside wider arrays: the NaN padding is never read."""
    M, N, K = 203, 150, 97
    g = inputs.generator(5)
    A = inputs.draw(M, K, "int4", g).to(DTYPE[path])
    B = inputs.draw(K, N, "int4", g).to(DTYPE[path])
    Astore = torch.full((K, M + 9), float("nan"), dtype=DTYPE[path])
    Astore[:, :M] = A.t()
    Bstore = torch.full((N, K + 5), float("nan"), dtype=DTYPE[path])
    Bstore[:, :K] = B.t()
    Ad, Bd = Astore.cuda()[:, :M], Bstore.cuda()[:, :K]
    C = tgemm.binding.gemm_ex(Ad, Bd, path, trans_a=True, trans_b=True)
    assert tgemm.device_status() == 0
    ref, _ = oracle.gemm(A, B)
    assert_bit_exact(C, ref, f"{path} padded transposed")


@pytest.mark.parametrize("path", ["f32", "bf16"])
def test_beta_zero_ignores_nan_in_C(tgemm, path):
    As, Bs, _, _ = case(64, 96, 40, "int4", path, 3, False, False)
    C = torch.full((64, 96), float("nan"), device="cuda")
    tgemm.binding.gemm_ex(As.cuda(), Bs.cuda(), path, alpha=3.0, beta=0.0, out=C)
    ref, _ = oracle.gemm_ex(As, Bs, alpha=3.0)
    assert_bit_exact(C, ref, "beta 0")


def test_k_zero_applies_output_rule(tgemm):
    C0 = torch.arange(12.0).view(3, 4)
    bias = torch.tensor([1.0, -2.0, 0.5, 4.0])
    C = C0.clone().cuda()
    tgemm.binding.gemm_ex(torch.empty(3, 0, device="cuda"), torch.empty(0, 4, device="cuda"),
                          "f32", beta=2.0, bias=bias.cuda(), out=C)
    assert torch.equal(C.cpu(), 2 * C0 + bias)


@pytest.mark.parametrize("path", PATHS)
def test_split_k_tail_applies_rule_once(tgemm, path):
    """A shape whose last wave is split along K: the reduction (FP32 path) or
    the owner of each shared tile (tensor paths, stream-K), not each piece,
    applies alpha, beta and bias."""
    M, N, K = 256, 512, 2048
    As, Bs, C0, bias = case(M, N, K, "int4", path, 77, False, True)
    C = C0.clone().cuda()
    if path != "f32":
        assert tgemm.binding.set_tc_streamk(40) == 0
    try:
        tgemm.binding.gemm_ex(As.cuda(), Bs.cuda(), path, trans_b=True, alpha=-1.0, beta=1.0,
                              bias=bias.cuda(), out=C)
        name = tgemm.binding.last_kernel()
    finally:
        tgemm.binding.set_tc_streamk(-1)
    assert ("splitk_reduce" if path == "f32" else "streamk:slots=40") in name, name
    ref, _ = oracle.gemm_ex(As, Bs, trans_b=True, alpha=-1.0, beta=1.0, C0=C0, bias=bias)
    assert_bit_exact(C, ref, f"{path} split rule")
