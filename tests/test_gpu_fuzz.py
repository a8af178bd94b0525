"""Seeded shape fuzzing of every path against the CPU oracle.

Random M, N, K (with the edge values 1 and tile boundaries mixed in), random
storage (row- or column-major A and B, optional NaN-filled padding of the
leading dimension), random small-integer alpha, beta and bias, on every
path, with the tensor-core tile shape (one SM, SM pair, wide SM pair) drawn
too. The data are small integers, so every product, partial sum and output
rule step is exact: each case must equal the oracle bit for bit.
"""
import random

import pytest
import torch

import oracle
from tests.parity import assert_bit_exact
from tiled_matrix_multiplication_sm_gb300 import inputs

pytestmark = pytest.mark.gpu

DTYPE = {"f32": torch.float32, "tf32": torch.float32, "bf16": torch.bfloat16,
         "tf32x3": torch.float32}
EDGES = [1, 2, 3, 7, 8, 31, 32, 33, 63, 64, 65, 127, 128, 129, 255, 256, 257, 300, 513]


def dim(rng):
    return rng.choice(EDGES) if rng.random() < 0.4 else rng.randint(1, 600)


def device_view(x, pad, rng):
    """x on the device, inside a wider NaN-filled array when ``pad``."""
    rows, cols = x.shape
    if not pad:
        return x.cuda()
    store = torch.full((rows, cols + rng.randint(1, 9)), float("nan"), dtype=x.dtype,
                       device="cuda")
    store[:, :cols] = x.cuda()
    return store[:, :cols]


@pytest.mark.parametrize("seed", range(40))
def test_fuzz_case(tgemm, seed):
    rng = random.Random(seed)
    path = ["f32", "tf32", "bf16", "tf32x3"][seed % 4]
    M, N, K = dim(rng), dim(rng), dim(rng)
    if K * 16 >= 2 ** 24:            # keep partial sums exact in FP32
        K = 1000
    ta, tb = rng.random() < 0.4, rng.random() < 0.4
    alpha = float(rng.choice([1, 1, 2, -1, 3]))
    beta = float(rng.choice([0, 0, 1, -2]))
    use_bias = rng.random() < 0.5
    g = inputs.generator(7000 + seed)
    A = inputs.draw(M, K, "int4", g).to(DTYPE[path])
    B = inputs.draw(K, N, "int4", g).to(DTYPE[path])
    C0 = inputs.draw(M, N, "int4", g)
    bias = inputs.draw(1, N, "int4", g)[0] if use_bias else None
    As = A.t().contiguous() if ta else A
    Bs = B.t().contiguous() if tb else B
    Ad = device_view(As, rng.random() < 0.3, rng)
    Bd = device_view(Bs, rng.random() < 0.3, rng)
    C = C0.clone().cuda()
    mode = rng.choice([-1, 0, 1, 2])
    assert tgemm.binding.set_tc_kernel(mode) == 0
    try:
        tgemm.binding.gemm_ex(Ad, Bd, path, trans_a=ta, trans_b=tb, alpha=alpha, beta=beta,
                              bias=None if bias is None else bias.cuda(), out=C)
    finally:
        tgemm.binding.set_tc_kernel(-1)
    assert tgemm.device_status() == 0
    ref, _ = oracle.gemm_ex(As, Bs, trans_a=ta, trans_b=tb, alpha=alpha, beta=beta, C0=C0,
                            bias=bias)
    assert_bit_exact(C, ref, f"seed {seed}: {path} {M}x{N}x{K} ta={ta} tb={tb} "
                             f"alpha={alpha} beta={beta} bias={use_bias} tc_mode={mode} "
                             f"kernel={tgemm.binding.last_kernel()}")
