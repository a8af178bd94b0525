"""Outputs larger than 2^31 elements: every element offset row * ldc + col
of the last rows needs 64-bit arithmetic in the kernels, the split-K
scratch and the TMA tensor maps. C is 48000 x 48000 FP32 (9.2 GB); K is
small so each launch takes milliseconds. Integer data, so the sampled rows
(all columns) must equal the oracle bit for bit."""
import pytest
import torch

import oracle
from tests.parity import assert_bit_exact
from tiled_matrix_multiplication_sm_gb300 import inputs

pytestmark = pytest.mark.gpu

M = N = 48000
DTYPE = {"f32": torch.float32, "tf32": torch.float32, "bf16": torch.bfloat16}


@pytest.mark.parametrize("path,K", [("f32", 24), ("tf32", 24), ("bf16", 40)])
def test_output_past_2_31_elements(tgemm, path, K):
    assert M * N > 2 ** 31
    g = inputs.generator(4800 + K)
    A = inputs.draw(M, K, "int4", g).to(DTYPE[path])
    B = inputs.draw(K, N, "int4", g).to(DTYPE[path])
    C = torch.empty(M, N, device="cuda")
    if path == "f32":
        tgemm.gemm_f32(A.cuda(), B.cuda(), out=C)
    else:
        tgemm.gemm_tc(A.cuda(), B.cuda(), path, out=C)
    assert tgemm.device_status() == 0
    rows = sorted(set([0, 1, M // 2, M - 256, M - 2, M - 1] +
                      torch.randint(0, M, (6,), generator=inputs.generator(48)).tolist()))
    got = C[rows].cpu()
    del C
    C_ref, _ = oracle.gemm_rows(A, B, rows)
    assert_bit_exact(got, C_ref, f"{path} {M}x{N}x{K} sampled rows")
