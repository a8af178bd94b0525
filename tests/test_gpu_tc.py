"""Parity of the tcgen05 tensor-core path (gemm_tc, TF32 and BF16) with the
CPU oracle.

Tolerance (tensor path): |C - C_ref| <= 1e-2 * absAB element by element.
Small integers are exact in TF32 and BF16 and their products are exact, so
integer-valued inputs whose partial sums stay below 2^24 must match the
oracle bit for bit on this path too. All calls go through the C ABI.
"""
import pytest
import torch

import oracle
from tests.parity import TC_ABS, TC_REL, assert_bit_exact, assert_within
from tiled_matrix_multiplication_sm_gb300 import inputs

pytestmark = pytest.mark.gpu

DTYPES = {"tf32": torch.float32, "bf16": torch.bfloat16}


def run_tc(tg, A, B, kind, out=None):
    C = tg.gemm_tc(A.cuda() if A.device.type == "cpu" else A,
                   B.cuda() if B.device.type == "cpu" else B, kind, out=out)
    assert tg.device_status() == 0
    return C


def operands(M, N, K, dist, kind, seed):
    g = inputs.generator(seed)
    A = inputs.draw(M, K, dist, g).to(DTYPES[kind])
    B = inputs.draw(K, N, dist, g).to(DTYPES[kind])
    return A, B


def padded_cuda(x, ld, pad=float("nan")):
    rows, cols = x.shape
    store = torch.full((rows, ld), pad, dtype=x.dtype, device="cuda")
    store[:, :cols] = x.cuda()
    return store[:, :cols]


# ---------------------------------------------------------------- workloads

def test_workload_n4096_tf32_full(tgemm, workload_reference):
    """Full-size launch, every output checked against the oracle."""
    A, B, C_ref, absAB = workload_reference("n4096")
    C = run_tc(tgemm, A, B, "tf32")
    assert_within(C, C_ref, absAB, TC_REL, TC_ABS, "n4096 tf32")


@pytest.mark.parametrize("name,kind", [("skinny_bf16", "bf16"), ("skinny_f32", "tf32")])
def test_workload_skinny_full(tgemm, workload_reference, name, kind):
    """The FFN shape with 16 rows (bound by reading B), every output checked."""
    A, B, C_ref, absAB = workload_reference(name)
    C = run_tc(tgemm, A, B, kind)
    assert_within(C, C_ref, absAB, TC_REL, TC_ABS, f"{name} {kind}")


def test_workload_ffn_bf16_checked_rows(tgemm):
    """Full FFN-shaped launch; the oracle checks the workload's 256 seeded rows."""
    w = inputs.WORKLOADS["ffn_bf16"]
    A, B = inputs.operands(w)
    C = run_tc(tgemm, A, B, "bf16").cpu()
    rows = inputs.check_rows(w).tolist()
    C_ref, absAB = oracle.gemm_rows(A, B, rows)
    assert_within(C[rows], C_ref, absAB, TC_REL, TC_ABS, "ffn bf16")


# ---------------------------------------------------------------- shapes

# Shapes keep K a multiple of 8 and N a multiple of 8 so packed operands meet
# the 16-byte leading-dimension rule of the tensor-memory copies.
SHAPES = [(1, 8, 8), (8, 8, 8), (128, 256, 64), (129, 264, 72), (127, 248, 40),
          (300, 520, 200), (64, 1000, 8), (1000, 64, 16), (256, 512, 1024), (5, 16, 4104)]


@pytest.mark.parametrize("kind", ["tf32", "bf16"])
@pytest.mark.parametrize("shape", SHAPES)
def test_integer_bit_exact(tgemm, kind, shape):
    M, N, K = shape
    A, B = operands(M, N, K, "int4", kind, seed=M + 3 * N + 7 * K)
    C_ref, _ = oracle.gemm(A, B)
    assert_bit_exact(run_tc(tgemm, A, B, kind), C_ref, f"{kind} {shape}")


@pytest.fixture(params=[0, 1, 2], ids=["one_sm", "sm_pair", "sm_pair_wide"])
def tc_mode(request, tgemm):
    """Force the one-SM kernel (0), the 2-SM CTA-pair kernel with 256 x 256
    tiles (1) or with 256 x 512 tiles (2)."""
    assert tgemm.binding.set_tc_kernel(request.param) == 0
    yield request.param
    tgemm.binding.set_tc_kernel(-1)


@pytest.mark.parametrize("kind", ["tf32", "bf16"])
@pytest.mark.parametrize("shape", [(1, 8, 8), (129, 264, 72), (300, 520, 200), (256, 512, 1024),
                                   (513, 1000, 136), (640, 256, 4104)])
def test_both_kernels_integer_bit_exact(tgemm, tc_mode, kind, shape):
    M, N, K = shape
    A, B = operands(M, N, K, "int4", kind, seed=11 * M + N + K)
    C_ref, _ = oracle.gemm(A, B)
    C = run_tc(tgemm, A, B, kind)
    name = tgemm.binding.last_kernel()
    assert ("2sm" in name) == (tc_mode >= 1)
    assert ("256x512" in name) == (tc_mode == 2)
    assert_bit_exact(C, C_ref, f"{kind} {shape} mode {tc_mode}")


@pytest.mark.parametrize("kind", ["tf32", "bf16"])
@pytest.mark.parametrize("shape", [(129, 264, 72), (513, 1000, 136)])
def test_both_kernels_b_stored_transposed(tgemm, tc_mode, kind, shape):
    """B stored N x K: every tile shape reads it K-major (no copy), the
    default K x N storage MN-major."""
    M, N, K = shape
    A, B = operands(M, N, K, "int4", kind, seed=3 * M + N + 7 * K)
    C = tgemm.binding.gemm_ex(A.cuda(), B.t().contiguous().cuda(), kind, trans_b=True)
    name = tgemm.binding.last_kernel()
    assert tgemm.device_status() == 0
    assert "transpose" not in name and "repack" not in name, name
    assert_bit_exact(C, oracle.gemm(A, B)[0], f"{kind} {shape} B^T mode {tc_mode}")


@pytest.mark.parametrize("kind", ["tf32", "bf16"])
@pytest.mark.parametrize("N", [64, 256, 544, 1024, 1056, 1064])
def test_b_column_chunks_nan_padding(tgemm, tc_mode, kind, N):
    """B read MN-major: a tile whose columns are all whole 128-byte chunks
    of B arrives as one 3-D copy, the last tile (past N rounded down to a
    chunk) as 2-D copies per chunk. N whole chunks or not, on every tile
    shape; ldb's NaN padding must never be read."""
    M, K = 260, 100
    A, B = operands(M, N, K, "int4", kind, seed=N + 17 * tc_mode)
    C = tgemm.gemm_tc(padded_cuda(A, K + 8), padded_cuda(B, N + 40), kind)
    assert tgemm.device_status() == 0
    assert_bit_exact(C, oracle.gemm(A, B)[0], f"{kind} N={N} mode {tc_mode}")


@pytest.mark.parametrize("kind", ["tf32", "bf16"])
def test_both_kernels_ragged_nan_padding(tgemm, tc_mode, kind):
    M, N, K = 389, 301, 97
    A, B = operands(M, N, K, "int4", kind, seed=6)
    C = torch.full((M, N), -1.0, device="cuda")
    tgemm.gemm_tc(padded_cuda(A, 104), padded_cuda(B, 312), kind, out=C)
    assert tgemm.device_status() == 0
    C_ref, _ = oracle.gemm(A, B)
    assert_bit_exact(C, C_ref, f"{kind} ragged mode {tc_mode}")


@pytest.mark.parametrize("kind", ["tf32", "bf16"])
@pytest.mark.parametrize("shape", [(200, 296, 136), (513, 1032, 520)])
def test_float_tolerance(tgemm, kind, shape):
    M, N, K = shape
    dist = "normal" if kind == "tf32" else "normal002"
    A, B = operands(M, N, K, dist, kind, seed=sum(shape))
    C_ref, absAB = oracle.gemm(A, B)
    assert_within(run_tc(tgemm, A, B, kind), C_ref, absAB, TC_REL, TC_ABS, f"{kind} {shape}")


@pytest.mark.parametrize("kind", ["tf32", "bf16"])
def test_ragged_edges_with_nan_padding(tgemm, kind):
    """M, N, K not multiples of any tile; NaN in the ld padding must never be
    read (the copies fill out-of-range elements with zeros)."""
    M, N, K = 203, 301, 97
    A, B = operands(M, N, K, "int4", kind, seed=5)
    Ad = padded_cuda(A, 104)
    Bd = padded_cuda(B, 312)
    ldc, guard = 307, 32
    store = torch.full((guard + M * ldc + guard,), -777.0, device="cuda")
    C = store[guard:guard + M * ldc].view(M, ldc)[:, :N]
    tgemm.gemm_tc(Ad, Bd, kind, out=C)
    assert tgemm.device_status() == 0
    C_ref, _ = oracle.gemm(A, B)
    assert_bit_exact(C, C_ref, f"{kind} ragged")
    host = store.cpu()
    assert (host[:guard] == -777.0).all() and (host[guard + M * ldc:] == -777.0).all()
    assert (host[guard:guard + M * ldc].view(M, ldc)[:, N:] == -777.0).all()


@pytest.mark.parametrize("kind", ["tf32", "bf16"])
@pytest.mark.parametrize("ldc,offset", [(521, 0), (522, 1), (523, 3), (524, 1)])
def test_unaligned_output_rows_every_phase(tgemm, tc_mode, kind, ldc, offset):
    """C rows that start 4, 8 or 12 bytes past a 16-byte boundary (every
    phase occurs across the rows): each row's values before its first 16-byte
    boundary are stored one by one, the rest as 16-byte vectors. Bit-exact on
    integers; the padding columns and the guard bands stay untouched."""
    M, N, K = 300, 520, 64
    A, B = operands(M, N, K, "int4", kind, seed=ldc + offset)
    guard = 64
    store = torch.full((guard + offset + M * ldc + guard,), -555.0, device="cuda")
    base = guard + offset
    C = store[base:base + M * ldc].view(M, ldc)[:, :N]
    tgemm.gemm_tc(A.cuda(), B.cuda(), kind, out=C)
    assert tgemm.device_status() == 0
    C_ref, _ = oracle.gemm(A, B)
    assert_bit_exact(C, C_ref, f"{kind} ldc={ldc} offset={offset}")
    host = store.cpu()
    assert (host[:base] == -555.0).all() and (host[base + M * ldc:] == -555.0).all()
    assert (host[base:base + M * ldc].view(M, ldc)[:, N:] == -555.0).all()


@pytest.mark.parametrize("kind", ["tf32", "bf16"])
@pytest.mark.parametrize("N", [33, 34, 35, 289, 291])
def test_unaligned_output_rows_short_last_block(tgemm, tc_mode, kind, N):
    """C rows off 16-byte boundaries (ldc = N + 1: every phase occurs) where
    the last 32-column block at N holds only 1-3 columns after a full block:
    the values carried from the full block must still be stored. Bit-exact on
    integers; padding and guard bands untouched."""
    M, K, ldc = 200, 40, N + 1
    A, B = operands(M, N, K, "int4", kind, seed=N)
    guard = 64
    store = torch.full((guard + M * ldc + guard,), -333.0, device="cuda")
    C = store[guard:guard + M * ldc].view(M, ldc)[:, :N]
    tgemm.gemm_tc(A.cuda(), B.cuda(), kind, out=C)
    assert tgemm.device_status() == 0
    assert_bit_exact(C, oracle.gemm(A, B)[0], f"{kind} N={N}")
    host = store.cpu()
    assert (host[:guard] == -333.0).all() and (host[guard + M * ldc:] == -333.0).all()
    assert (host[guard:guard + M * ldc].view(M, ldc)[:, N:] == -333.0).all()


@pytest.mark.parametrize("kind", ["tf32", "bf16"])
@pytest.mark.parametrize("shape", [(16, 12, 12), (130, 261, 77), (300, 1001, 517),
                                   (203, 2051, 1031)])
def test_unaligned_leading_dimensions(tgemm, tc_mode, kind, shape):
    """Packed operands whose rows do not start on 16-byte boundaries: the
    library repacks them for the tensor-memory copies (bit-exact on integers)."""
    M, N, K = shape
    A, B = operands(M, N, K, "int4", kind, seed=M * N + K)
    C = run_tc(tgemm, A, B, kind)
    name = tgemm.binding.last_kernel()
    a_off = (K * A.element_size()) % 16 != 0
    b_off = (N * B.element_size()) % 16 != 0
    expect = "repack_ab+" if a_off and b_off else "repack_a+" if a_off else "repack_b+" if b_off else None
    assert (expect in name) if expect else ("repack" not in name), name
    C_ref, _ = oracle.gemm(A, B)
    assert_bit_exact(C, C_ref, f"{kind} unaligned {shape}")


def test_unaligned_operand_offsets(tgemm):
    """A and B starting 2 and 6 bytes past a 16-byte boundary (bf16)."""
    M, N, K = 100, 90, 64
    A, B = operands(M, N, K, "int4", "bf16", seed=9)
    baseA = torch.zeros(M * K + 1, dtype=torch.bfloat16, device="cuda")
    baseB = torch.zeros(K * N + 3, dtype=torch.bfloat16, device="cuda")
    Ad = baseA[1:].view(M, K)
    Bd = baseB[3:].view(K, N)
    Ad.copy_(A)
    Bd.copy_(B)
    C = run_tc(tgemm, Ad, Bd, "bf16")
    C_ref, _ = oracle.gemm(A, B)
    assert_bit_exact(C, C_ref, "bf16 offset operands")


def test_workload_ragged_tf32_full(tgemm, workload_reference):
    """The 3000 x 5001 x 1537 packed workload on the tensor path (TF32),
    every output checked."""
    A, B, C_ref, absAB = workload_reference("ragged")
    C = run_tc(tgemm, A, B, "tf32")
    assert_within(C, C_ref, absAB, TC_REL, TC_ABS, "ragged tf32")


def test_k_zero_writes_zeros(tgemm):
    C = torch.full((9, 16), 5.0, device="cuda")
    tgemm.gemm_tc(torch.empty(9, 0, device="cuda"), torch.empty(0, 16, device="cuda"),
                  "tf32", out=C)
    assert tgemm.device_status() == 0
    assert (C == 0).all()


def test_back_to_back_launches_reuse_tensor_memory(tgemm):
    """Many launches in a row (each allocates and frees tensor memory)."""
    A, B = operands(256, 512, 256, "int4", "bf16", seed=77)
    C_ref, _ = oracle.gemm(A, B)
    Ad, Bd = A.cuda(), B.cuda()
    outs = [tgemm.gemm_tc(Ad, Bd, "bf16") for _ in range(20)]
    assert tgemm.device_status() == 0
    for C in outs:
        assert_bit_exact(C, C_ref, "repeat")


@pytest.mark.parametrize("kind", ["tf32", "bf16"])
def test_matmul_host_round_trip(tgemm, kind):
    A, B = operands(64, 72, 40, "int4", kind, seed=3)
    C = tgemm.matmul(A.pin_memory(), B.pin_memory(), kind)
    assert C.device.type == "cpu"
    C_ref, _ = oracle.gemm(A, B)
    assert_bit_exact(C, C_ref, f"matmul {kind}")


# ---------------------------------------------------------------- tile shapes

def test_auto_shape_takes_wide_tiles_for_long_k(tgemm):
    """By shape (mode -1): 256 x 512 tiles where the main loop dominates (the
    FFN-shaped product, K = 4096), 256 x 256 tiles at small K."""
    g = inputs.generator(31)
    A = inputs.draw(2048, 2048, "int4", g).to(torch.bfloat16).cuda()
    B = inputs.draw(2048, 2048, "int4", g).to(torch.bfloat16).cuda()
    run_tc(tgemm, A, B, "bf16")
    assert "2sm_256x256" in tgemm.binding.last_kernel()
    w = inputs.WORKLOADS["ffn_bf16"]
    A = torch.zeros(w.M, w.K, dtype=torch.bfloat16, device="cuda")
    B = torch.zeros(w.K, w.N, dtype=torch.bfloat16, device="cuda")
    C = run_tc(tgemm, A, B, "bf16")
    assert "2sm_256x512" in tgemm.binding.last_kernel()
    assert (C == 0).all()


@pytest.mark.parametrize("kind", ["tf32", "bf16"])
@pytest.mark.parametrize("slots", [7, 76])
def test_wide_tiles_stream_k_full_output_rule(tgemm, kind, slots):
    """256 x 512 tiles whose only (partial) round is shared by `slots` SM
    pairs (stream-K): contributions leave raw partial tiles and each owner
    adds them and applies alpha, beta and bias once; C's rows are not
    16-byte aligned (register stores). Integer data: bit-exact."""
    M, N, K = 512, 1530, 2048
    g = inputs.generator(32)
    A = inputs.draw(M, K, "int4", g).to(DTYPES[kind])
    B = inputs.draw(K, N, "int4", g).to(DTYPES[kind])
    C0 = inputs.draw(M, N, "int4", g)
    bias = inputs.draw(1, N, "int4", g)[0]
    C = C0.clone().cuda()
    assert tgemm.binding.set_tc_kernel(2) == 0
    assert tgemm.binding.set_tc_streamk(slots) == 0
    try:
        tgemm.binding.gemm_ex(A.cuda(), B.cuda(), kind, alpha=2.0, beta=-1.0, bias=bias.cuda(),
                              out=C)
        name = tgemm.binding.last_kernel()
    finally:
        tgemm.binding.set_tc_kernel(-1)
        tgemm.binding.set_tc_streamk(-1)
    assert tgemm.device_status() == 0
    assert "256x512" in name and f"streamk:slots={slots},tiles=6" in name, name
    ref, _ = oracle.gemm_ex(A, B, alpha=2.0, beta=-1.0, C0=C0, bias=bias)
    assert_bit_exact(C, ref, f"wide stream-K {kind}")


# ---------------------------------------------------------------- split TF32 (TGEMM_TF32X3)

@pytest.mark.parametrize("shape", [(1, 8, 8), (130, 261, 77), (300, 520, 200), (513, 1032, 520),
                                   (256, 512, 4104)])
def test_tf32x3_meets_fp32_tolerance(tgemm, shape):
    """Three TF32 products on hi/lo splits reach the FP32 path's bound
    |C - C_ref| <= 1e-5 absAB + 1e-6."""
    M, N, K = shape
    g = inputs.generator(3 * M + N + K)
    A = inputs.draw(M, K, "normal", g)
    B = inputs.draw(K, N, "normal", g)
    C = run_tc(tgemm, A, B, "tf32x3")
    assert "tf32x3" in tgemm.binding.last_kernel()
    C_ref, absAB = oracle.gemm(A, B)
    from tests.parity import F32_ABS, F32_REL
    assert_within(C, C_ref, absAB, F32_REL, F32_ABS, f"tf32x3 {shape}")


def test_tf32x3_integer_bit_exact(tgemm):
    A, B = operands(333, 517, 300, "int4", "tf32", seed=8)
    C_ref, _ = oracle.gemm(A, B)
    assert_bit_exact(run_tc(tgemm, A, B, "tf32x3"), C_ref, "tf32x3 int")


def test_tf32x3_much_closer_than_tf32(tgemm):
    """The split form's worst error relative to absAB is far below plain TF32's."""
    g = inputs.generator(31337)
    A = inputs.draw(256, 384, "uniform", g)
    B = inputs.draw(384, 320, "uniform", g)
    C_ref, absAB = oracle.gemm(A, B)
    e1 = (run_tc(tgemm, A, B, "tf32").cpu().double().numpy() - C_ref) / absAB
    e3 = (run_tc(tgemm, A, B, "tf32x3").cpu().double().numpy() - C_ref) / absAB
    assert abs(e3).max() < abs(e1).max() / 50


def test_workload_n4096_tf32x3_full(tgemm, workload_reference):
    A, B, C_ref, absAB = workload_reference("n4096")
    C = run_tc(tgemm, A, B, "tf32x3")
    from tests.parity import F32_ABS, F32_REL
    assert_within(C, C_ref, absAB, F32_REL, F32_ABS, "n4096 tf32x3")


def test_auto_shape_prefers_narrow_tiles_for_unaligned_output_rows(tgemm):
    """The wide tiles' single accumulator leaves part of each epilogue
    exposed, more so when C's rows are not 16-byte aligned (no TMA stores):
    4096 x 14336 x 4096 BF16 takes 256 x 512 tiles with ldc = N and
    256 x 256 tiles with ldc = N + 1. Sampled rows checked in both layouts."""
    M, N, K = 4096, 14336, 4096
    g = inputs.generator(4242)
    A = inputs.draw(M, K, "normal002", g).to(torch.bfloat16)
    B = inputs.draw(K, N, "normal002", g).to(torch.bfloat16)
    Ad, Bd = A.cuda(), B.cuda()
    rows = [0, 255, 256, 4095] + torch.randint(0, M, (4,), generator=g).tolist()
    C_ref, absAB = oracle.gemm_rows(A, B, rows)
    for ldc, tile in ((N, "256x512"), (N + 1, "256x256")):
        C = torch.empty(M, ldc, device="cuda")[:, :N]
        tgemm.gemm_tc(Ad, Bd, "bf16", out=C)
        assert tgemm.device_status() == 0
        assert tile in tgemm.binding.last_kernel(), (ldc, tgemm.binding.last_kernel())
        assert_within(C.cpu()[rows], C_ref, absAB, TC_REL, TC_ABS, f"ldc={ldc}")
        del C
