"""Stream-K tails of the tensor-core kernels.

When a product's tiles do not fill whole rounds of the SMs (one-SM kernel)
or SM pairs, the K blocks of the partial last round can be shared evenly by
S of them inside the same launch. A share that does not end its tile leaves
a raw partial tile in scratch and raises the tile's counter. The share that
ends a tile waits (bounded) for the counter. It then adds the partial tiles
of the shares before it, in a fixed order, and stores the tile. These tests
force S (gemm_set_tc_streamk) on every kernel shape and input type. The
widths go up to many shares per tile, and a whole round of tiles precedes
the tail in one case. Every result is checked against the oracle: bit for bit
on integer data, within the path's tolerance on random data.
"""
import re
import threading

import pytest
import torch

import oracle
from tests.parity import F32_ABS, F32_REL, TC_ABS, TC_REL, assert_bit_exact, assert_within
from tiled_matrix_multiplication_sm_gb300 import inputs

pytestmark = pytest.mark.gpu

DTYPES = {"tf32": torch.float32, "bf16": torch.bfloat16, "tf32x3": torch.float32}


def forced(tg, mode, slots, fn):
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


def streamk_slots(name):
    m = re.search(r"streamk:slots=(\d+),tiles=(\d+)", name)
    return (int(m.group(1)), int(m.group(2))) if m else None


# (mode, M, N, K): tile counts below one round, a ragged edge in every
# dimension, and one case with a whole round of 256 x 256 tiles before the tail.
SHAPES = [(0, 100, 1000, 2048),        # one SM: 4 tiles of 128 x 256
          (1, 300, 700, 1032),         # pair: 2 x 3 tiles of 256 x 256, ragged K
          (2, 512, 1500, 2048),        # pair, wide: 2 x 3 tiles of 256 x 512
          (1, 2304, 2304, 512)]        # pair: 81 tiles = one round of 76 + 5


@pytest.mark.parametrize("kind", ["tf32", "bf16"])
@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("slots", [7, 33, 152])
def test_integer_bit_exact(tgemm, kind, shape, slots):
    mode, M, N, K = shape
    g = inputs.generator(M + 7 * N + K + slots)
    A = inputs.draw(M, K, "int4", g).to(DTYPES[kind])
    B = inputs.draw(K, N, "int4", g).to(DTYPES[kind])
    C, name = forced(tgemm, mode, slots, lambda: tgemm.gemm_tc(A.cuda(), B.cuda(), kind))
    sk = streamk_slots(name)
    assert sk is not None, name
    assert sk[0] <= slots and sk[0] > sk[1], name
    assert_bit_exact(C, oracle.gemm(A, B)[0], f"{kind} {shape} S={slots} {name}")


@pytest.mark.parametrize("kind", ["tf32", "bf16", "tf32x3"])
def test_random_within_tolerance_unaligned_c(tgemm, kind):
    """Random data, C rows off 16 bytes (ldc = N + 1: the owners store from
    registers), a ragged product on 256 x 256 pair tiles shared by 40 pairs."""
    M, N, K = 300, 700, 1032
    g = inputs.generator(4242)
    dist = "normal002" if kind == "bf16" else "normal"
    A = inputs.draw(M, K, dist, g).to(DTYPES[kind])
    B = inputs.draw(K, N, dist, g).to(DTYPES[kind])
    store = torch.full((M, N + 1), float("nan"), device="cuda")
    C = store[:, :N]
    _, name = forced(tgemm, 1, 40, lambda: tgemm.gemm_tc(A.cuda(), B.cuda(), kind, out=C))
    assert streamk_slots(name) is not None, name
    assert torch.isnan(store[:, N]).all()           # the padding column is never written
    C_ref, absAB = oracle.gemm(A, B)
    rel, abs_ = (F32_REL, F32_ABS) if kind == "tf32x3" else (TC_REL, TC_ABS)
    assert_within(C, C_ref, absAB, rel, abs_, f"{kind} stream-K unaligned C")


def test_two_streams_at_once(tgemm):
    """Two stream-K products in flight together on two streams (their SMs
    interleave): every owner's wait is on shares of lower index, which were
    dispatched first, so both finish and match the oracle."""
    g = inputs.generator(5151)
    A = inputs.draw(300, 1032, "int4", g)
    B = inputs.draw(1032, 700, "int4", g)
    C_ref = oracle.gemm(A, B)[0]
    Ad, Bd = A.cuda(), B.cuda()
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    outs = [torch.empty(300, 700, device="cuda") for _ in range(4)]
    assert tgemm.binding.set_tc_kernel(1) == 0
    assert tgemm.binding.set_tc_streamk(76) == 0
    try:
        for i, out in enumerate(outs):
            with torch.cuda.stream(streams[i % 2]):
                tgemm.gemm_tc(Ad, Bd, "tf32", out=out)
        torch.cuda.synchronize()
    finally:
        tgemm.binding.set_tc_kernel(-1)
        tgemm.binding.set_tc_streamk(-1)
    assert tgemm.device_status() == 0
    for i, out in enumerate(outs):
        assert_bit_exact(out, C_ref, f"stream {i % 2} call {i}")


def test_automatic_choice_is_exact(tgemm):
    """The planner's own choice on the 4096^3 TF32 shape (128 wide tiles over
    76 pairs) on integer data."""
    g = inputs.generator(777)
    A = inputs.draw(4096, 4096, "int4", g)
    B = inputs.draw(4096, 4096, "int4", g)
    C = tgemm.gemm_tc(A.cuda(), B.cuda(), "tf32")
    assert tgemm.device_status() == 0
    rows = list(range(0, 4096, 97)) + [4095]
    C_ref, _ = oracle.gemm_rows(A, B, rows)
    assert_bit_exact(C.cpu()[rows], C_ref, f"4096^3 {tgemm.binding.last_kernel()}")


# ---------------------------------------------------------------- the split form

@pytest.mark.parametrize("kind", ["tf32", "bf16"])
@pytest.mark.parametrize("mode,shape,k", [(1, (300, 700, 1032), 4), (1, (2304, 2304, 512), 2),
                                          (2, (512, 1500, 2048), 3), (0, (100, 1000, 2048), 6),
                                          (1, (389, 301, 97), 2), (3, (100, 1000, 2048), 5),
                                          (4, (100, 1000, 2048), 7)])
def test_split_form_integer_bit_exact(tgemm, kind, mode, shape, k):
    """The tail tiles in k equal shares that wait for nothing, summed in K
    order by the reduction kernel (which also stores rows and columns past
    the shares' tiles exactly once)."""
    M, N, K = shape
    g = inputs.generator(M + 3 * N + K + k)
    A = inputs.draw(M, K, "int4", g).to(DTYPES[kind])
    B = inputs.draw(K, N, "int4", g).to(DTYPES[kind])
    C, name = forced(tgemm, mode, -k, lambda: tgemm.gemm_tc(A.cuda(), B.cuda(), kind))
    m = re.search(r"\+tc_split_reduce\(split=(\d+),tiles=(\d+)\)", name)
    assert m is not None, name
    assert_bit_exact(C, oracle.gemm(A, B)[0], f"{kind} {shape} split {k}")


@pytest.mark.parametrize("kind", ["tf32", "bf16"])
def test_split_form_full_output_rule_and_guard_bands(tgemm, kind):
    """alpha, beta and bias applied once per element by the reduction; C
    rows off 16-byte boundaries; the padding and guard bands untouched."""
    M, N, K = 512, 1530, 2048
    g = inputs.generator(91)
    A = inputs.draw(M, K, "int4", g).to(DTYPES[kind])
    B = inputs.draw(K, N, "int4", g).to(DTYPES[kind])
    C0 = inputs.draw(M, N, "int4", g)
    bias = inputs.draw(1, N, "int4", g)[0]
    ldc, guard = N + 3, 64
    store = torch.full((guard + M * ldc + guard,), -99.0, device="cuda")
    C = store[guard:guard + M * ldc].view(M, ldc)[:, :N]
    C.copy_(C0.cuda())
    _, name = forced(tgemm, 1, -3, lambda: tgemm.binding.gemm_ex(A.cuda(), B.cuda(), kind, alpha=2.0,
                                                                  beta=-1.0, bias=bias.cuda(), out=C))
    assert "+tc_split_reduce(split=3," in name, name
    ref, _ = oracle.gemm_ex(A, B, alpha=2.0, beta=-1.0, C0=C0, bias=bias)
    assert_bit_exact(C, ref, f"{kind} split rule")
    host = store.cpu()
    assert (host[:guard] == -99.0).all() and (host[guard + M * ldc:] == -99.0).all()
    assert (host[guard:guard + M * ldc].view(M, ldc)[:, N:] == -99.0).all()


def test_split_form_float_deterministic(tgemm):
    M, N, K = 600, 1000, 1537
    g = inputs.generator(92)
    A = inputs.draw(M, K, "normal", g)
    B = inputs.draw(K, N, "normal", g)
    Ad, Bd = A.cuda(), B.cuda()
    outs = []
    for _ in range(4):
        C, name = forced(tgemm, 1, -4, lambda: tgemm.gemm_tc(Ad, Bd, "tf32"))
        outs.append(C)
    assert "+tc_split_reduce(split=4," in name, name
    C_ref, absAB = oracle.gemm(A, B)
    assert_within(outs[0], C_ref, absAB, TC_REL, TC_ABS, "split float")
    for C in outs[1:]:
        assert torch.equal(C, outs[0])
