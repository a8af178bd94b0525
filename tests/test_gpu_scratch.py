"""Per-call scratch of the product entry points, as gemm_scratch_bytes reports it.

The library draws stream-ordered scratch from its own pool for operands it
rewrites (TF32's B transposed, repacked unaligned rows, TF32X3's high/low
copies) and for the partial tiles of a last wave split along K; a call that
needs neither allocates nothing. These tests pin the sizes the query reports
for each case against the rule written in the header, and run each product to
check that the planned call gives the oracle's result.
"""
import re

import pytest
import torch

import oracle
from tests.parity import assert_bit_exact
from tiled_matrix_multiplication_sm_gb300 import inputs

pytestmark = pytest.mark.gpu


def num_sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


def int_operands(M, N, K, dtype, seed):
    g = inputs.generator(seed)
    return (inputs.draw(M, K, "int4", g).to(dtype).cuda(),
            inputs.draw(K, N, "int4", g).to(dtype).cuda())


def round_up(x, m):
    return (x + m - 1) // m * m


def check_product(tg, A, B, path):
    C = tg.binding.gemm_ex(A, B, path)
    assert tg.device_status() == 0
    assert_bit_exact(C, oracle.gemm(A.cpu(), B.cpu())[0], f"{path} {tuple(A.shape)}")


def test_f32_whole_waves_allocate_nothing(tgemm):
    """128 x 256 tiles filling exactly one wave, 16-byte rows: no scratch."""
    sms = num_sms()
    assert sms % 8 == 0
    M, N, K = 128 * (sms // 8), 256 * 8, 256
    A, B = int_operands(M, N, K, torch.float32, 1)
    assert tgemm.binding.scratch_bytes(A, B, "f32") == 0
    check_product(tgemm, A, B, "f32")


def test_f32_split_tail_draws_its_partials(tgemm):
    """4096^3: 512 tiles of 128 x 256 over the SMs; the last partial wave is
    split along K and its partial tiles are the whole scratch."""
    A = torch.empty(4096, 4096, device="cuda")
    n = tgemm.binding.scratch_bytes(A, A, "f32")
    tile = 128 * 256 * 4
    rem = 512 % num_sms()
    assert n > 0 and n % tile == 0
    assert n // tile % rem == 0                      # rem tiles x split pieces
    if num_sms() == 152:
        assert n == 56 * 8 * tile                    # 59 MB, as the header states


def test_bf16_whole_waves_allocate_nothing(tgemm):
    """256 x 256 pair tiles filling exactly one round of SM pairs."""
    pairs = num_sms() // 2
    assert pairs % 4 == 0
    M, N, K = 256 * 4, 256 * (pairs // 4), 512
    A, B = int_operands(M, N, K, torch.bfloat16, 2)
    tgemm.binding.set_tc_kernel(1)
    try:
        assert tgemm.binding.scratch_bytes(A, B, "bf16") == 0
        check_product(tgemm, A, B, "bf16")
    finally:
        tgemm.binding.set_tc_kernel(-1)


def streamk_bytes(name):
    """Scratch of a shared tail named in a last-kernel record: for stream-K,
    one partial tile per sharing slot, then one counter per tail tile; for
    the split form (k shares a tile, a reduction kernel), k partial tiles
    per tail tile and no counters."""
    m = re.search(r"(\d+)x(\d+)x\d+_s\d+(?:_btrans)?_persistent\(streamk:slots=(\d+),tiles=(\d+)\)", name)
    if m:
        rows, cols, slots, tiles = (int(x) for x in m.groups())
        if "2sm" in name:
            rows = 256
        return round_up(slots * rows * cols * 4, 256) + round_up(tiles * 4, 256)
    m = re.search(r"(\d+)x(\d+)x\d+_s\d+(?:_btrans)?_persistent\+tc_split_reduce\(split=(\d+),tiles=(\d+)\)",
                  name)
    if m:
        rows, cols, k, tiles = (int(x) for x in m.groups())
        if "2sm" in name:
            rows = 256
        return round_up(k * tiles * rows * cols * 4, 256)
    return 0


def test_tf32_reads_b_as_stored(tgemm):
    """TF32 with B's rows on 16-byte boundaries reads B MN-major as stored:
    no scratch beyond the shared tail's partial tiles (and stream-K
    counters) when the planner shares the two tiles among SM pairs."""
    M, N, K = 200, 300, 1000
    A, B = int_operands(M, N, K, torch.float32, 3)
    n = tgemm.binding.scratch_bytes(A, B, "tf32")
    check_product(tgemm, A, B, "tf32")
    name = tgemm.binding.last_kernel()
    assert "transpose_b" not in name and "repack" not in name, name
    assert n == streamk_bytes(name), name


@pytest.mark.parametrize("M", [16, 100])
def test_tf32_few_rows_read_b_in_place(tgemm, M):
    """TF32 with at most 128 rows of A: no scratch beyond a stream-K tail's,
    with the default kernel and with the one that transposes B's blocks in
    shared memory (mode 3)."""
    N, K = 1000, 512
    A, B = int_operands(M, N, K, torch.float32, 6)
    for mode in (-1, 3):
        assert tgemm.binding.set_tc_kernel(mode) == 0
        try:
            n = tgemm.binding.scratch_bytes(A, B, "tf32")
            check_product(tgemm, A, B, "tf32")
            name = tgemm.binding.last_kernel()
        finally:
            tgemm.binding.set_tc_kernel(-1)
        assert ("btrans" in name) == (mode == 3) and "transpose_b" not in name, name
        assert n == streamk_bytes(name), name


def test_unaligned_rows_are_repacked(tgemm):
    """BF16 with rows off 16 bytes: A (lda = K = 1001) and B (ldb = N = 301)
    repacked to 128-byte rows."""
    M, N, K = 200, 301, 1001
    A, B = int_operands(M, N, K, torch.bfloat16, 4)
    want = round_up(M * round_up(K, 64) * 2, 256) + round_up(K * round_up(N, 64) * 2, 256)
    n = tgemm.binding.scratch_bytes(A, B, "bf16")
    check_product(tgemm, A, B, "bf16")
    assert n == want + streamk_bytes(tgemm.binding.last_kernel()), tgemm.binding.last_kernel()


def test_forced_stream_k_draws_partials_and_counters(tgemm):
    """256 x 256 pair tiles, 6 tiles shared by 40 pairs: 40 partial tiles and
    6 counters (rows of A and B on 16-byte boundaries: nothing repacked)."""
    M, N, K = 300, 704, 1032
    A, B = int_operands(M, N, K, torch.bfloat16, 5)
    tgemm.binding.set_tc_kernel(1)
    tgemm.binding.set_tc_streamk(40)
    try:
        n = tgemm.binding.scratch_bytes(A, B, "bf16")
        check_product(tgemm, A, B, "bf16")
        name = tgemm.binding.last_kernel()
    finally:
        tgemm.binding.set_tc_kernel(-1)
        tgemm.binding.set_tc_streamk(-1)
    assert "streamk:slots=40,tiles=6" in name, name
    assert n == round_up(40 * 256 * 256 * 4, 256) + 256
