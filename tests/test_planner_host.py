"""The planner's choices, pinned on the host (no GPU).

gemm_plan_name reports the kernels a call would launch on a device with a
given SM count, in gemm_last_kernel's form, without touching the GPU. Each
expected name below is what the library chose and ran on a GB300 (152 SMs)
for that workload -- choices measured against the alternatives (tile
shape, stream-K or split width, pre-passes) -- so a change to the timing
model or the tile tables that moves any of them fails here first.
"""
import pytest

from tiled_matrix_multiplication_sm_gb300 import binding

ALIGNED = 256          # a 16-byte-aligned stand-in address (never dereferenced)
SMS = 152


def plan(M, N, K, path, lda=None, ldb=None, ldc=None, trans_a=False, trans_b=False, sms=SMS):
    lda = lda or (M if trans_a else K)
    ldb = ldb or (K if trans_b else N)
    return binding.plan_name_raw(M, N, K, ALIGNED, lda, ALIGNED, ldb, ALIGNED, ldc or N, path,
                                 trans_a=trans_a, trans_b=trans_b, num_sms=sms)


MEASURED = [
    # FP32 CUDA cores
    ((128, 128, 128, "f32"), "f32_64x64x16_s4_ffma_vecA_vecB"),
    ((1024, 1024, 1024, "f32"), "f32_128x256x32_s3_ffma2_vecA_vecB+splitk_reduce(split=4,tiles=32)"),
    ((4096, 4096, 4096, "f32"), "f32_128x256x32_s3_ffma2_vecA_vecB+splitk_reduce(split=8,tiles=56)"),
    ((3000, 5001, 1537, "f32"),
     "repack_ab+f32_128x256x32_s3_ffma2_vecA_vecB+splitk_reduce(split=6,tiles=24)"),
    ((16, 14336, 4096, "f32"), "f32_16x256x32_s3_ffma2_2blk_vecA_vecB+splitk_reduce(split=5,tiles=56)"),
    # tcgen05 TF32 (B read MN-major as stored)
    ((4096, 4096, 4096, "tf32"), "tc_tf32_2sm_256x512x32_s4_persistent(streamk:slots=76,tiles=52)"),
    ((3000, 5001, 1537, "tf32"),
     "repack_ab+tc_tf32_2sm_256x256x32_s6_persistent+tc_split_reduce(split=6,tiles=12)"),
    ((512, 1500, 2048, "tf32"), "tc_tf32_2sm_256x256x32_s6_persistent+tc_split_reduce(split=6,tiles=12)"),
    ((16, 14336, 4096, "tf32"), "tc_tf32_128x256x32_s4_persistent(streamk:slots=112,tiles=56)"),
    ((16, 4096, 14336, "tf32"), "tc_tf32_128x128x32_s6_persistent(streamk:slots=128,tiles=32)"),
    # tcgen05 TF32X3 (split form)
    ((4096, 4096, 4096, "tf32x3"),
     "split_a+transpose_split_b+tc_tf32x3_2sm_256x256x32_s3_persistent(streamk:slots=75,tiles=28)"),
    # tcgen05 BF16
    ((8192, 14336, 4096, "bf16"), "tc_bf16_2sm_256x512x64_s4_persistent"),
    ((16, 14336, 4096, "bf16"), "tc_bf16_128x128x64_s6_persistent"),
    ((16, 28672, 4096, "bf16"), "tc_bf16_128x256x64_s4_persistent"),
    ((16, 4096, 4096, "bf16"), "tc_bf16_128x128x64_s6_persistent(streamk:slots=96,tiles=32)"),
]


@pytest.mark.parametrize("args,expected", MEASURED, ids=[f"{a[3]}-{a[0]}x{a[1]}x{a[2]}" for a, _ in MEASURED])
def test_measured_choices(args, expected):
    M, N, K, path = args
    assert plan(M, N, K, path) == expected


def test_transposed_storage_pre_passes():
    # A stored K x M -> transposed for the tensor paths; B stored N x K is
    # read K-major with no copy.
    assert plan(3000, 3000, 2048, "tf32", trans_a=True) == \
        "transpose_a+tc_tf32_2sm_256x512x32_s4_persistent"
    assert "transpose" not in plan(3000, 3000, 2048, "tf32", trans_b=True)
    # FP32 reads B row-major: stored transposed -> transposed first.
    assert plan(1024, 1024, 1024, "f32", trans_b=True).startswith("transpose_b+")


def test_unaligned_rows_pick_the_right_repacks():
    assert plan(300, 512, 517, "bf16").startswith("repack_a+")           # lda = 517 (2-byte)
    assert plan(300, 517, 512, "bf16").startswith("repack_b+")           # ldb = 517
    assert plan(300, 517, 517, "bf16").startswith("repack_ab+")
    assert "repack" not in plan(300, 520, 520, "bf16")


def test_degenerate_shapes():
    assert plan(0, 100, 100, "tf32") == ""
    assert plan(100, 0, 100, "f32") == ""
    assert plan(100, 100, 0, "bf16") == "empty_product"


def test_settings_are_honoured():
    b = binding
    try:
        assert b.set_tc_kernel(1) == 0
        assert plan(4096, 4096, 4096, "tf32").startswith("tc_tf32_2sm_256x256x32_s6_persistent")
        assert b.set_tc_kernel(3) == 0
        assert plan(100, 1000, 512, "tf32").startswith("tc_tf32_128x128x32_s6_btrans_persistent")
        assert b.set_tc_kernel(-1) == 0
        assert b.set_tc_streamk(0) == 0
        assert plan(4096, 4096, 4096, "tf32") == "tc_tf32_2sm_256x512x32_s4_persistent"
        assert b.set_tc_kernel(1) == 0                  # 256 x 256 pair tiles, tail in 3 shares
        assert b.set_tc_streamk(-3) == 0
        assert plan(3000, 5001, 1537, "tf32").endswith("+tc_split_reduce(split=3,tiles=12)")
    finally:
        b.set_tc_kernel(-1)
        b.set_tc_streamk(-1)


def test_the_sm_count_drives_the_plan():
    # Fewer SMs: the same FP32 product fills waves differently.
    assert plan(4096, 4096, 4096, "f32", sms=152) != plan(4096, 4096, 4096, "f32", sms=132)


def test_invalid_arguments():
    with pytest.raises(binding.TgemmError):
        plan(16, 16, 16, "f32", sms=1)
    with pytest.raises(binding.TgemmError):
        plan(16, 16, 16, "f32", lda=8)            # lda < K


TOKEN = (r"(repack_ab|repack_a|repack_b|transpose_a|transpose_b|split_a|split_b|transpose_split_a|"
         r"transpose_split_b)")


def test_random_problems_always_plan():
    """Random shapes, paths, storage, alignment and SM counts (including
    counts no GB300 has): every valid call gets a plan whose name is made of
    known parts, and the tensor paths keep one-SM tiles for M <= 128."""
    import random
    import re
    rng = random.Random(20262)
    name_re = re.compile(rf"^(?:{TOKEN}\+)*(?:f32_\w+|tc_\w+)(?:\(a_loader\))?"
                         r"(?:\(streamk:slots=\d+,tiles=\d+\)|\+(?:tc_split_reduce|splitk_reduce)"
                         r"\(split=\d+,tiles=\d+\))?$")
    for _ in range(3000):
        path = rng.choice(["f32", "tf32", "bf16", "tf32x3"])
        M = rng.choice([1, 2, 15, 16, 17, 127, 128, 129, 255, 256, 257]) if rng.random() < 0.4 \
            else rng.randint(1, 20000)
        N = rng.randint(1, 30000)
        K = rng.choice([1, 7, 8, 31, 32, 33, 4096]) if rng.random() < 0.3 else rng.randint(1, 20000)
        ta, tb = rng.random() < 0.2, rng.random() < 0.2
        pad = lambda: rng.choice([0, 0, 0, 1, 3, 8])
        lda = (M if ta else K) + pad()
        ldb = (K if tb else N) + pad()
        sms = rng.choice([2, 8, 76, 132, 148, 152])
        name = plan(M, N, K, path, lda=lda, ldb=ldb, ldc=N + pad(), trans_a=ta, trans_b=tb, sms=sms)
        assert name_re.match(name), (path, M, N, K, ta, tb, lda, ldb, sms, name)
        if path != "f32" and M <= 128 and path != "tf32x3":
            assert "2sm" not in name, (path, M, N, K, name)
