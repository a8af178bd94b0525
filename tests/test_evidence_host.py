"""Host-side logic of the ncu evidence harness (no GPU, no ncu): parsing of
ncu's raw CSV, pairing of profiled launches with the library's kernel names,
algorithmic work and roofline fractions of each kind of kernel."""
import json

import pytest

from tiled_matrix_multiplication_sm_gb300 import evidence

RAW = '''"ID","Kernel Name","gpu__time_duration.sum","dram__bytes_read.sum","dram__bytes_write.sum","sm__cycles_elapsed.avg.per_second","l1tex__data_bank_conflicts_pipe_lsu_mem_shared_op_ld.sum"
"","","nsecond","byte","byte","hz",""
"0","void tgemm::(anonymous namespace)::transpose_kernel<float>(const T1 *, long, T1 *, long, int, int)","20,000","67,108,864","67,108,864","2,070,000,000","0"
"1","void tgemm::(anonymous namespace)::tc_gemm_2sm_kernel<4, true, false, 2>(CUtensorMap, CUtensorMap)","160,000","134,217,728","67,108,864","2,000,000,000","12"
'''


def test_parse_raw_csv_drops_units_row_and_commas():
    rows = evidence.parse_raw_csv("==PROF== noise\n" + RAW)
    assert len(rows) == 2
    assert evidence.number(rows[0]["gpu__time_duration.sum"]) == 20000.0
    assert evidence.short_name(rows[1]["Kernel Name"]) == "tc_gemm_2sm_kernel"
    assert evidence.source_of(rows[0]["Kernel Name"]) == "transpose_f32.cu"
    assert evidence.source_of(rows[1]["Kernel Name"]) == "gemm_tcgen05.cu"


def test_short_names_of_ncu_renderings():
    for raw in ["void unnamed>::repack_kernel<float>(const T1 *, long, T1 *, long, int, int)",
                "unnamed>::tc_splitk_reduce(unnamed>::TcParams)",
                "void tgemm::<unnamed>::tc_gemm_2sm_kernel<4, 1, 0, 1>(CUtensorMap_st, "
                "unnamed>::TcParams)",
                "void unnamed>::sgemm_kernel<unnamed>::Tile<128, 256, 32, 32, 128, 3, 1, 1>, 1, "
                "1>(unnamed>::F32Params)",
                "void tgemm::(anonymous namespace)::splitk_reduce<tgemm::(anonymous namespace)::"
                "Tile<1, 2>>(tgemm::(anonymous namespace)::F32Params)"]:
        assert evidence.short_name(raw) in ("repack_kernel", "tc_splitk_reduce",
                                            "tc_gemm_2sm_kernel", "sgemm_kernel",
                                            "splitk_reduce"), raw


def test_records_pair_launches_with_library_names():
    rows = evidence.parse_raw_csv(RAW)
    peaks = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "sm_max_mhz": 2070.0, "source": "test"}
    recs = evidence.make_records(rows, ["transpose_b", "tc_tf32_2sm_256x512x32_s4_persistent"],
                                 "n4096:tf32", "cmd", "ncu cmd", peaks, 152)
    t, g = recs
    # transpose: 8 K N bytes algorithmic, 134 MB in 20 us = 6710.9 GB/s
    assert t["roofline"]["bound"] == "hbm"
    assert t["roofline"]["algorithmic_bytes"] == 8 * 4096 * 4096
    assert t["roofline"]["achieved"] == pytest.approx(8 * 4096 ** 2 / 20000, rel=1e-3)
    assert t["roofline"]["traffic_over_algorithmic"] == pytest.approx(1.0)
    # GEMM: 2 M N K over 160 us against 1900 x 1.1 / 2.25
    assert g["roofline"]["bound"] == "tensor"
    assert g["roofline"]["achieved"] == pytest.approx(2 * 4096 ** 3 / 160000 / 1e3, rel=1e-3)
    assert g["roofline"]["peak"] == pytest.approx(1900 * 1.1 / 2.25, rel=1e-3)
    assert g["metrics"]["l1tex__data_bank_conflicts_pipe_lsu_mem_shared_op_ld.sum"] == 12
    assert evidence.record_filename(g).startswith("tc_gemm_2sm_kernel__n4096_tf32__1_")
    json.dumps(recs)


def test_algorithmic_work_of_each_kind():
    w = evidence.algorithmic_work
    assert w("repack_a", "ragged:tf32")["bytes"] == 2 * 3000 * 1537 * 4
    assert w("repack_b", "ragged:f32")["bytes"] == 2 * 1537 * 5001 * 4
    assert w("repack_ab", "ragged:tf32")["bytes"] == 2 * (3000 * 1537 + 1537 * 5001) * 4
    assert w("split_a", "n4096:tf32x3")["bytes"] == 12 * 4096 * 4096
    assert w("tc_tf32x3_2sm_256x256x32_s3_persistent", "n4096:tf32x3")["flop"] == 3 * 2 * 4096 ** 3
    assert w("f32_128x256x32_s3_ffma2_vecA_vecB", "u1024:f32") == {"bound": "alu",
                                                                   "flop": 2 * 1024 ** 3}
    assert w("empty_product", "k0:f32")["bytes"] == 4 * 4096 * 4096
    r = w("splitk_reduce(split=8,tiles=56)", "n4096:f32")
    assert (r["split"], r["tiles"], r["bytes_per_tile_elem"]) == (8, 56, 36)
    r = w("tc_split_reduce(split=6,tiles=12)", "ragged:tf32")
    assert (r["bound"], r["split"], r["tiles"], r["bytes_per_tile_elem"]) == ("hbm", 6, 12, 28)
    assert evidence.tile_elems("f32_128x256x32_s3_ffma2_vecA_vecB") == 128 * 256
    # The few-row workloads are stated against HBM: A + B read once, C written once.
    r = w("tc_bf16_128x256x64_s4_persistent(streamk:slots=112,tiles=56)", "skinny_bf16:bf16")
    assert r["bound"] == "hbm" and r["bytes"] == 2 * (16 * 4096 + 4096 * 14336) + 4 * 16 * 14336
    r = w("tc_tf32_128x128x32_s6_btrans_persistent", "skinny_f32:tf32")
    assert r["bound"] == "hbm" and r["bytes"] == 4 * (16 * 4096 + 4096 * 14336) + 4 * 16 * 14336
    assert w("f32_16x256x32_s3_ffma2_2blk_vecA_vecB", "skinny_f32:f32")["bound"] == "hbm"


def test_every_case_names_a_workload():
    for case in evidence.CASES:
        wl, path, M, N, K, dtype = evidence.case_shape(case)
        assert path in ("f32", "tf32", "bf16", "tf32x3")
        assert (wl is None) == (K == 0)


def test_code_hash_ignores_comments_and_layout_only(tmp_path):
    """A record stays current while only comments or layout change, and
    goes stale when the code does; "//" inside a string is code."""
    src = tmp_path / "k.cu"
    src.write_text('// header\n__global__ void k(float* p) {  /* body */\n'
                   '    const char* s = "a // b";\n    p[0] = 1.0f;  // store\n}\n')
    h = evidence.code_sha256(str(src))
    src.write_text('// a new header\n// more words\n__global__ void k(float* p) {\n'
                   '    const char* s = "a // b";   /* moved */\n        p[0] = 1.0f;\n}\n')
    assert evidence.code_sha256(str(src)) == h
    src.write_text('__global__ void k(float* p) {\n    const char* s = "a // c";\n    p[0] = 1.0f;\n}\n')
    assert evidence.code_sha256(str(src)) != h
    src.write_text('__global__ void k(float* p) {\n    const char* s = "a // b";\n    p[0] = 2.0f;\n}\n')
    assert evidence.code_sha256(str(src)) != h


def test_record_current_prefers_the_code_hash(tmp_path):
    src = tmp_path / "k.cu"
    src.write_text("int f() { return 1; } // v1\n")
    rec = {"source": "k.cu", "source_sha256": evidence.file_sha256(str(src)),
           "code_sha256": evidence.code_sha256(str(src))}
    assert evidence.record_current(rec, str(tmp_path))
    src.write_text("int f() { return 1; } // v2, a comment edit\n")
    assert evidence.record_current(rec, str(tmp_path))
    old = {"source": "k.cu", "source_sha256": rec["source_sha256"]}     # whole-file hash only
    assert not evidence.record_current(old, str(tmp_path))
    src.write_text("int f() { return 2; }\n")
    assert not evidence.record_current(rec, str(tmp_path))
    assert not evidence.record_current({"source": "gone.cu", "code_sha256": "x"}, str(tmp_path))
