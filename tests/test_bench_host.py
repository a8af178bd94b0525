"""Host-side logic of bench.py (no GPU): roofline arithmetic, clock-sample
parsing, the committed-traffic lookup and the max-over-ranks aggregation
across processes (gloo, world size 2)."""
import json
import os

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def test_fp32_peak_from_unit_counts():
    # 152 SMs x 128 lanes x 2 FLOP x 2070 MHz
    assert bench.fp32_peak_tflops(152, 2070.0) == pytest.approx(80.5478, rel=1e-6)


def test_pipe_peak_and_algorithmic_bytes():
    probe = {"bf16": {"flop_per_clk_per_sm": 8192.0}, "tf32": {"flop_per_clk_per_sm": 4096.0}}
    # 8192 FLOP/clk/SM x 152 SMs x 2070 MHz = 2577.5 TFLOP/s
    assert bench.pipe_peak_tflops(probe, "bf16", 152, 2070.0) == pytest.approx(2577.5, rel=1e-4)
    # the split-TF32 form runs TF32 MMAs
    assert bench.pipe_peak_tflops(probe, "tf32x3", 152, 2070.0) == pytest.approx(1288.7, rel=1e-4)
    from tiled_matrix_multiplication_sm_gb300 import inputs
    w = inputs.WORKLOADS["skinny_bf16"]
    # A and B read once (bf16), C written once (fp32)
    assert bench.algorithmic_bytes(w) == 2 * (16 * 4096 + 4096 * 14336) + 4 * 16 * 14336
    assert bench.algorithmic_bytes(inputs.WORKLOADS["skinny_f32"]) == \
        4 * (16 * 4096 + 4096 * 14336) + 4 * 16 * 14336


def test_load_peaks_fallback(tmp_path):
    p = bench.load_peaks(str(tmp_path / "missing.json"))
    assert p["source"] == "fallback" and p["hbm_gbs"] == 6800.0
    f = tmp_path / "peaks.json"
    f.write_text(json.dumps({"hbm_gbs": 1.0, "bf16_tflops": 2.0, "sm_max_mhz": 3.0}))
    p = bench.load_peaks(str(f))
    assert p["source"] == "measured" and p["bf16_tflops_sustained"] == 2.0


def test_parse_clock_samples():
    rows = ["1965, 2070, 900.5, 0x0, Not Active, Not Active, Not Active, Not Active",
            "1447, 2070, 1380.0, 0x4, Not Active, Not Active, Not Active, Active",
            "1500, 2070, 1390.0, 0x4, Not Active, Not Active, Not Active, Active",
            "garbage line"]
    s = bench.parse_clock_samples(rows)
    assert s["samples"] == 3 and s["sm_mhz"] == 1500 and s["sm_max_mhz"] == 2070
    assert s["reasons"] == ["sw_power_cap"]
    assert bench.parse_clock_samples([])["sm_mhz"] is None


def test_committed_traffic_requires_matching_source(tmp_path):
    src = tmp_path / "k.cu"
    src.write_text("kernel v1")
    recs = tmp_path / "ncu"
    recs.mkdir()
    rec = {"source": "k.cu", "source_sha256": bench.file_sha256(str(src)),
           "derived": {"dram_bytes": 123456}}
    (recs / "sgemm_kernel__n4096_f32__0_f32_128x256.json").write_text(json.dumps(rec))
    assert bench.committed_traffic(str(recs), root=str(tmp_path)) == 123456
    src.write_text("kernel v2")
    assert bench.committed_traffic(str(recs), root=str(tmp_path)) is None
    assert bench.committed_traffic(str(tmp_path / "none"), root=str(tmp_path)) is None


def test_aggregate_uses_slowest_rank():
    v, t = bench.aggregate([2.0, 4.0], 100.0)
    assert t == 4.0 and v == 50.0


def test_args_force_three_warmups():
    a = bench.parse_args(["--warmup", "1", "--steps", "7"])
    assert a.warmup == 3 and a.steps == 7 and a.impl == "ours"


def _rank_main(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port),
                      RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ws, r, _ = bench.dist_env()
    assert (ws, r) == (world, rank)
    local_seconds = 1.0 + rank           # rank 1 is the slowest
    bench.barrier(ws)
    t = bench.max_over_ranks(local_seconds, ws)
    value, tmax = bench.aggregate([t] * ws, 10.0)
    with open(os.path.join(out_dir, f"r{rank}.json"), "w") as f:
        json.dump({"t": t, "value": value}, f)
    dist.destroy_process_group()


def test_max_over_ranks_gloo(tmp_path):
    import socket
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    mp.spawn(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, join=True)
    for r in range(2):
        d = json.loads((tmp_path / f"r{r}.json").read_text())
        assert d["t"] == 2.0                 # the slowest rank's time everywhere
        assert d["value"] == pytest.approx(10.0)   # 2 ranks x 10 units / 2 s
