"""Benchmark of the tiled GEMM library on one GB300 (or N replicas).

A step is one pass of the whole hot path over one batch of synthetic input:
the square 4096^3 product (A, B ~ N(0,1) fp32, row-major) computed once on
each path of the library -- the FP32 CUDA-core SGEMM (gemm_f32) and the
tcgen05 tensor-core GEMM in TF32 (gemm_tc; one kernel, B read MN-major as
stored). The metric is TFLOP/s = (2 M N K per product x 2 products) / device
time, timed with CUDA events on the launching stream, L2 flushed before
every timed step (a 256 MiB write, then a 256 MiB read of another buffer, so
that the timed kernels start on a cold L2 holding no dirty lines).

The JSON line also reports
  roofline     - for the dominant kernel (the FP32 SGEMM): achieved TFLOP/s
                 against the FP32 CUDA-core peak (SMs x 128 lanes x 2 FLOP x
                 the maximum SM clock), with DRAM traffic from the committed
                 ncu evidence record (profiles/ncu) when it matches the
                 current kernel source;
  paths        - each path's own TFLOP/s and roofline fraction in the step;
  workloads    - the other measured shapes: 1024^3 and 3000x5001x1537 on the
                 FP32 path, the FFN shape 8192x14336x4096 on the BF16 path;
  e2e          - the same step through the host API (pinned host operands
                 copied in, results copied out, inside the timed region);
  cpu_baseline - the CPU oracle (double-precision triple loop) on a sample of
                 rows of the same workload, on this host's cores;
  clocks       - nvidia-smi samples taken during the timed region.

``--impl reference`` times the CPU oracle as the reference arm instead.
Multi-GPU runs (torchrun, one rank per GPU) are independent replicas: the
product does not need any exchange between GPUs.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "GEMM TFLOP/s (2MNK/device time) and % of FP32 / tensor-core peak"
UNIT = "TFLOP/s"
WORKLOAD = "n4096"
FLUSH_BYTES = 256 * 1024 * 1024
NCU_RECORDS = os.path.join(ROOT, "profiles", "ncu")

# Nominal dense tensor rates (PFLOP/s) used to scale the measured BF16 peak to
# another input type: TF32 runs at 1.1 / 2.25 of the BF16 rate.
NOMINAL_TF32_OVER_BF16 = 1.1 / 2.25
FP32_LANES_PER_SM = 128


# ---------------------------------------------------------------- host logic

def fp32_peak_tflops(num_sms: int, sm_mhz: float) -> float:
    """CUDA-core FP32 peak: every lane retires one FMA (2 FLOP) per clock."""
    return num_sms * FP32_LANES_PER_SM * 2 * sm_mhz * 1e6 / 1e12


def load_peaks(path=os.path.join(ROOT, "MEASURED_PEAKS.json")):
    """Measured roofline denominators, or the documented fallback."""
    try:
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "sm_max_mhz": float(d.get("sm_max_mhz", 2070.0)), "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                "sm_max_mhz": 2070.0, "source": "fallback"}


def file_sha256(path: str) -> str:
    h = hashlib.sha256()
    with open(path, "rb") as f:
        h.update(f.read())
    return h.hexdigest()


def committed_traffic(records=NCU_RECORDS, case="n4096:f32", kernel="sgemm_kernel", root=ROOT):
    """DRAM bytes (read + write) of one launch of `kernel` in `case`, from the
    committed ncu evidence record, or None when there is none or the kernel's
    code changed since it was taken (comments aside)."""
    from tiled_matrix_multiplication_sm_gb300 import evidence
    rec = evidence.find_record(records, case, kernel)
    if rec is None or not rec.get("source"):
        return None
    try:
        if not evidence.record_current(rec, root):
            return None
        return int(rec["derived"]["dram_bytes"])
    except (OSError, KeyError, TypeError, ValueError):
        return None


SMI_FIELDS = ["clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active",
              "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]
REASON_NAMES = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]


def parse_clock_samples(lines):
    """Summarise nvidia-smi CSV rows (fields SMI_FIELDS, no header, no units)."""
    sm, mx, reasons = [], [], set()
    for line in lines:
        parts = [p.strip() for p in line.split(",")]
        if len(parts) < len(SMI_FIELDS):
            continue
        try:
            sm.append(float(parts[0]))
            mx.append(float(parts[1]))
        except ValueError:
            continue
        for name, val in zip(REASON_NAMES, parts[4:8]):
            if val.lower() == "active":
                reasons.add(name)
    if not sm:
        return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
    return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
            "reasons": sorted(reasons), "samples": len(sm)}


class ClockSampler:
    """nvidia-smi polling in the background while the timed region runs."""

    def __init__(self, uuid=None, period_ms=50):
        self.cmd = ["nvidia-smi", f"--query-gpu={','.join(SMI_FIELDS)}",
                    "--format=csv,noheader,nounits", f"-lms={period_ms}"]
        if uuid:
            self.cmd.append(f"--id={uuid}")
        self.proc = None
        self.lines = []
        self.thread = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(self.cmd, stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line)

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.thread.join(timeout=5)
        return False

    def summary(self):
        return parse_clock_samples(self.lines)


def aggregate(per_rank_seconds, units_per_rank):
    """Whole-job throughput: units all ranks processed / the slowest rank's time."""
    t = max(per_rank_seconds)
    return (units_per_rank * len(per_rank_seconds)) / t, t


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(value: float, ws: int, device=None) -> float:
    if ws == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(ws: int):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


# ---------------------------------------------------------------- CPU oracle

def oracle_rate(A, B, seconds_target: float, max_rows=None):
    """Time the CPU oracle on a seeded sample of rows sized to ~seconds_target;
    when every row fits in the target, the whole product is repeated.

    Returns (TFLOP/s, rows, seconds, threads, passes)."""
    import oracle
    import torch
    from tiled_matrix_multiplication_sm_gb300 import inputs

    threads = len(os.sched_getaffinity(0))
    oracle.set_threads(threads)
    M, K = A.shape
    N = B.shape[1]
    A64 = oracle.to_float64(A)
    B64 = oracle.to_float64(B)
    perm = torch.randperm(M, generator=inputs.generator(99)).tolist()
    probe = perm[: min(M, max(threads, 8))]
    t0 = time.perf_counter()
    oracle.gemm_rows(A64, B64, probe)
    t_probe = time.perf_counter() - t0
    per_row = t_probe / len(probe)
    want = int(seconds_target / max(per_row, 1e-9))
    cap = M if max_rows is None else max_rows
    rows = max(len(probe), min(want, cap))
    rows = (rows // threads) * threads or rows
    passes = max(1, int(round(want / cap))) if want > cap and cap == M else 1
    sample = sorted(perm[:rows])
    t0 = time.perf_counter()
    for _ in range(passes):
        oracle.gemm_rows(A64, B64, sample)
    dt = time.perf_counter() - t0
    return 2.0 * rows * passes * N * K / dt / 1e12, rows, dt, threads, passes


def oracle_workloads(inputs, threads):
    """The oracle on the other workloads, as the parity tests run it: the
    whole product, or the rows the tests check (the FFN shape's 256)."""
    import oracle
    res = {}
    for name, w in inputs.WORKLOADS.items():
        if name == "n4096":
            continue                           # the main figure above
        A, B = inputs.operands(w)
        A64, B64 = oracle.to_float64(A), oracle.to_float64(B)
        rows = inputs.check_rows(w).tolist()
        t0 = time.perf_counter()
        if len(rows) == w.M:
            oracle.gemm(A64, B64)
        else:
            oracle.gemm_rows(A64, B64, rows)
        dt = time.perf_counter() - t0
        res[name] = {"rows": len(rows), "seconds": round(dt, 3),
                     "tflops": round(2.0 * len(rows) * w.N * w.K / dt / 1e12, 6)}
    res["cores"] = threads
    return res


# ---------------------------------------------------------------- GPU arm

def event_pair():
    import torch
    return torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)


class L2Flush:
    """Leaves the 129 MB L2 cold and clean: a write of one buffer larger than
    L2 evicts everything, then a read of a second one evicts the written
    (dirty) lines, so that the next kernel neither hits in L2 nor pays for
    the write-back of the flush's own lines."""

    def __init__(self, device, nbytes=FLUSH_BYTES):
        import torch
        self.w = torch.empty(nbytes // 4, dtype=torch.float32, device=device)
        self.r = torch.zeros(nbytes // 4, dtype=torch.float32, device=device)

    def zero_(self):
        self.w.zero_()
        self.r.sum()


def time_calls(fn, reps, flush):
    """Median device time (ms) of fn() with L2 flushed before each call."""
    import torch
    times = []
    for _ in range(reps):
        flush.zero_()
        s, e = event_pair()
        s.record()
        fn()
        e.record()
        e.synchronize()
        times.append(s.elapsed_time(e))
    return statistics.median(times)


def run_gpu(args):
    import torch
    import tiled_matrix_multiplication_sm_gb300 as tg
    from tiled_matrix_multiplication_sm_gb300 import inputs

    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    tg.load()
    props = torch.cuda.get_device_properties(local)
    num_sms = props.multi_processor_count
    peaks = load_peaks()
    fp32_peak = fp32_peak_tflops(num_sms, peaks["sm_max_mhz"])
    tf32_peak = peaks["bf16_tflops"] * NOMINAL_TF32_OVER_BF16

    w = inputs.WORKLOADS[WORKLOAD]
    A_host, B_host = inputs.operands(w)
    A = A_host.to(dev)
    B = B_host.to(dev)
    C32 = torch.empty(w.M, w.N, device=dev)
    Ctf = torch.empty(w.M, w.N, device=dev)
    flush = L2Flush(dev)
    def step():
        tg.gemm_f32(A, B, out=C32)
        n32 = len(tg.binding.last_kernel().split("+"))
        tg.gemm_tc(A, B, "tf32", out=Ctf)
        return n32 + len(tg.binding.last_kernel().split("+"))

    for _ in range(args.warmup):
        launches_per_step = step()     # kernels of the library per step
    torch.cuda.synchronize()
    if tg.device_status() != 0:
        raise RuntimeError("a kernel wait timed out during warm-up")

    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    uuid = getattr(props, "uuid", None)
    uuid = f"GPU-{uuid}" if uuid is not None and not str(uuid).startswith("GPU-") else uuid
    barrier(ws)
    torch.cuda.synchronize()
    with ClockSampler(uuid) as sampler:
        for i in range(K):
            flush.zero_()
            ev[i][0].record()
            tg.gemm_f32(A, B, out=C32)
            ev[i][1].record()
            tg.gemm_tc(A, B, "tf32", out=Ctf)
            ev[i][2].record()
        torch.cuda.synchronize()
    barrier(ws)
    if tg.device_status() != 0:
        raise RuntimeError("a kernel wait timed out during the timed region")
    f32_ms = [e[0].elapsed_time(e[1]) for e in ev]
    tf32_ms = [e[1].elapsed_time(e[2]) for e in ev]
    step_s = sum(a + b for a, b in zip(f32_ms, tf32_ms)) / 1e3
    step_s = max_over_ranks(step_s, ws, dev)
    units = K * 2 * w.flops                      # FLOPs of K steps on one rank
    value, _ = aggregate([step_s] * ws, units)
    value /= 1e12
    f32_avg = statistics.mean(f32_ms)
    tf32_avg = statistics.mean(tf32_ms)
    f32_tflops = w.flops / (f32_avg * 1e-3) / 1e12
    tf32_tflops = w.flops / (tf32_avg * 1e-3) / 1e12
    clocks = sampler.summary()

    out = {
        "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": ws,
        "steps": K, "warmup": args.warmup, "ms_per_step": round(step_s * 1e3 / K, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": "square GEMM M=N=K=4096, A,B ~ N(0,1) fp32 row-major "
                               "(seed 20262); one product on the FP32 CUDA-core path and one on "
                               "the tcgen05 TF32 path per step",
                   "M": w.M, "N": w.N, "K": w.K, "paths": ["f32", "tf32"],
                   "l2": "flushed before every timed step: a 256 MiB write, then a 256 MiB "
                         "read of a second buffer (cold, clean L2)",
                   "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU"},
        "gpu_launches": K * launches_per_step,
        "roofline": {"bound": "alu", "kernel": "gemm_f32 (CUDA-core FFMA)",
                     "achieved": round(f32_tflops, 3), "peak": round(fp32_peak, 3),
                     "unit": "TFLOP/s", "frac": round(f32_tflops / fp32_peak, 4),
                     "traffic": committed_traffic(),
                     "peak_basis": f"{num_sms} SMs x {FP32_LANES_PER_SM} FP32 lanes x 2 FLOP x "
                                   f"{peaks['sm_max_mhz']:.0f} MHz (max SM clock)"},
        "paths": {
            "f32": {"ms": round(f32_avg, 4), "tflops": round(f32_tflops, 3),
                    "peak": round(fp32_peak, 3), "frac": round(f32_tflops / fp32_peak, 4),
                    "bound": "alu"},
            "tf32": {"ms": round(tf32_avg, 4), "tflops": round(tf32_tflops, 3),
                     "peak": round(tf32_peak, 3), "frac": round(tf32_tflops / tf32_peak, 4),
                     "bound": "tensor",
                     "peak_basis": f"measured bf16 {peaks['bf16_tflops']} x nominal tf32/bf16 "
                                   f"{NOMINAL_TF32_OVER_BF16:.3f} ({peaks['source']})"},
        },
        "clocks": {"sm_mhz": clocks["sm_mhz"], "sm_max_mhz": clocks["sm_max_mhz"],
                   "reasons": clocks["reasons"], "samples": clocks["samples"]},
    }

    if not args.no_extras:
        probe = run_tensor_probe(tg, dev, peaks)
        out["tensor_probe"] = probe
        if clocks["sm_mhz"]:
            pipe = pipe_peak_tflops(probe, "tf32", num_sms, clocks["sm_mhz"])
            out["paths"]["tf32"]["frac_vs_pipe"] = round(tf32_tflops / pipe, 4)
            out["paths"]["tf32"]["pipe_peak"] = round(pipe, 1)
        out["e2e"] = run_e2e(tg, A_host, B_host, w, dev, max(3, min(K, 20)))
        out["workloads"] = run_workloads(tg, inputs, dev, flush, peaks, fp32_peak, probe, num_sms,
                                         uuid)
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        rate, rows, dt, threads, passes = oracle_rate(A_host, B_host, args.cpu_seconds)
        what = (f"{rows} of {w.M} rows of the 4096^3 product" if passes == 1 else
                f"the whole 4096^3 product, {passes} times")
        out["cpu_baseline"] = {
            "value": round(rate, 6), "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": f"{what} (double accumulation), {dt:.1f} s",
            "workloads": oracle_workloads(inputs, threads)}
    if rank == 0:
        print(json.dumps(out), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_e2e(tg, A_host, B_host, w, dev, reps):
    """The step through the host API: pinned operands in, results out. The
    step's two products are two gemm_host calls in flight together on two
    streams (each copies its own operands and result); the step ends when
    both results are on the host."""
    import torch
    Ah = A_host.pin_memory()
    Bh = B_host.pin_memory()
    C1 = torch.empty(w.M, w.N, pin_memory=True)
    C2 = torch.empty(w.M, w.N, pin_memory=True)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()

    def e2e_step():
        cur = torch.cuda.current_stream()
        s1.wait_stream(cur)
        s2.wait_stream(cur)
        tg.binding.gemm_host(Ah, Bh, "f32", out=C1, stream=s1, synchronize=False)
        tg.binding.gemm_host(Ah, Bh, "tf32", out=C2, stream=s2, synchronize=False)
        cur.wait_stream(s1)
        cur.wait_stream(s2)
        s1.synchronize()
        s2.synchronize()

    for _ in range(3):                  # warm-up: pool blocks, streams, pinned pages
        e2e_step()
    torch.cuda.synchronize()
    times = []
    for _ in range(reps):
        s, e = event_pair()
        s.record()
        e2e_step()
        e.record()
        e.synchronize()
        times.append(s.elapsed_time(e))
    ms = statistics.mean(times)
    in_bytes = 2 * (Ah.numel() * Ah.element_size() + Bh.numel() * Bh.element_size())
    out_bytes = C1.numel() * 4 + C2.numel() * 4
    return {"value": round(2 * w.flops / (ms * 1e-3) / 1e12, 3), "unit": UNIT,
            "h2d_bytes_per_step": in_bytes, "d2h_bytes_per_step": out_bytes,
            "ms_per_step": round(ms, 4),
            "ms_median": round(statistics.median(times), 4), "ms_min": round(min(times), 4),
            "steps": reps,
            "api": "tiled_matrix_multiplication_sm_gb300.binding.gemm_host -> C ABI gemm_host: "
                   "the f32 and tf32 products in flight together on two streams, each "
                   "copying its operands in and its result out (copies overlapped)"}


def run_tensor_probe(tg, dev, peaks):
    """The tensor cores' dense MMA rate on this GPU (gemm_tc_peak: back-to-back
    SM-pair MMAs from resident shared memory), as context next to the
    measured cuBLAS peak that the roofline fractions use."""
    import torch
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    out = {}
    for kind in ("bf16", "tf32"):
        per_clk, tflops = tg.binding.tc_peak(kind, True, iters=200000)
        out[kind] = {"flop_per_clk_per_sm": round(per_clk, 1),
                     "tflops_probe": round(tflops, 1),
                     "tflops_at_max_clock": round(per_clk * sms * peaks["sm_max_mhz"] * 1e6 / 1e12,
                                                  1)}
    out["note"] = ("back-to-back 256x256 cta_group::2 MMAs, no loads; tflops_probe at the "
                   "clock the probe ran at, tflops_at_max_clock = FLOP/clk/SM x SMs x max SM clock")
    return out


def pipe_peak_tflops(probe, kind, num_sms, sm_mhz):
    """The tensor pipe's dense rate for `kind` ("bf16" or "tf32"; TF32X3 runs
    TF32 MMAs) from the library's probe, at the SM clock `sm_mhz`."""
    per_clk = probe["tf32" if kind == "tf32x3" else kind]["flop_per_clk_per_sm"]
    return per_clk * num_sms * sm_mhz * 1e6 / 1e12


# Workloads bound by reading their operands once (few rows): stated against
# HBM bandwidth with algorithmic bytes A + B read once and C written once.
HBM_BOUND = ("skinny_bf16", "skinny_f32")

SWEEP = [("int128", "f32"), ("u1024", "f32"), ("ragged", "f32"), ("ragged", "tf32"),
         ("n4096", "tf32x3"), ("ffn_bf16", "bf16"), ("skinny_bf16", "bf16"),
         ("skinny_f32", "f32"), ("skinny_f32", "tf32")]


def algorithmic_bytes(w):
    esz = 2 if w.dtype == "bf16" else 4
    return esz * (w.M * w.K + w.K * w.N) + 4 * w.M * w.N


def run_workloads(tg, inputs, dev, flush, peaks, fp32_peak, probe=None, num_sms=None, uuid=None):
    """Device-time TFLOP/s of the other measured shapes (median of 10); the
    128^3 product is bound by launch latency, so its time (us) is the figure
    to read there. Tensor-path entries also carry frac_vs_pipe: the rate
    against the library's tensor-pipe probe at the SM clock sampled during
    the sweep; the few-row shapes are stated against HBM bandwidth."""
    import torch
    res = {}
    with ClockSampler(uuid) as sampler:
        for name, path in SWEEP:
            w = inputs.WORKLOADS[name]
            A_host, B_host = inputs.operands(w)
            A, B = A_host.to(dev), B_host.to(dev)
            C = torch.empty(w.M, w.N, device=dev)
            if path == "f32":
                fn = lambda: tg.gemm_f32(A, B, out=C)   # noqa: E731
                peak, bound = fp32_peak, "alu"
            else:
                fn = lambda: tg.gemm_tc(A, B, path, out=C)   # noqa: E731
                peak = peaks["bf16_tflops"] * (1.0 if path == "bf16" else NOMINAL_TF32_OVER_BF16)
                bound = "tensor"
            for _ in range(3):
                fn()
            ms = time_calls(fn, 10, flush)
            tf = w.flops / (ms * 1e-3) / 1e12
            pipe = tf * (3 if path == "tf32x3" else 1)    # three tensor products per useful one
            entry = {"M": w.M, "N": w.N, "K": w.K, "ms": round(ms, 4), "us": round(ms * 1e3, 2),
                     "tflops": round(tf, 3), "peak": round(peak, 3), "frac": round(pipe / peak, 4),
                     "bound": bound, "kernel": tg.binding.last_kernel()}
            if name in HBM_BOUND:
                nbytes = algorithmic_bytes(w)
                gbs = nbytes / (ms * 1e-3) / 1e9
                entry.update({"bound": "hbm", "algorithmic_bytes": nbytes,
                              "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                              "frac": round(gbs / peaks["hbm_gbs"], 4)})
            res[f"{name}_{path}"] = entry
            del A, B, C
    clocks = sampler.summary()
    if tg.device_status() != 0:
        raise RuntimeError("a kernel wait timed out in the workload sweep")
    if probe is not None and num_sms and clocks["sm_mhz"]:
        for key, entry in res.items():
            path = key.rsplit("_", 1)[1]
            if path in ("tf32", "bf16", "tf32x3") and entry["bound"] == "tensor":
                pipe_peak = pipe_peak_tflops(probe, path, num_sms, clocks["sm_mhz"])
                pipe = entry["tflops"] * (3 if path == "tf32x3" else 1)
                entry["frac_vs_pipe"] = round(pipe / pipe_peak, 4)
    res["clocks"] = clocks
    res["note"] = ("frac: against MEASURED_PEAKS (tensor: cuBLAS bf16 burst, TF32 scaled by the "
                   "nominal ratio; hbm: measured copy); frac_vs_pipe: against the tensor-pipe "
                   "probe's FLOP/clk/SM x SMs x the median SM clock sampled during this sweep")
    return res


# ---------------------------------------------------------------- reference arm

def run_reference(args):
    """The CPU oracle as the reference arm: each step computes a bounded
    sample of rows of the same 4096^3 product."""
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    from tiled_matrix_multiplication_sm_gb300 import inputs
    import oracle

    w = inputs.WORKLOADS[WORKLOAD]
    A_host, B_host = inputs.operands(w)
    threads = len(os.sched_getaffinity(0))
    oracle.set_threads(threads)
    A64 = oracle.to_float64(A_host)
    B64 = oracle.to_float64(B_host)
    total_budget = args.ref_seconds
    t0 = time.perf_counter()
    oracle.gemm_rows(A64, B64, list(range(threads)))
    per_row = (time.perf_counter() - t0) / threads
    steps = args.steps + args.warmup
    rows = max(threads, int(total_budget / steps / max(per_row, 1e-9)) // threads * threads)
    rows = min(rows, w.M)
    for i in range(args.warmup):
        oracle.gemm_rows(A64, B64, list(range(rows)))
    t0 = time.perf_counter()
    for i in range(args.steps):
        start = (i * rows) % max(w.M - rows + 1, 1)
        oracle.gemm_rows(A64, B64, list(range(start, start + rows)))
    dt = time.perf_counter() - t0
    value = 2.0 * rows * w.N * w.K * args.steps / dt / 1e12
    sample = (f"{rows} of {w.M} rows of the 4096^3 product per step "
              f"(double accumulation, {threads} threads)")
    out = {"impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": UNIT,
           "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": round(dt * 1e3 / args.steps, 3), "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
           "config": {"workload": "square GEMM M=N=K=4096, A,B ~ N(0,1) fp32 row-major "
                                  "(seed 20262); CPU oracle on a row sample",
                      "M": w.M, "N": w.N, "K": w.K},
           "cpu_baseline": {"value": round(value, 6), "unit": UNIT, "cores": threads,
                            "kind": "oracle", "sample": sample},
           "e2e": {"value": round(value, 6), "unit": UNIT, "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0},
           "gpu_launches": 0}
    print(json.dumps(out), flush=True)


def run_single(args):
    """Time one (workload, path) product alone: --workload NAME:PATH."""
    import torch
    import tiled_matrix_multiplication_sm_gb300 as tg
    from tiled_matrix_multiplication_sm_gb300 import inputs

    name, _, path = args.workload.partition(":")
    w = inputs.WORKLOADS[name]
    path = path or w.paths[0]
    if path not in ("f32", "tf32", "bf16", "tf32x3"):
        raise SystemExit(f"unknown path {path!r}")
    dev = torch.device("cuda", 0)
    tg.load()
    props = torch.cuda.get_device_properties(0)
    peaks = load_peaks()
    A_host, B_host = inputs.operands(w)
    A, B = A_host.to(dev), B_host.to(dev)
    C = torch.empty(w.M, w.N, device=dev)
    flush = L2Flush(dev)
    if path == "f32":
        fn = lambda: tg.gemm_f32(A, B, out=C)          # noqa: E731
        peak, bound = fp32_peak_tflops(props.multi_processor_count, peaks["sm_max_mhz"]), "alu"
    else:
        fn = lambda: tg.gemm_tc(A, B, path, out=C)     # noqa: E731
        peak = peaks["bf16_tflops"] * (1.0 if path == "bf16" else NOMINAL_TF32_OVER_BF16)
        bound = "tensor"
    for _ in range(args.warmup):
        fn()
    ms = time_calls(fn, args.steps, flush)
    if tg.device_status() != 0:
        raise RuntimeError("a kernel wait timed out")
    tf = w.flops / (ms * 1e-3) / 1e12
    # The split-TF32 form issues three tensor products per useful one.
    pipe_tf = tf * (3 if path == "tf32x3" else 1)
    print(json.dumps({"metric": METRIC, "value": round(tf, 3), "unit": UNIT, "n_gpus": 1,
                      "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4),
                      "higher_is_better": True, "config": {"workload": w.description,
                                                          "path": path},
                      "kernel": tg.binding.last_kernel(),
                      "roofline": {"bound": bound, "achieved": round(pipe_tf, 3),
                                   "peak": round(peak, 3), "unit": UNIT,
                                   "frac": round(pipe_tf / peak, 4)}}), flush=True)


def run_cublas_context(args):
    """Context only, not the product: torch.matmul (cuBLAS) on the same
    workloads and paths, timed like the product (L2 flushed, CUDA events,
    median). FP32 with TF32 math off, TF32 with it on; BF16 writes a BF16
    result (half the output bytes of the product's FP32 C) and, where torch
    offers it, an FP32 result ("_fp32_out")."""
    import torch
    from tiled_matrix_multiplication_sm_gb300 import inputs

    dev = torch.device("cuda", 0)
    flush = L2Flush(dev)
    res = {}
    cases = {"u1024": ("f32",), "n4096": ("f32", "tf32"), "ragged": ("f32", "tf32"),
             "ffn_bf16": ("bf16",)}
    for name, paths in cases.items():
        w = inputs.WORKLOADS[name]
        A_host, B_host = inputs.operands(w)
        A, B = A_host.to(dev), B_host.to(dev)
        for path in paths:
            torch.backends.cuda.matmul.allow_tf32 = path == "tf32"
            fns = {"": lambda: torch.matmul(A, B)}
            if path == "bf16":
                # FP32 result like the product, where this torch offers it
                try:
                    torch.mm(A[:8, :8], B[:8, :8], out_dtype=torch.float32)
                    fns["_fp32_out"] = lambda: torch.mm(A, B, out_dtype=torch.float32)
                except (TypeError, RuntimeError):
                    pass
            for tag, fn in fns.items():
                for _ in range(args.warmup):
                    fn()
                ms = time_calls(fn, args.steps, flush)
                res[f"{name}_{path}{tag}"] = {"M": w.M, "N": w.N, "K": w.K, "ms": round(ms, 4),
                                              "tflops": round(w.flops / (ms * 1e-3) / 1e12, 3)}
        del A, B
    torch.backends.cuda.matmul.allow_tf32 = False
    print(json.dumps({"context": "cuBLAS via torch.matmul on the bench workloads (not the "
                                 "product; torch " + torch.__version__ + ")",
                      "unit": UNIT, "steps": args.steps, "warmup": args.warmup,
                      "results": res}), flush=True)


def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=300)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--no-extras", action="store_true", help="skip e2e and the workload sweep")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-seconds", type=float, default=10.0)
    p.add_argument("--ref-seconds", type=float, default=90.0)
    p.add_argument("--cublas-context", action="store_true",
                   help="time torch.matmul (cuBLAS) on the same workloads as context and exit")
    p.add_argument("--workload", default=None,
                   help="time one product alone, NAME:PATH (e.g. ffn_bf16:bf16); median "
                        "of --steps calls")
    args = p.parse_args(argv)
    args.warmup = max(args.warmup, 3)      # at least three warm-up steps, always
    return args


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        run_reference(args)
    elif args.workload:
        run_single(args)
    elif args.cublas_context:
        run_cublas_context(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
