"""Nsight Compute evidence for every kernel of the library.

For each measured case (a workload and a path), this module

1. runs the product plainly in a child process (two warm-up products and one
   more), which must exit 0, and reads from the library which kernels one
   product launches (``gemm_last_kernel``);
2. runs the same command under ``ncu --clock-control none`` capturing exactly
   the kernels of the last product (``--launch-skip`` past the warm-ups,
   ``--launch-count`` = kernels per product) with a short list of counters:
   device time, DRAM bytes read and written, FMA / tensor / TMA pipe
   utilisation, shared-memory wavefronts and bank conflicts of loads and
   stores, L2 hit rate, instructions, registers;
3. writes one JSON record per kernel: the counters, the kernel's algorithmic
   work (FLOP for the GEMM kernels, bytes for the data-movement kernels:
   transposes, repacks, TF32 splits, split-K reductions), its roofline
   fraction against the measured peaks of this GPU, and the SHA-256 of the
   kernel's source file, so that a record is recognisably stale once the
   kernel changes.

Usage (on a machine with the GPU, after ``build()``)::

    python -m tiled_matrix_multiplication_sm_gb300.evidence capture \\
        --out <raw-output-dir> [--case n4096:f32 ...]
    python -m tiled_matrix_multiplication_sm_gb300.evidence summary \\
        --records profiles/ncu > profiles/ncu_evidence.md

``run --case NAME:PATH`` is the child that ``capture`` profiles. The cases'
device memory is a few hundred MB to 1 GB (every workload's inputs exceed
the 129 MB L2, so DRAM figures are meaningful), each capture is one product's
few launches, so every ncu run ends by itself within a minute or two.
"""
from __future__ import annotations

import argparse
import csv
import datetime
import hashlib
import io
import json
import os
import re
import shutil
import subprocess
import sys
from typing import Dict, List, Optional

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")

WARMUP_PRODUCTS = 2

# Every kernel of the library appears in at least one case.
CASES = ["n4096:f32", "n4096:tf32", "ragged:f32", "ragged:tf32", "n4096:tf32x3",
         "ffn_bf16:bf16", "skinny_bf16:bf16", "skinny_f32:f32", "skinny_f32:tf32",
         "u1024:f32", "int128:f32", "k0:f32"]

METRICS = [
    "gpu__time_duration.sum",
    "sm__cycles_elapsed.avg.per_second",
    "dram__bytes_read.sum",
    "dram__bytes_write.sum",
    "gpu__dram_throughput.avg.pct_of_peak_sustained_elapsed",
    "sm__pipe_fma_cycles_active.avg.pct_of_peak_sustained_active",
    "sm__pipe_tensor_cycles_active.avg.pct_of_peak_sustained_active",
    "sm__pipe_tma_cycles_active.avg.pct_of_peak_sustained_active",
    "l1tex__data_pipe_lsu_wavefronts_mem_shared_op_ld.sum",
    "l1tex__data_pipe_lsu_wavefronts_mem_shared_op_st.sum",
    "l1tex__data_bank_conflicts_pipe_lsu_mem_shared_op_ld.sum",
    "l1tex__data_bank_conflicts_pipe_lsu_mem_shared_op_st.sum",
    "lts__t_sector_hit_rate.pct",
    "smsp__inst_executed.sum",
    "launch__registers_per_thread",
    "launch__grid_size",
    "launch__block_size",
]

# Source file of each kernel (by the name ncu reports).
KERNEL_SOURCES = [
    ("sgemm_kernel", "sgemm_f32.cu"),
    ("splitk_reduce", "sgemm_f32.cu"),
    ("empty_product_kernel", "sgemm_f32.cu"),
    ("zero_rows_vec_kernel", "sgemm_f32.cu"),
    ("tc_", "gemm_tcgen05.cu"),
    ("transpose_split_kernel", "transpose_f32.cu"),
    ("transpose_kernel", "transpose_f32.cu"),
    ("repack_kernel", "transpose_f32.cu"),
    ("split_rows_kernel", "transpose_f32.cu"),
    ("split_rows_vec_kernel", "transpose_f32.cu"),
]


def source_of(kernel_name: str) -> Optional[str]:
    base = short_name(kernel_name)
    for key, src in KERNEL_SOURCES:
        if key in base:
            return src
    return None


def file_sha256(path: str) -> str:
    h = hashlib.sha256()
    with open(path, "rb") as f:
        h.update(f.read())
    return h.hexdigest()


def strip_comments(text: str) -> str:
    """C/C++/CUDA source without its comments, whitespace runs collapsed to
    one space: what the compiler sees, so that a record stays current while
    only the comments of its kernel's file change. String and character
    literals are kept as they are (a "//" inside one is not a comment)."""
    out = []
    i, n = 0, len(text)
    while i < n:
        c = text[i]
        if c == "/" and i + 1 < n and text[i + 1] == "/":
            j = text.find("\n", i)
            i = n if j < 0 else j
            out.append(" ")
        elif c == "/" and i + 1 < n and text[i + 1] == "*":
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        elif c in "\"'":
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def code_sha256(path: str) -> str:
    """SHA-256 of a source file's code with comments and layout removed."""
    with open(path, encoding="utf-8") as f:
        return hashlib.sha256(strip_comments(f.read()).encode()).hexdigest()


def record_current(rec: dict, root: str = None) -> bool:
    """Whether the kernel source a record names still has the code it was
    taken from (by the comment-free hash; records that carry only the
    whole-file hash are compared by that)."""
    if not rec.get("source"):
        return False
    path = os.path.join(root or ROOT, rec["source"])
    if not os.path.exists(path):
        return False
    if rec.get("code_sha256"):
        return code_sha256(path) == rec["code_sha256"]
    return file_sha256(path) == rec.get("source_sha256")


def short_name(kernel_name: str) -> str:
    """The kernel's function name without namespaces and template arguments:
    the first identifier of the demangled name that is followed by a template
    or parameter list and is not a namespace or a return type."""
    name = kernel_name.replace("(anonymous namespace)", "anon")
    for m in re.finditer(r"([A-Za-z_]\w*)\s*([<(]|::)", name):
        ident, nxt = m.group(1), m.group(2)
        if nxt == "::" or ident in ("void", "unnamed", "anon", "tgemm"):
            continue
        return ident
    return ""


# ---------------------------------------------------------------- case set-up

def case_shape(case: str):
    """(workload object or None, path, M, N, K, dtype) of a case."""
    from . import inputs
    name, _, path = case.partition(":")
    if name == "k0":
        return None, path, 4096, 4096, 0, "f32"
    w = inputs.WORKLOADS[name]
    return w, path, w.M, w.N, w.K, w.dtype


def run_case(case: str, products: int, tc_mode: int = -1, streamk: int = -1) -> str:
    """Run ``products`` products of the case on cuda:0; return the library's
    record of the kernels the last one launched. ``tc_mode`` and ``streamk``
    force the tensor-core tile shape and stream-K width (-1: automatic)."""
    import torch
    import tiled_matrix_multiplication_sm_gb300 as tg
    from . import inputs

    w, path, M, N, K, dtype = case_shape(case)
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(0)
    tg.load()
    tg.binding.set_tc_kernel(tc_mode)
    tg.binding.set_tc_streamk(streamk)
    if w is None:
        A = torch.empty(M, K, device=dev)
        B = torch.empty(K, N, device=dev)
    else:
        A_host, B_host = inputs.operands(w)
        A, B = A_host.to(dev), B_host.to(dev)
    C = torch.empty(M, N, device=dev)
    torch.cuda.synchronize()
    for _ in range(products):
        if path == "f32":
            tg.gemm_f32(A, B, out=C)
        else:
            tg.gemm_tc(A, B, path, out=C)
    torch.cuda.synchronize()
    if tg.device_status() != 0:
        raise RuntimeError("a kernel wait timed out")
    return tg.binding.last_kernel()


# ---------------------------------------------------------------- algorithmic work

def algorithmic_work(token: str, case: str) -> Dict[str, object]:
    """Roofline class and algorithmic work of one launch, from the library's
    name for it (a ``gemm_last_kernel`` token) and the case's shape."""
    _, path, M, N, K, dtype = case_shape(case)
    esz = 2 if dtype == "bf16" else 4
    if token == "empty_product":
        return {"bound": "hbm", "bytes": 4 * M * N}
    if token in ("repack_a", "transpose_a"):
        return {"bound": "hbm", "bytes": 2 * M * K * esz}
    if token in ("repack_b", "transpose_b"):
        return {"bound": "hbm", "bytes": 2 * K * N * esz}
    if token == "repack_ab":             # both operands in one launch
        return {"bound": "hbm", "bytes": 2 * (M * K + K * N) * esz}
    if token == "split_a":               # read fp32, write hi and lo
        return {"bound": "hbm", "bytes": 12 * M * K}
    if token == "split_b":
        return {"bound": "hbm", "bytes": 12 * K * N}
    if token == "transpose_split_a":
        return {"bound": "hbm", "bytes": 12 * M * K}
    if token == "transpose_split_b":
        return {"bound": "hbm", "bytes": 12 * K * N}
    m = re.match(r"(?:tc_split_reduce|splitk_reduce)\(split=(\d+),tiles=(\d+)\)", token)
    if m:
        split, tiles = int(m.group(1)), int(m.group(2))
        return {"bound": "hbm", "split": split, "tiles": tiles,
                "tile_shape": "from the GEMM kernel's name",
                "bytes_per_tile_elem": 4 * (split + 1)}
    # The few-row workloads are bound by reading B once: their GEMM kernels
    # are stated against HBM (A and B read once, C written once).
    few_rows = case.split(":")[0] in ("skinny_bf16", "skinny_f32")
    if few_rows and (token.startswith("f32_") or token.startswith("tc_")):
        return {"bound": "hbm", "bytes": esz * (M * K + K * N) + 4 * M * N,
                "flop": 2 * M * N * K}
    if token.startswith("f32_"):
        return {"bound": "alu", "flop": 2 * M * N * K}
    if token.startswith("tc_"):
        mult = 3 if path == "tf32x3" else 1     # three TF32 products per useful one
        return {"bound": "tensor", "flop": 2 * M * N * K * mult, "useful_flop": 2 * M * N * K}
    return {"bound": "unknown"}


def tile_elems(gemm_token: str) -> Optional[int]:
    """Elements of one output tile of the GEMM configuration name."""
    m = re.search(r"(\d+)x(\d+)x\d+", gemm_token)
    if not m:
        return None
    return int(m.group(1)) * int(m.group(2))


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "sm_max_mhz": float(d.get("sm_max_mhz", 2070.0)), "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "sm_max_mhz": 2070.0,
                "source": "fallback"}


# ---------------------------------------------------------------- ncu output

def parse_raw_csv(text: str) -> List[Dict[str, str]]:
    """Rows of ``ncu --page raw --csv`` output: one dict per profiled launch
    (the units row is dropped)."""
    lines = [ln for ln in text.splitlines() if ln.startswith('"')]
    if not lines:
        return []
    rows = list(csv.reader(io.StringIO("\n".join(lines))))
    header = rows[0]
    out = []
    for r in rows[1:]:
        if len(r) != len(header):
            continue
        d = dict(zip(header, r))
        if d.get("ID", "").strip() == "" or not d["ID"].strip().isdigit():
            continue                      # the units row
        out.append(d)
    return out


def number(s: str) -> Optional[float]:
    try:
        return float(str(s).replace(",", ""))
    except ValueError:
        return None


def make_records(rows, tokens, case, command, ncu_command, peaks, num_sms=None):
    """One record per profiled launch, paired in launch order with the
    library's names for the launches of one product."""
    records = []
    gemm_token = next((t for t in tokens if t.startswith(("f32_", "tc_"))), "")
    for i, (row, token) in enumerate(zip(rows, tokens)):
        kname = row.get("Kernel Name", "")
        metrics = {m: number(row[m]) for m in METRICS if m in row}
        t_ns = metrics.get("gpu__time_duration.sum") or 0.0
        work = algorithmic_work(token, case)
        if "bytes_per_tile_elem" in work:
            te = tile_elems(gemm_token)
            if te:
                work["bytes"] = work["tiles"] * te * work["bytes_per_tile_elem"]
        rd = metrics.get("dram__bytes_read.sum") or 0.0
        wr = metrics.get("dram__bytes_write.sum") or 0.0
        derived = {"time_us": round(t_ns / 1e3, 3),
                   "dram_bytes": int(rd + wr),
                   "dram_gbs": round((rd + wr) / t_ns, 1) if t_ns else None,
                   "dram_frac_of_hbm": round((rd + wr) / t_ns / peaks["hbm_gbs"], 4) if t_ns else None,
                   "sm_clock_mhz": round((metrics.get("sm__cycles_elapsed.avg.per_second") or 0) / 1e6)}
        roof = {"bound": work["bound"]}
        if work["bound"] == "hbm" and "bytes" in work and t_ns:
            gbs = work["bytes"] / t_ns
            roof.update({"algorithmic_bytes": work["bytes"], "achieved": round(gbs, 1),
                         "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": round(gbs / peaks["hbm_gbs"], 4),
                         "traffic_over_algorithmic": round((rd + wr) / work["bytes"], 3)})
        elif work["bound"] == "alu" and t_ns:
            tf = work["flop"] / t_ns / 1e3
            sms = num_sms or 152
            peak = sms * 128 * 2 * peaks["sm_max_mhz"] * 1e6 / 1e12
            roof.update({"algorithmic_flop": work["flop"], "achieved": round(tf, 2), "peak": round(peak, 2),
                         "unit": "TFLOP/s", "frac": round(tf / peak, 4),
                         "peak_basis": f"{sms} SMs x 128 FP32 lanes x 2 x max SM clock"})
        elif work["bound"] == "tensor" and t_ns:
            tf = work["flop"] / t_ns / 1e3
            _, path, *_ = case_shape(case)
            peak = peaks["bf16_tflops"] * (1.0 if path == "bf16" else 1.1 / 2.25)
            roof.update({"algorithmic_flop": work["flop"], "achieved": round(tf, 2), "peak": round(peak, 2),
                         "unit": "TFLOP/s", "frac": round(tf / peak, 4),
                         "peak_basis": "measured bf16 (cuBLAS burst)" +
                                       ("" if path == "bf16" else " x nominal tf32/bf16 1.1/2.25")})
        src = source_of(kname)
        rec = {"kernel": kname, "kernel_short": short_name(kname), "library_name": token,
               "case": case, "launch_index": i, "launches_per_product": len(tokens),
               "command": command, "ncu_command": ncu_command,
               "source": f"tiled_matrix_multiplication_sm_gb300/csrc/{src}" if src else None,
               "source_sha256": file_sha256(os.path.join(CSRC, src)) if src else None,
               "code_sha256": code_sha256(os.path.join(CSRC, src)) if src else None,
               "metrics": metrics, "derived": derived, "roofline": roof,
               "peaks_source": peaks["source"],
               "taken": datetime.datetime.now(datetime.timezone.utc).strftime("%Y-%m-%d")}
        records.append(rec)
    return records


def record_filename(rec) -> str:
    case = rec["case"].replace(":", "_")
    tok = re.sub(r"[^A-Za-z0-9_]+", "_", rec["library_name"]).strip("_")
    return f"{rec['kernel_short']}__{case}__{rec['launch_index']}_{tok}.json"


# ---------------------------------------------------------------- capture

def ncu_binary() -> str:
    path = shutil.which("ncu")
    if path:
        return path
    cand = "/usr/local/cuda/bin/ncu"
    if os.path.exists(cand):
        return cand
    raise RuntimeError("ncu not found")


def capture(cases, out_dir, timeout_s=600):
    import torch
    os.makedirs(out_dir, exist_ok=True)
    peaks = load_peaks()
    num_sms = torch.cuda.get_device_properties(0).multi_processor_count
    products = WARMUP_PRODUCTS + 1
    summary = []
    for case in cases:
        child = [sys.executable, "-m", "tiled_matrix_multiplication_sm_gb300.evidence", "run",
                 "--case", case, "--products", str(products)]
        # 1. the plain run: must exit 0 before the same command runs under ncu
        plain = subprocess.run(child, capture_output=True, text=True, cwd=ROOT, timeout=timeout_s)
        if plain.returncode != 0:
            raise RuntimeError(f"{case}: plain run failed\n{plain.stdout}\n{plain.stderr}")
        last = json.loads(plain.stdout.strip().splitlines()[-1])["kernels"]
        tokens = [t for t in last.split("+") if t]
        if not tokens:
            continue
        # 2. the capture: the kernels of the last product only
        log = os.path.join(out_dir, case.replace(":", "_") + ".csv")
        ncu_cmd = [ncu_binary(), "--clock-control", "none", "--metrics", ",".join(METRICS),
                   "--launch-skip", str(WARMUP_PRODUCTS * len(tokens)),
                   "--launch-count", str(len(tokens)), "--page", "raw", "--csv",
                   "--print-units", "base", "--log-file", log] + child
        res = subprocess.run(ncu_cmd, capture_output=True, text=True, cwd=ROOT, timeout=timeout_s)
        if res.returncode != 0:
            raise RuntimeError(f"{case}: ncu exited {res.returncode}\n{res.stdout[-2000:]}\n"
                               f"{res.stderr[-2000:]}")
        with open(log) as f:
            rows = parse_raw_csv(f.read())
        if len(rows) != len(tokens):
            raise RuntimeError(f"{case}: {len(rows)} profiled launches for {len(tokens)} kernels "
                               f"({last})")
        command = ("python -m tiled_matrix_multiplication_sm_gb300.evidence run --case "
                   f"{case} --products {products}")
        ncu_text = ("ncu --clock-control none --metrics <METRICS of evidence.py> --launch-skip "
                    f"{WARMUP_PRODUCTS * len(tokens)} --launch-count {len(tokens)} --page raw "
                    f"--csv --print-units base {command}")
        for rec in make_records(rows, tokens, case, command, ncu_text, peaks, num_sms):
            with open(os.path.join(out_dir, record_filename(rec)), "w") as f:
                json.dump(rec, f, indent=1, sort_keys=True)
            summary.append(rec)
        print(f"{case}: {len(tokens)} kernels captured", flush=True)
    return summary


# ---------------------------------------------------------------- summary table

def summary_table(records_dir: str) -> str:
    recs = []
    for fn in sorted(os.listdir(records_dir)):
        if fn.endswith(".json"):
            with open(os.path.join(records_dir, fn)) as f:
                recs.append(json.load(f))
    recs.sort(key=lambda r: (r["case"], r["launch_index"]))
    lines = ["| case | # | kernel | library name | us | DRAM GB/s | bound | achieved | frac | "
             "FMA pipe % | tensor pipe % | smem ld/st wavefronts | ld/st bank conflicts | "
             "DRAM / algorithmic | source current |",
             "|---|---|---|---|---|---|---|---|---|---|---|---|---|---|---|"]
    for r in recs:
        m, d, roof = r["metrics"], r["derived"], r["roofline"]
        cur = record_current(r) if r.get("source") else None

        def fmt(v, nd=1):
            return "" if v is None else (f"{v:.{nd}f}" if isinstance(v, float) else str(v))

        ach = f"{roof.get('achieved', '')} {roof.get('unit', '')}".strip()
        lines.append(
            f"| {r['case']} | {r['launch_index']} | `{r['kernel_short']}` | {r['library_name']} | "
            f"{fmt(d['time_us'])} | {fmt(d['dram_gbs'])} | {roof['bound']} | {ach} | "
            f"{fmt(roof.get('frac'), 3)} | "
            f"{fmt(m.get('sm__pipe_fma_cycles_active.avg.pct_of_peak_sustained_active'))} | "
            f"{fmt(m.get('sm__pipe_tensor_cycles_active.avg.pct_of_peak_sustained_active'))} | "
            f"{fmt(m.get('l1tex__data_pipe_lsu_wavefronts_mem_shared_op_ld.sum'), 0)} / "
            f"{fmt(m.get('l1tex__data_pipe_lsu_wavefronts_mem_shared_op_st.sum'), 0)} | "
            f"{fmt(m.get('l1tex__data_bank_conflicts_pipe_lsu_mem_shared_op_ld.sum'), 0)} / "
            f"{fmt(m.get('l1tex__data_bank_conflicts_pipe_lsu_mem_shared_op_st.sum'), 0)} | "
            f"{fmt(roof.get('traffic_over_algorithmic'), 2)} | {'yes' if cur else 'no'} |")
    return "\n".join(lines) + "\n"


def find_record(records_dir: str, case: str, kernel_short: str) -> Optional[dict]:
    """The record of `kernel_short` in `case`, or None."""
    try:
        names = sorted(os.listdir(records_dir))
    except OSError:
        return None
    for fn in names:
        if fn.endswith(".json") and fn.startswith(f"{kernel_short}__{case.replace(':', '_')}__"):
            with open(os.path.join(records_dir, fn)) as f:
                return json.load(f)
    return None


def main(argv=None):
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    sub = p.add_subparsers(dest="cmd", required=True)
    r = sub.add_parser("run", help="run one case's products (the profiled child)")
    r.add_argument("--case", required=True)
    r.add_argument("--products", type=int, default=WARMUP_PRODUCTS + 1)
    r.add_argument("--tc-mode", type=int, default=-1)
    r.add_argument("--streamk", type=int, default=-1)
    c = sub.add_parser("capture", help="plain run, then ncu, for each case")
    c.add_argument("--case", action="append", default=None)
    c.add_argument("--out", required=True,
                   help="directory for the .ncu-rep files, logs and JSON records")
    s = sub.add_parser("summary", help="markdown table of the records in a directory")
    s.add_argument("--records", default=os.path.join(ROOT, "profiles", "ncu"))
    args = p.parse_args(argv)
    if args.cmd == "run":
        print(json.dumps({"kernels": run_case(args.case, args.products, args.tc_mode,
                                              args.streamk)}), flush=True)
    elif args.cmd == "capture":
        capture(args.case or CASES, args.out)
    else:
        sys.stdout.write(summary_table(args.records))


if __name__ == "__main__":
    main()
