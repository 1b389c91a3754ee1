"""Benchmark of the MSA index-branch block score on GB300.

One step = one full call of the op (plan kernel + persistent tensor-core score
kernel) over one resident batch of synthetic inputs.  Default workload: the
long-context prefill (B=1, T=16384 query tokens at kv_len=131072, H_q=64,
H_kv=8, D=P=128, bf16, a randomly permuted [1, 1100] block table; output
[64, 16384, 1104] fp32, 4.63 GB; 3.3e13 flop).  The same run also measures
the other four workloads (tiny prefill, batched decode, varlen chunked
prefill, int8 mixed) and the int8 decode subset as sub-records.

Prints ONE JSON line (rank 0).  ``value`` is microseconds per call for the
whole job (lower is better); the line also carries TFLOP/s, K-cache GB/s, the
roofline of the dominant kernel (timed with CUDA events in the same
clock-sampled window as the calls), the CPU oracle timed on the host cores,
an end-to-end figure through the C ABI with host buffers, and the SM clocks
seen during the timed region.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload 1..5]
    python bench.py --impl reference ...   # the CPU oracle as the reference arm

Multi-GPU: the op does not shard across GPUs in a way that needs an
exchange; N>1 runs N independent replicas (one process per GPU under
torchrun), times them between barriers and takes the max over ranks.
"""
from __future__ import annotations

import argparse
import dataclasses
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

import torch  # noqa: E402

L2_BYTES = 126 * 1024 * 1024   # GB300 L2 (spec: ~129 MB); inputs below it are cache-resident

import synth  # noqa: E402

METRIC = "MsaIndexScore µs/call, TFLOP/s and K-cache GB/s vs GB300 roofline (1 GPU)"
DEFAULT_WORKLOAD = 5
# calls per timed pass when --steps is not given (about 0.2-0.6 s of GPU time each)
DEFAULT_STEPS = {1: 5000, 2: 2000, 3: 300, 4: 400, 5: 30}
DEFAULT_STEPS_DECODE_SUBSET = 5000
# (workload, decode subset, FP4 format): the other workloads, the int8 decode
# subset, and FP4 inputs on the batched decode and the varlen prefill
SUB_WORKLOADS = [(1, False, None), (2, False, None), (3, False, None), (4, False, None),
                 (4, True, None), (2, False, "nv"), (3, False, "mx")]
DTYPE_NAME = {torch.float16: "f16", torch.bfloat16: "bf16", torch.int8: "i8",
              torch.float8_e4m3fn: "e4m3", torch.float8_e5m2: "e5m2"}
FP8 = {"e4m3": torch.float8_e4m3fn, "e5m2": torch.float8_e5m2}


# ----------------------------------------------------------------------------
# algorithmic work of a case (what the op must do, not what the tiles do)
# ----------------------------------------------------------------------------
def algorithmic_work(case):
    """FLOPs = 2*D*sum over (h,t) of visible keys; bytes = visible K once per kv head
    (+ int8 scale) + Q + the fp32 output + the table entries read."""
    D, P = case.D, case.P
    fp4 = getattr(case, "fp4", None)
    # bytes of one key row of D values: FP4 codes are half a byte each, plus
    # one scale byte per group of 32 (MXFP4) or 16 (NVFP4)
    row_k = (D // 2 + D // (32 if fp4 == "mx" else 16)) if fp4 else D * case.key.element_size()
    vis_rows = 0
    k_tokens = 0
    tab = 0
    for Lq, L in zip(case.q_lens, case.kv_lens):
        if Lq == 0:
            continue
        if case.sparse_mode == 3:
            # row i sees min(L, L - Lq + i + 1) keys (none if negative)
            for i in range(Lq):
                vis_rows += max(0, min(L, L - Lq + i + 1))
        else:
            vis_rows += Lq * L
        k_tokens += L
        tab += -(-L // P)
    flops = 2.0 * D * case.H_q * vis_rows
    k_bytes = k_tokens * case.H_kv * row_k
    if case.key.dtype == torch.int8:
        k_bytes += k_tokens * case.H_kv * 4
    q_bytes = case.T * case.H_q * (row_k if fp4 else D * case.query.element_size())
    out_bytes = case.H_q * case.T * case.MBp * 4
    total = k_bytes + q_bytes + out_bytes + 4 * tab
    return {"flops": flops, "k_bytes": k_bytes, "q_bytes": q_bytes, "out_bytes": out_bytes,
            "bytes": total}


# sources each score kernel is built from (an ncu figure is only valid for the
# code it measured)
KERNEL_SOURCES = {
    "tile_kernel": ["msa_tile.cuh", "msa_units.cuh", "msa_ptx.cuh", "msa_common.cuh",
                    "msa_score_16.cu", "msa_score_i8.cu", "msa_score_f8.cu"],
    "short_kernel": ["msa_short.cuh", "msa_units.cuh", "msa_ptx.cuh", "msa_common.cuh",
                     "msa_short.cu", "msa_short_fp4.cu"],
}


def code_only(text: str) -> str:
    """C/CUDA source with its comments, trailing blanks and empty lines
    removed (string and character literals kept as written), so that a
    change to a comment alone leaves the hash of a kernel's sources as it was."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c in "\"'":
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            out.append(" ")
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    lines = (line.rstrip() for line in "".join(out).split("\n"))
    return "\n".join(line for line in lines if line)


def kernel_source_hash(kernel: str) -> str:
    """Hash of the code (comments left out) of the CUDA sources of one kernel."""
    import hashlib
    h = hashlib.sha256()
    d = os.path.join(ROOT, "block_score_gb300", "csrc")
    for name in KERNEL_SOURCES[kernel]:
        with open(os.path.join(d, name), encoding="utf-8") as f:
            h.update(name.encode() + b"\0" + code_only(f.read()).encode())
    return h.hexdigest()[:16]


def dominant_kernel(case) -> str:
    """The kernel that does the work of a workload: the short-query kernel when
    every request is a short request with int8 or FP4 keys, else the tile kernel."""
    g = case.H_q // case.H_kv
    short = (case.key.dtype == torch.int8 or bool(getattr(case, "fp4", None))) and all(
        lq == 0 or lq * g <= 32 for lq in case.q_lens)
    return "short_kernel" if short and any(lq > 0 for lq in case.q_lens) else "tile_kernel"


def launches_per_call(case) -> int:
    """Kernels one call launches: the plan (FP4: after the query
    dequantisation), the tile kernel unless the host length bound puts every
    request on the short path (with int8 paged keys, and FP4 paged keys of a
    prefill-heavy call, preceded by the conversion of their pages into the
    16-bit mirror), and, for int8 or FP4 keys with a query-row group of at
    most 32, the short-query kernel."""
    g = case.H_q // case.H_kv
    fp4 = bool(getattr(case, "fp4", None))
    i8 = case.key.dtype == torch.int8
    short_ok = (i8 or fp4) and g <= 32
    max_q = max(case.q_lens) if case.q_lens else 0
    tile = not (short_ok and max_q > 0 and max_q * g <= 32)
    paged = case.layout.upper() != "TND"
    if fp4:
        mirror = tile and paged and case.T * g >= 128 * case.B
    else:
        mirror = tile and i8 and paged
    return ((2 if fp4 else 1) + (1 if tile else 0) + (1 if mirror else 0)
            + (1 if short_ok else 0))


def recorded_traffic(workload_key: str, kernel: str):
    """DRAM bytes per launch of the dominant kernel from the committed ncu
    summary, if it was taken on the current sources of that kernel (else None)."""
    path = os.path.join(ROOT, "profiles", "kernel_dram_traffic.txt")
    try:
        with open(path) as f:
            for line in f:
                parts = line.split()
                if (len(parts) >= 4 and not line.startswith("#") and parts[0] == workload_key
                        and parts[1] == kernel and parts[3] == kernel_source_hash(kernel)):
                    return float(parts[2])
    except OSError:
        pass
    return None


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return {"hbm_gbs": float(pk["hbm_gbs"]), "bf16_tflops": float(pk["bf16_tflops"]),
                "bf16_tflops_sustained": float(pk.get("bf16_tflops_sustained",
                                                      pk["bf16_tflops"])),
                "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                "source": "fallback"}


# ----------------------------------------------------------------------------
# clocks during the timed region
# ----------------------------------------------------------------------------
class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.rows = []
        self.proc = None
        self.t_start = self.t_stop = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self._th = threading.Thread(target=self._reader, daemon=True)
        self._th.start()

    def _reader(self):
        for line in self.proc.stdout:
            self.rows.append((time.time(), line.strip()))

    def mark(self, which):
        if which == "start":
            self.t_start = time.time()
        else:
            self.t_stop = time.time()

    def stop(self):
        if self.proc is None:
            return
        time.sleep(0.12)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self._th.join(timeout=2)

    def summary(self):
        if not self.rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no nvidia-smi samples"]}
        inside = [r for t, r in self.rows
                  if self.t_start is not None and self.t_start - 0.05 <= t <= self.t_stop + 0.05]
        use = inside if inside else [r for _, r in self.rows]
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in use:
            f = [x.strip() for x in r.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons),
                "samples": len(use), "samples_in_timed_region": len(inside)}


# ----------------------------------------------------------------------------
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(x: float, ws: int, device) -> float:
    if ws == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_us_per_call(step_ms_local: float, ws: int, device, calls_per_rank: int = 1):
    """Replicas: every rank runs its own calls; the job's step time is the
    slowest rank's, and the job processes ws * calls_per_rank calls per step.
    Returns (step_ms, us_per_call) for the whole job."""
    step_ms = max_over_ranks(step_ms_local, ws, device)
    return step_ms, step_ms * 1e3 / (ws * calls_per_rank)


def barrier(ws: int):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def cpu_oracle_baseline(case, target_s: float = 12.0):
    """Time the CPU oracle (as it stands) on a bounded row sample; scale to one call."""
    import oracle
    rows_total = case.H_q * case.T
    threads = oracle.oracle_threads()
    # probe a small sample, then size the sample for ~target_s of CPU work
    probe = list(range(0, rows_total, max(1, rows_total // 64)))
    t0 = time.perf_counter()
    oracle.oracle_rows(case, probe)
    dt = max(time.perf_counter() - t0, 1e-4)
    per_row = dt / len(probe)
    n = int(min(rows_total, max(len(probe), target_s / per_row)))
    step = max(1, rows_total // n)
    rows = list(range(0, rows_total, step))
    t0 = time.perf_counter()
    oracle.oracle_rows(case, rows)
    dt = time.perf_counter() - t0
    us_per_call = dt / len(rows) * rows_total * 1e6
    frac = len(rows) / rows_total
    sample = ("full workload" if len(rows) == rows_total else
              f"{len(rows)} of {rows_total} (h,t) output rows, every {step}th, scaled by row count")
    return {"value": us_per_call, "unit": "us/call", "cores": threads, "kind": "oracle",
            "sample": sample, "sample_fraction": frac, "seconds": dt}


def make_workload(args):
    case = synth.config(args.workload, layout=args.layout,
                        q_len=getattr(args, "q_len", None) if args.workload == 5 else None)
    if args.decode_subset:
        case = synth.decode_subset(case)
    if getattr(args, "fp4", None):
        # the same workload (lengths, table, pages) with FP4 query and keys
        if case.key.dtype == torch.int8:
            raise SystemExit("--fp4 applies to the fp16 / bf16 workloads")
        return synth.to_fp4(case, args.fp4)
    if args.fp8:
        # the same workload with FP8 query and keys of one type (no scale):
        # the 16-bit draws rounded to FP8
        if case.key.dtype == torch.int8:
            raise SystemExit("--fp8 applies to the fp16 / bf16 workloads")
        dt = FP8[args.fp8]
        case = dataclasses.replace(case, query=case.query.float().to(dt), key=case.key.float().to(dt),
                                   name=f"{case.name}_{args.fp8}")
    return case


def workload_key(args) -> str:
    q = getattr(args, "q_len", None)
    return (f"cfg{args.workload}" + ("_decode" if args.decode_subset else "")
            + (f"_q{q}" if q and args.workload == 5 else "")
            + (f"_{args.layout.lower()}" if args.layout else "")
            + (f"_{args.fp8}" if args.fp8 else "")
            + (f"_fp4{args.fp4}" if getattr(args, "fp4", None) else ""))


def default_steps(args) -> int:
    if args.steps is not None:
        return args.steps
    if args.decode_subset:
        return DEFAULT_STEPS_DECODE_SUBSET
    return DEFAULT_STEPS[args.workload]


def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    case = make_workload(args)
    work = algorithmic_work(case)
    import oracle
    rows_total = case.H_q * case.T
    # each step: a bounded, fixed row sample (about a second of CPU work)
    probe = list(range(0, rows_total, max(1, rows_total // 64)))
    t0 = time.perf_counter()
    oracle.oracle_rows(case, probe)
    per_row = max(time.perf_counter() - t0, 1e-4) / len(probe)
    n = int(min(rows_total, max(len(probe), 1.0 / per_row)))
    step = max(1, rows_total // n)
    rows = list(range(0, rows_total, step))
    steps = args.steps if args.steps is not None else 5
    for _ in range(args.warmup):
        oracle.oracle_rows(case, rows)
    times = []
    for _ in range(steps):
        t0 = time.perf_counter()
        oracle.oracle_rows(case, rows)
        times.append(time.perf_counter() - t0)
    per_call_s = statistics.mean(times) / len(rows) * rows_total
    us = per_call_s * 1e6
    threads = oracle.oracle_threads()
    sample = (f"{len(rows)} of {rows_total} (h,t) output rows per step, every {step}th, "
              "scaled by row count")
    line = {
        "impl": "reference", "metric": METRIC, "value": us, "unit": "us/call",
        "n_gpus": ws, "steps": steps, "warmup": args.warmup,
        "ms_per_step": statistics.mean(times) * 1e3, "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": config_block(case, workload_key(args)),
        "tflops": work["flops"] / per_call_s / 1e12,
        "k_cache_gbs": work["k_bytes"] / per_call_s / 1e9,
        "cpu_baseline": {"value": us, "unit": "us/call", "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": us, "unit": "us/call", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def dtype_name(case) -> str:
    """The arithmetic type the path computes in."""
    fp4 = getattr(case, "fp4", None)
    if fp4:
        return "e2m1 codes x group scales, dequantised to " + ("f16" if fp4 == "nv" else "bf16")
    return DTYPE_NAME[case.query.dtype] if case.key.dtype != torch.int8 else "f16xi8"


def config_block(case, workload):
    kb = algorithmic_work(case)["k_bytes"]
    total_in = kb + case.query.numel() * case.query.element_size()
    return {"workload": f"{workload}:{case.name}", "B": case.B, "T": case.T,
            "H_q": case.H_q, "H_kv": case.H_kv, "D": case.D, "P": case.P, "MB": case.MB,
            "layout": case.layout,
            "k_dtype": ("fp4" + case.fp4) if getattr(case, "fp4", None) else DTYPE_NAME[case.key.dtype],
            "sparse_mode": case.sparse_mode, "init_blocks": case.init_blocks,
            "local_blocks": case.local_blocks,
            "l2": (f"inputs larger than L2 (no flush): K cache {kb / 1e6:.0f} MB > 129 MB"
                   if kb > 129e6 else
                   (f"inputs larger than L2 (no flush): K + Q {total_in / 1e6:.0f} MB > 129 MB"
                    if total_in > 129e6 else
                    "inputs fit in L2 (no flush; launch- or latency-bound case)"))}


def is_fp8(case) -> bool:
    """FP8 query and keys (FP4 codes are bytes too, but they are multiplied on
    the 16-bit tensor path)."""
    return case.query.element_size() == 1 and not getattr(case, "fp4", None)


def tensor_peak(case, peaks) -> float:
    """Dense tensor peak (TFLOP/s) of the case's operand type: the measured bf16
    burst peak, times the nominal dense ratio 4.5 / 2.25 for FP8 operands."""
    return peaks["bf16_tflops"] * (2.0 if is_fp8(case) else 1.0)


def roofline_of(case, work, kern_ms, peaks, traffic):
    """Roofline record of the dominant kernel from its per-launch duration."""
    kern_s = kern_ms / 1e3
    hbm_gbs_kernel = work["bytes"] / kern_s / 1e9
    tflops_kernel = work["flops"] / kern_s / 1e12
    fp8 = is_fp8(case)
    tensor_peak_tf = tensor_peak(case, peaks)
    # the binding roof: the longer of the two roofline times, each at its own peak
    bound = "hbm" if work["bytes"] / (peaks["hbm_gbs"] * 1e9) >= \
        work["flops"] / (tensor_peak_tf * 1e12) else "tensor"
    if bound == "hbm":
        roof = {"bound": "hbm", "achieved": hbm_gbs_kernel, "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "frac": hbm_gbs_kernel / peaks["hbm_gbs"],
                "traffic": traffic, "peak_source": peaks["source"] + " hbm_gbs"}
    elif fp8:
        pk = tensor_peak_tf
        roof = {"bound": "tensor", "achieved": tflops_kernel, "peak": pk, "unit": "TFLOP/s",
                "frac": tflops_kernel / pk, "traffic": traffic,
                "peak_source": peaks["source"] + " bf16_tflops (burst) x 2 (nominal fp8 / bf16)"}
    else:
        pk = peaks["bf16_tflops"]
        roof = {"bound": "tensor", "achieved": tflops_kernel, "peak": pk, "unit": "TFLOP/s",
                "frac": tflops_kernel / pk, "traffic": traffic,
                "peak_source": peaks["source"] + " bf16_tflops (burst)",
                "frac_of_sustained": tflops_kernel / peaks["bf16_tflops_sustained"]}
    if getattr(case, "fp4", None) and roof["bound"] == "tensor":
        roof["peak_source"] += ("; FP4 operands are dequantised to 16-bit and multiplied on the "
                                "16-bit tensor path, whose peak applies")
    roof["kernel"] = dominant_kernel(case)
    roof["kernel_us"] = kern_ms * 1e3
    roof["algorithmic_bytes"] = work["bytes"]
    roof["algorithmic_flops"] = work["flops"]
    return roof


def measure(case, key, steps, warmup, device, stream, peaks, ws, traffic=None):
    """Time one workload: pass A (K back-to-back calls, events at the ends)
    gives the per-call time; pass B (K calls with events before each call and
    around its score launches) gives the dominant kernel's per-launch time and,
    from the same events, its own per-call time, so a launch never reads longer
    than the call it belongs to.  Both passes run inside one clock-sampled
    window."""
    import block_score_gb300 as bs
    work = algorithmic_work(case)
    # the caller knows its requests' query lengths (as a serving loop does)
    prep = bs.from_case(case, device, max_seqlen_q=max(case.q_lens) if case.q_lens else None)
    # correctness gate before timing (the parity tests are the full check)
    prep(stream)
    if prep.device_error(stream):
        raise RuntimeError(f"{key}: device error during the first call")
    for _ in range(warmup):
        prep(stream)
    torch.cuda.synchronize(device)

    sampler = ClockSampler(device.index if device.index is not None else 0)
    sampler.start()
    time.sleep(0.25)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev_b = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(3)) for _ in range(steps)]
    barrier(ws)
    torch.cuda.synchronize(device)
    sampler.mark("start")
    # pass A: back-to-back calls; the score kernel's launch overlaps the plan
    ev0.record(stream)
    for _ in range(steps):
        prep(stream)
    ev1.record(stream)
    # pass B: events before each call and around its score launches
    for i in range(steps):
        ev_b[i][0].record(stream)
        prep.plan(stream)
        ev_b[i][1].record(stream)
        prep.run(stream)
        ev_b[i][2].record(stream)
    torch.cuda.synchronize(device)
    sampler.mark("stop")
    sampler.stop()
    barrier(ws)
    total_ms = ev0.elapsed_time(ev1)
    kern_ms = statistics.mean(b.elapsed_time(c) for _, b, c in ev_b)
    call_b_ms = statistics.mean(a.elapsed_time(c) for a, _, c in ev_b)
    step_ms, us_per_call = whole_job_us_per_call(total_ms / steps, ws, device)
    kern_ms = max_over_ranks(kern_ms, ws, device)
    call_b_ms = max_over_ranks(call_b_ms, ws, device)
    if prep.device_error(stream):
        raise RuntimeError(f"{key}: device error during the timed region")
    call_s = step_ms / 1e3
    roof = roofline_of(case, work, kern_ms, peaks, traffic)
    roof["kernel_timing"] = ("CUDA events around the score launches of each call (tile "
                             "kernel, plus the short-query kernel for int8 keys) after its "
                             "plan, in a second pass of K calls inside the same clock-sampled "
                             "window as the per-call timing")
    roof["call_us_same_pass"] = call_b_ms * 1e3
    rec = {
        "workload": f"{key}:{case.name}", "value": us_per_call, "unit": "us/call",
        "steps": steps, "ms_per_step": step_ms,
        "tflops": work["flops"] / call_s / 1e12,
        "k_cache_gbs": work["k_bytes"] / call_s / 1e9,
        "frac_hbm": (work["bytes"] / call_s / 1e9) / peaks["hbm_gbs"],
        "frac_tensor": work["flops"] / call_s / 1e12 / tensor_peak(case, peaks),
        "roofline": roof,
        "gpu_launches": launches_per_call(case) * steps,
        "clocks": sampler.summary(),
    }
    return rec, prep


def run_ours(args):
    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    import block_score_gb300 as bs
    bs.load_library()
    peaks = load_peaks()
    stream = torch.cuda.current_stream(device)

    case = make_workload(args)
    key = workload_key(args)
    if args.sparse_only:
        # the sparse main branch alone on this workload (a profiler's target)
        prep = bs.from_case(case, device)
        rec = sparse_run(case, prep, device, stream, peaks, args.steps or 10)
        if rank == 0:
            print(json.dumps({"impl": "ours", "sparse_attention": rec, "config": config_block(case, key)}),
                  flush=True)
        return
    steps = default_steps(args)
    traffic = args.traffic
    if traffic is None:
        traffic = recorded_traffic(key, dominant_kernel(case))
    head, prep = measure(case, key, steps, args.warmup, device, stream, peaks, ws, traffic)

    # end to end through the C ABI with host buffers: H2D of the inputs, the
    # call, D2H of the scores, every step
    e2e = e2e_run(case, device, stream, args, steps=min(steps, 5 if case.T * case.H_q > 1e6 else 20))
    # the block top-k selection over this call's scores (the scores' consumer;
    # not part of the metric above), and the fused per-group selection
    topk = topk_run(prep.out, case.MB, 16, device, stream, peaks, min(steps * 5, 200))
    fused = fused_select_run(case, prep, device, stream, min(steps, 30), head, topk)
    sparse = sparse_run(case, prep, device, stream, peaks, min(steps, 10))
    del prep
    torch.cuda.empty_cache()

    line = {
        "metric": METRIC, "value": head["value"], "unit": "us/call", "n_gpus": ws,
        "steps": steps, "warmup": args.warmup, "ms_per_step": head["ms_per_step"],
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None,
        "dtype": dtype_name(case),
        "data": "synthetic (seeded; shapes and length mix of the workload recipe)",
        "config": config_block(case, key),
        "tflops": head["tflops"], "k_cache_gbs": head["k_cache_gbs"],
        "frac_hbm": head["frac_hbm"], "frac_tensor": head["frac_tensor"],
        "roofline": head["roofline"],
        "e2e": e2e,
        "topk": topk,
        "fused_select": fused,
        "sparse_attention": sparse,
        "gpu_launches": head["gpu_launches"],
        "clocks": head["clocks"],
    }
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_oracle_baseline(case)
    del case

    # the other workloads (and the int8 decode subset), each measured the same way
    if not args.no_sub and args.workload == DEFAULT_WORKLOAD and not args.decode_subset \
            and args.layout is None and args.fp8 is None and args.fp4 is None \
            and getattr(args, "q_len", None) is None:
        subs = []
        for n, dsub, fp4 in SUB_WORKLOADS:
            sa = argparse.Namespace(workload=n, decode_subset=dsub, layout=None, fp8=None,
                                    fp4=fp4, q_len=None, steps=None)
            scase = make_workload(sa)
            skey = workload_key(sa)
            rec, sprep = measure(scase, skey, default_steps(sa), args.warmup, device, stream,
                                 peaks, ws, recorded_traffic(skey, dominant_kernel(scase)))
            rec["topk"] = topk_run(sprep.out, scase.MB, 16, device, stream, peaks, 200)
            rec["fused_select"] = fused_select_run(scase, sprep, device, stream, 30, rec, rec["topk"])
            if n == 3 and fp4 is None:
                rec["sparse_attention"] = sparse_run(scase, sprep, device, stream, peaks, 20)
            del sprep
            rec["e2e"] = e2e_run(scase, device, stream, args, steps=20)
            if rank == 0 and ws == 1 and not args.no_cpu_baseline:
                rec["cpu_baseline"] = cpu_oracle_baseline(scase, target_s=3.0)
            rec["config"] = config_block(scase, skey)
            subs.append(rec)
            del scase
            torch.cuda.empty_cache()
        line["sub_workloads"] = subs
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def fused_select_run(case, prep, device, stream, steps, head, topk):
    """The fused per-group selection (msa_index_score_topk, k = 16, own-block
    slot on), with and without storing the scores: microseconds per call of
    the whole op, against one score call plus the unfused top-k over its
    scores."""
    if 32 % (case.H_q // case.H_kv) or getattr(case, "fp4", None):
        return None
    res = {"k": 16, "local_slot": True, "groups": case.H_kv,
           "rows": case.T * case.H_kv, "unfused_us": head["value"] + topk["us_per_call"]}
    ws = torch.empty(prep.select_workspace_bytes(16), dtype=torch.uint8, device=device)
    idx = torch.empty((case.T, case.H_kv, 16), dtype=torch.int32, device=device)
    for scores in (True, False):
        for _ in range(3):
            prep.topk(16, True, scores, idx, ws, stream)
        torch.cuda.synchronize(device)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            prep.topk(16, True, scores, idx, ws, stream)
        e1.record(stream)
        torch.cuda.synchronize(device)
        res["with_scores_us" if scores else "without_scores_us"] = e0.elapsed_time(e1) / steps * 1e3
    if prep.select_device_error(stream):
        raise RuntimeError("device error in the fused selection")
    res["workspace_bytes"] = ws.numel()
    res["launches_per_call"] = launches_per_call(case) + 1
    return res


def sparse_work(case, sel):
    """Algorithmic work of the sparse main branch for selection ``sel``
    ``[T, H_kv, k]``: FLOPs = 4 * D * sum over (token, head) of the visible
    keys in its selected blocks (S = Q K^T and O = P V); bytes = the query,
    the K and V pages of every distinct selected (kv head, request, block)
    once, the fp32 output and LSE."""
    import numpy as np
    sel = sel.cpu().numpy().astype(np.int64)
    T, H_kv, k = sel.shape
    g = case.H_q // case.H_kv
    P, D = case.P, case.D
    cu = case.cu_seqlens_q.tolist()
    req = np.zeros(T, dtype=np.int64)
    for b in range(len(cu) - 1):
        req[cu[b]:cu[b + 1]] = b
    L = np.asarray(case.kv_lens, dtype=np.int64)[req]                  # [T]
    Lq = np.asarray(case.q_lens, dtype=np.int64)[req]
    qpos = L - Lq + (np.arange(T) - np.asarray(cu[:-1], dtype=np.int64)[req])
    last = np.minimum(L - 1, qpos) if case.sparse_mode == 3 else L - 1  # last visible key
    nb = -(-L // P)
    valid = (sel >= 0) & (sel < case.MB) & (sel < nb[:, None, None])
    vis = np.clip(last[:, None, None] + 1 - sel * P, 0, P) * valid
    flops = 4.0 * D * g * float(vis.sum())
    blocks = set()
    for r in range(H_kv):
        t_idx, s_idx = np.nonzero(valid[:, r, :])
        blocks.update(zip([r] * len(t_idx), req[t_idx].tolist(), sel[t_idx, r, s_idx].tolist()))
    es = case.key.element_size()
    nbytes = (case.T * case.H_q * D * case.query.element_size() + len(blocks) * 2 * P * D * es
              + case.T * case.H_q * (D + 1) * 4)
    return flops, nbytes, len(blocks)


def sparse_run(case, prep, device, stream, peaks, steps: int):
    """The sparse main branch (msa_sparse_attention) over the fused top-16
    selection of this workload, the workload's query and keys as the main
    branch's, random values of the key cache's layout: microseconds per call."""
    if (case.key.dtype not in (torch.float16, torch.bfloat16) or getattr(case, "fp4", None)
            or 32 % (case.H_q // case.H_kv)):
        return None
    sel = prep.topk(16, local_slot=True, scores=False, stream=stream)
    key = prep.call.key
    base = key
    while base._base is not None:
        base = base._base
    gen = torch.Generator(device=device).manual_seed(99)
    vbase = torch.randn(base.shape, generator=gen, device=device, dtype=torch.float32).to(key.dtype)
    value = torch.as_strided(vbase, key.shape, key.stride(), key.storage_offset())
    out, lse = prep.sparse_attention(value, sel, stream=stream)
    for _ in range(2):
        prep.sparse_attention(value, sel, out=out, lse=lse, workspace=prep.sparse_workspace,
                              stream=stream)
    torch.cuda.synchronize(device)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        prep.sparse_attention(value, sel, out=out, lse=lse, workspace=prep.sparse_workspace,
                              stream=stream)
    e1.record(stream)
    torch.cuda.synchronize(device)
    if prep.sparse_device_error(stream):
        raise RuntimeError("device error in the sparse attention")
    us = e0.elapsed_time(e1) / steps * 1e3
    flops, nbytes, nblocks = sparse_work(case, sel)
    tfl = flops / us / 1e6
    gbs = nbytes / us / 1e3
    bound = "tensor" if flops / (peaks["bf16_tflops"] * 1e12) >= nbytes / (peaks["hbm_gbs"] * 1e9) else "hbm"
    res = {"k": 16, "selection": "fused per-group top-16 with the own-block slot",
           "us_per_call": us, "tflops": tfl, "gbs": gbs, "algorithmic_flops": flops,
           "algorithmic_bytes": nbytes, "selected_blocks": nblocks, "bound": bound,
           "frac": (tfl / peaks["bf16_tflops"]) if bound == "tensor" else (gbs / peaks["hbm_gbs"]),
           "partials_bytes": case.T * case.H_q * 16 * (case.D * 2 + 4) * 2,
           "kernels": "count, scan, scatter, units, K1 (sparse_k1_kernel), K2 (combine); 2 memsets"}
    del vbase, value, out, lse
    return res


def topk_run(score, MB: int, k: int, device, stream, peaks, steps: int):
    """Time msa_block_topk over a score tensor: events around each launch."""
    import block_score_gb300 as bs
    H, T, MBp = score.shape
    out = bs.msa_block_topk(score, k=k, MB=MB, stream=stream)
    for _ in range(3):
        bs.msa_block_topk(score, k=k, MB=MB, out=out, stream=stream)
    torch.cuda.synchronize(device)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    for a, b in evs:
        a.record(stream)
        bs.msa_block_topk(score, k=k, MB=MB, out=out, stream=stream)
        b.record(stream)
    torch.cuda.synchronize(device)
    us = statistics.mean(a.elapsed_time(b) for a, b in evs) * 1e3
    nbytes = H * T * MBp * 4 + T * H * k * 4      # scores read once, indices written
    gbs = nbytes / us / 1e3
    return {"k": k, "rows": H * T, "us_per_call": us, "bytes": nbytes, "achieved_gbs": gbs,
            "peak_gbs": peaks["hbm_gbs"], "frac": gbs / peaks["hbm_gbs"],
            "inputs_in_l2": nbytes < L2_BYTES, "kernel": "topk_kernel"}


def e2e_run(case, device, stream, args, steps=None):
    """Same metric through the public call with pinned host inputs."""
    import block_score_gb300 as bs
    host = {}
    for name in ("query", "block_table", "cu_seqlens_q", "kv_len", "cu_seqlens_k",
                 "start_loc", "scale", "q_scale", "k_scale"):
        t = getattr(case, name, None)
        host[name] = None if t is None else t.contiguous().pin_memory()
    key = case.key
    base = key
    while base._base is not None:
        base = base._base
    host_key_base = base.contiguous().pin_memory()
    dev = {k: (None if v is None else torch.empty_like(v, device=device)) for k, v in host.items()}
    key_base_dev = torch.empty_like(host_key_base, device=device)
    key_dev = torch.as_strided(key_base_dev, key.shape, key.stride(), key.storage_offset())
    klen = dev["cu_seqlens_k"] if case.layout == "TND" else dev["kv_len"]
    prep = bs.Prepared(dev["query"], key_dev, dev["start_loc"], block_table=dev["block_table"],
                       scale=dev["scale"], actual_seq_qlen=dev["cu_seqlens_q"],
                       actual_seq_klen=klen, layout_key=case.layout,
                       sparse_mode=case.sparse_mode, init_blocks=case.init_blocks,
                       local_blocks=case.local_blocks,
                       max_blocks=case.MB if case.layout == "TND" else None,
                       max_seqlen_q=max(case.q_lens) if case.q_lens else None,
                       **(dict(fp4=case.fp4, q_scale=dev["q_scale"], k_scale=dev["k_scale"])
                          if getattr(case, "fp4", None) else {}))
    out_host = torch.empty(prep.shape, dtype=torch.float32, pin_memory=True)
    h2d = sum(v.numel() * v.element_size() for v in host.values() if v is not None)
    h2d += host_key_base.numel() * host_key_base.element_size()
    d2h = out_host.numel() * 4

    def step():
        for k, v in host.items():
            if v is not None:
                dev[k].copy_(v, non_blocking=True)
        key_base_dev.copy_(host_key_base, non_blocking=True)
        prep(stream)
        out_host.copy_(prep.out, non_blocking=True)

    steps = max(1, steps if steps is not None else 20)
    for _ in range(min(args.warmup, 3)):
        step()
    torch.cuda.synchronize(device)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize(device)
    ms = e0.elapsed_time(e1) / steps
    return {"value": ms * 1e3, "unit": "us/call", "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(d2h), "steps": steps}


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None,
                    help="calls per timed pass (default: per workload, ~0.2-0.6 s of GPU time)")
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", type=int, default=DEFAULT_WORKLOAD, choices=[1, 2, 3, 4, 5])
    ap.add_argument("--decode-subset", action="store_true",
                    help="time only the single-token requests of the workload (cfg4)")
    ap.add_argument("--layout", choices=["BBND", "BNBD", "TND"], default=None,
                    help="draw the workload's keys in another layout (same lengths)")
    ap.add_argument("--fp8", choices=sorted(FP8), default=None,
                    help="run the (fp16 / bf16) workload with FP8 query and keys")
    ap.add_argument("--fp4", choices=["mx", "nv"], default=None,
                    help="run the (fp16 / bf16) workload with FP4 query and keys (MXFP4 / NVFP4)")
    ap.add_argument("--q-len", type=int, default=None,
                    help="workload 5 only: its last Q_LEN query positions (profiler captures)")
    ap.add_argument("--no-sub", action="store_true",
                    help="measure the selected workload only (no sub-records)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--sparse-only", action="store_true",
                    help="time only the sparse main branch (msa_sparse_attention) on the workload")
    ap.add_argument("--traffic", type=float, default=None,
                    help="DRAM bytes per launch of the score kernel from an ncu capture")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
