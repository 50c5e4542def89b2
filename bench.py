"""Bench: fused residual-add + RMSNorm (and its no-residual variant) on GB300.

One step = one pass of the whole hot path over one batch of the fp16
65536 x 8192 workload (the largest one-GPU workload; per-row log-uniform scales
in [0.1, 10]): fused_add_rmsnorm(x, r, w) -> (out, residual_out), then
rmsnorm(x, w) -> out2 on the same x.  Inputs are resident in HBM when the
timed region starts; every tensor (1 GiB each) is far larger than the 129 MB
L2, so no flush is needed between steps.

Metric: achieved HBM GB/s from the algorithmic bytes (x, r, out, residual_out
once each plus w once for the fused op; x, out2 plus w for the variant),
tokens/s beside it.  Also reported: the end-to-end rate through the host-buffer
entry points (copies inside the timed region), the dominant kernel's roofline
from its own CUDA-event-timed launches, SM clocks sampled during the timed
region, and the CPU oracle timed on the host cores as a baseline.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl far|reference]
                  [--op rmsnorm|layernorm|rmsnorm_int8|rmsnorm_fp8]
                  [--row-schedule claimed|fixed]
Under torchrun each rank runs its own replica (weak scaling, no collective on
the data path); rank 0 prints one JSON line.  --op measures one of the other
operations of the library the same way (its fused form, then its no-residual
variant), the end-to-end leg through that op's host-buffer entry points.

For the RMSNorm op the line also carries `configs`: every workload (bf16
8x2048 up to fp16 65536x8192), the fused op and the variant each, timed per
launch with CUDA events both after an L2 read sweep and back to back, with the
mean, median, min and max launch time, GB/s, tokens/s and the fraction of the
measured copy rate.

--row-schedule: `claimed` (the default here) opts in to rows claimed from a
per-launch counter by the library's automatic rule (far_set_row_schedule(0));
`fixed` times the library's default, the fixed stride (mode 1), which keeps no
state between calls.  The line says which was timed.
"""
from __future__ import annotations

import argparse
import csv
import hashlib
import io
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

METRIC = "achieved HBM GB/s and tokens/s of fused add+RMSNorm at 1 GB300 (% of HBM peak)"
OP_METRIC = {
    "rmsnorm": METRIC,
    "layernorm": "achieved HBM GB/s and tokens/s of fused add+LayerNorm at 1 GB300 (% of HBM peak)",
    "rmsnorm_int8": "achieved HBM GB/s and tokens/s of fused add+RMSNorm with int8 per-token output at 1 GB300",
    "rmsnorm_fp8": "achieved HBM GB/s and tokens/s of fused add+RMSNorm with FP8 E4M3 per-token output at 1 GB300",
    "gemm": "achieved TFLOP/s of the fp16-storage / fp32-compute GEMM y = fp16(x @ wt^T) + bias at 1 GB300",
}
OP_STEP = {
    "rmsnorm": "fused_add_rmsnorm then rmsnorm on the same x",
    "layernorm": "fused_add_layernorm then layernorm on the same x",
    "rmsnorm_int8": "fused_add_rmsnorm_quant then rmsnorm_quant (int8) on the same x",
    "rmsnorm_fp8": "fused_add_rmsnorm_quant then rmsnorm_quant (FP8 E4M3) on the same x",
    "gemm": "gemm_f16_f32acc with an fp16 bias and fp16 output",
}
WORKLOAD = "c5"
CSRC = os.path.join(ROOT, "mixed_precision_residual_gb300", "csrc")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")
DSIZE = {torch.float16: 2, torch.bfloat16: 2, torch.float32: 4}


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["far", "reference"], default="far")
    ap.add_argument("--workload", default=WORKLOAD)
    ap.add_argument("--tokens", type=int, default=0,
                    help="time only the first N rows of the workload (profiling captures)")
    ap.add_argument("--e2e-steps", type=int, default=4)
    ap.add_argument("--e2e-chunk", type=int, default=4096, help="rows per chunk of the host-buffer pipeline")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--op", choices=sorted(OP_METRIC), default="rmsnorm")
    ap.add_argument("--gemm-shape", default="8192x8192x8192", help="M x N x K of the GEMM op")
    ap.add_argument("--row-schedule", choices=["claimed", "fixed"], default="claimed",
                    help="claimed: the library's opt-in automatic claimed-row rule; fixed: its default")
    ap.add_argument("--config-launches", type=int, default=30,
                    help="launches timed per workload, op and L2 condition in `configs` (0: none)")
    return ap.parse_args()


ROW_SCHEDULE_MODE = {"claimed": 0, "fixed": 1}
ROW_SCHEDULE_TEXT = {"claimed": "claimed rows by the automatic rule (opt-in: far_set_row_schedule(0))",
                     "fixed": "fixed stride (the library default, far_set_row_schedule(1))"}


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(value: float, dist, device) -> float:
    """The largest of every rank's value (the job's time is its slowest rank's)."""
    if dist is None:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(units_per_rank: float, world: int, ms_per_step: float) -> float:
    """Whole-job rate: the units all ranks processed in one step over the slowest rank's step time."""
    return units_per_rank * world / (ms_per_step * 1e-3)


def step_bytes(tokens, hidden, act, wd, od, op="rmsnorm"):
    """Algorithmic bytes of one step: (fused, variant).

    Each input and output byte once, the weight once per launch (LayerNorm: gamma and
    beta); a quantised output is one byte an element plus a binary32 scale per row."""
    sa, sw, so = DSIZE[act], DSIZE[wd], DSIZE[od]
    nw = 2 if op == "layernorm" else 1
    if op.startswith("rmsnorm_"):
        fused = tokens * hidden * (3 * sa + 1) + 4 * tokens + hidden * sw
        norm = tokens * hidden * (sa + 1) + 4 * tokens + hidden * sw
        return fused, norm
    fused = tokens * hidden * (2 * sa + sa + so) + nw * hidden * sw
    norm = tokens * hidden * (sa + so) + nw * hidden * sw
    return fused, norm


def oracle_step(op, d, x, r, threads):
    """The oracle, as it stands, on rows x (and residual r): the fused op, then the variant."""
    import oracle

    act, wd, eps = d["act"], d["wd"], d["eps"]
    if op == "rmsnorm":
        oracle.fused_add_rmsnorm(x, r, d["w"], eps, act, wd, threads=threads)
        oracle.rmsnorm(x, d["w"], eps, act, wd, threads=threads)
    elif op == "layernorm":
        oracle.fused_add_layernorm(x, r, d["w"], d["b"], eps, act, wd, threads=threads)
        oracle.layernorm(x, d["w"], d["b"], eps, act, wd, threads=threads)
    else:
        q = op.split("_")[1]
        oracle.fused_add_rmsnorm_quant(x, r, d["w"], eps, act, wd, q, threads=threads)
        oracle.rmsnorm_quant(x, d["w"], eps, act, wd, q, threads=threads)


KERNEL_SOURCES = ("far_kernels.cuh", "far_device.cuh", "far_params.h")


def source_hash() -> str:
    """Hash of the sources that define the staged kernel (the captured counters' validity)."""
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(CSRC, f), "rb") as fh:
            h.update(f.encode() + fh.read())
    return h.hexdigest()[:16]


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


PLAN_KEYS = ("kind", "nch", "warps_per_row", "groups", "stages")


def traffic_from_profile(workload: str, op: str = "rmsnorm", plan: dict | None = None, tokens: int | None = None):
    """DRAM bytes per fused launch from a committed ncu summary, if the kernel sources, the
    launch plan and the token count are still the captured ones."""
    if not os.path.exists(TRAFFIC_FILE):
        return None
    with open(TRAFFIC_FILE) as f:
        d = json.load(f)
    e = d.get(workload if op == "rmsnorm" else f"{workload}:{op}")
    if not e or e.get("source_hash") != source_hash():
        return None
    if plan is not None and e.get("launch_plan") != [plan[k] for k in PLAN_KEYS]:
        return None
    if tokens is not None and e.get("captured_tokens") != tokens:
        return None
    return e.get("dram_bytes_per_launch")


def row_schedule_text(far, claimed, tokens, hidden, act, wd, residual, op, sms):
    """How a launch's CTAs shared rows (the library's flag after the launch, and its rule for
    the rows a claim)."""
    if not claimed:
        return "fixed stride"
    n = far.row_schedule_for_sms(tokens, hidden, act, wd, residual,
                                 {"rmsnorm": "rmsnorm", "layernorm": "layernorm"}.get(op, "quant"), sms)
    # the automatic rule's three-row claims cover only the last quarter of each CTA's rows
    tail = ", over the last quarter of each CTA's rows" if n == 3 and far.get_row_schedule() == 0 else ""
    return f"rows claimed from a per-launch counter, {n} a claim{tail}"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.dev}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.3)  # let the first sample land before the timed region
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.15)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sms, maxes, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for row in csv.reader(io.StringIO(out)):
            if len(row) < 9:
                continue
            try:
                sms.append(float(row[1]))
                maxes.append(float(row[2]))
                power.append(float(row[3]))
            except ValueError:
                continue
            for name, v in zip(names, row[5:9]):
                if v.strip().lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sms) if sms else None, "sm_max_mhz": max(maxes) if maxes else None,
                "reasons": sorted(reasons), "samples": len(sms),
                "power_w_median": statistics.median(power) if power else None}


# Arm core names by (implementer, part), for CPUs whose /proc/cpuinfo gives no model name
ARM_PARTS = {(0x41, 0xd4f): "Arm Neoverse-V2", (0x41, 0xd40): "Arm Neoverse-V1", (0x41, 0xd0c): "Arm Neoverse-N1",
             (0x41, 0xd49): "Arm Neoverse-N2", (0x41, 0xd8f): "Arm Neoverse-V3"}


def cpu_model() -> str:
    """The host CPU's model, from /proc/cpuinfo (x86: its model name; Arm: the core named by
    implementer and part), with the logical CPU count."""
    try:
        with open("/proc/cpuinfo") as f:
            text = f.read()
    except OSError:
        return "unknown"
    fields = {}
    for line in text.splitlines():
        if ":" in line:
            k, v = line.split(":", 1)
            fields.setdefault(k.strip().lower(), v.strip())
    n = os.cpu_count() or 0
    if "model name" in fields:
        return f"{fields['model name']} ({n} logical CPUs)"
    try:
        key = (int(fields.get("cpu implementer", "0"), 0), int(fields.get("cpu part", "0"), 0))
    except ValueError:
        key = (0, 0)
    if key in ARM_PARTS:
        return f"{ARM_PARTS[key]} ({n} logical CPUs)"
    if key != (0, 0):
        return f"Arm implementer {key[0]:#x} part {key[1]:#x} ({n} logical CPUs)"
    return f"unknown ({n} logical CPUs)"


def oracle_sample(d, seconds: float, op: str, threads: int):
    """The oracle, as it stands, on the first rows of the batch (fused + variant) for about
    `seconds`: rows done and elapsed seconds."""
    rows_done, t0 = 0, time.perf_counter()
    chunk = max(threads * 4, 64)
    while time.perf_counter() - t0 < seconds and rows_done < d["tokens"]:
        sl = slice(rows_done, min(d["tokens"], rows_done + chunk))
        oracle_step(op, d, d["x"][sl], d["r"][sl], threads)
        rows_done = sl.stop
    return rows_done, time.perf_counter() - t0


def cpu_baseline(d, seconds: float, op: str = "rmsnorm"):
    """The oracle, as it stands, timed on the host cores on the first rows of the batch:
    on every core (row blocks over threads), then on one thread; GB/s of the same
    algorithmic bytes, tokens/s, and the CPU model."""
    import oracle

    threads = oracle.default_threads()
    H = d["hidden"]
    act, wd = d["act"], d["wd"]
    od = "f32" if "f32" in (act, wd) else act
    tdt = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}
    model = cpu_model()
    legs = {}
    for name, n, secs in (("threads_all", threads, seconds), ("threads_1", 1, seconds / 2)):
        rows_done, el = oracle_sample(d, secs, op, n)
        fb, nb = step_bytes(rows_done, H, tdt[act], tdt[wd], tdt[od], op)
        legs[name] = {"value": round((fb + nb) / el / 1e9, 4), "unit": "GB/s", "threads": n,
                      "seconds": round(el, 2), "tokens_per_s": round(rows_done / el, 1),
                      "sample": f"first {rows_done} of {d['tokens']} rows of the {d['workload']} batch"}
    return {"value": legs["threads_all"]["value"], "unit": "GB/s", "cores": threads, "kind": "oracle",
            "cpu_model": model, "seconds": legs["threads_all"]["seconds"],
            "tokens_per_s": legs["threads_all"]["tokens_per_s"],
            "sample": f"{legs['threads_all']['sample']}, {OP_STEP[op]}, oracle on {threads} host threads "
                      f"(row blocks over threads); threads_1: the same on one thread",
            "threads_all": legs["threads_all"], "threads_1": legs["threads_1"]}


def launch_stats(ms):
    """Mean, median, min and max of per-launch times (ms)."""
    return {"mean_ms": round(statistics.fmean(ms), 5), "median_ms": round(statistics.median(ms), 5),
            "min_ms": round(min(ms), 5), "max_ms": round(max(ms), 5), "launches": len(ms)}


def time_launches(fn, stream, n, flush=None):
    """CUDA-event times (ms) of n launches of fn on `stream` (torch's current stream): back to
    back, or each after a read sweep of `flush` (outside the events), which leaves the L2
    holding no line of the launch's tensors and no dirty line to write back."""
    ev0 = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
    ev1 = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
    for k in range(n):
        if flush is not None:
            flush.sum()
        ev0[k].record(stream)
        if fn():
            raise RuntimeError("launch failed")
        ev1[k].record(stream)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in zip(ev0, ev1)]


def time_stream(fn, stream, n, blocks=5):
    """Launches in a stream: `blocks` blocks of n launches back to back, each block between
    two CUDA events (no event between launches, so a launch may be dispatched while the one
    ahead of it finishes); each block's mean time a launch (ms)."""
    out = []
    for _ in range(blocks):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(n):
            if fn():
                raise RuntimeError("launch failed")
        b.record(stream)
        torch.cuda.synchronize()
        out.append(a.elapsed_time(b) / n)
    return out


def measure_configs(far, dev, stream, launches, flush, peak, sms, resident=None):
    """Every workload's fused add+RMSNorm and no-residual RMSNorm, timed per launch both after
    an L2 read sweep and back to back; GB/s and tokens/s from the mean launch time, the
    fraction of the measured copy rate, and the spread.  `resident` maps a workload name to
    device tensors already allocated (the bench step's own batch)."""
    import far_gen

    L = far.lib
    sh = stream.cuda_stream
    entries = []
    for name in ("c1", "c2", "c3", "c4", "c5"):
        w = far_gen.WORKLOADS[name]
        if resident and name in resident:
            x, r, wt, eps = resident[name]
        else:
            d = far_gen.make_inputs(w)
            x, r, wt, eps = d["x"].to(dev), d["r"].to(dev), d["w"].to(dev), d["eps"]
        T, H = x.shape
        od = far.output_dtype(x.dtype, wt.dtype)
        out = torch.empty(x.shape, dtype=od, device=dev)
        res = torch.empty_like(x)
        out2 = torch.empty(x.shape, dtype=od, device=dev)
        code = far.dtypes(x.dtype, wt.dtype)
        xp, rp, wp, op, rop, o2p = (t.data_ptr() for t in (x, r, wt, out, res, out2))
        fb, nb = step_bytes(T, H, x.dtype, wt.dtype, od)
        ops = (("fused", lambda: L.fused_add_rmsnorm(xp, rp, wp, eps, op, rop, T, H, code, sh), fb, True),
               ("variant", lambda: L.rmsnorm(xp, wp, eps, o2p, T, H, code, sh), nb, False))
        e = {"workload": name, "note": w.note, "tokens": T, "hidden": H, "act_dtype": w.act, "weight_dtype": w.wd}
        for kind, fn, nbytes, residual in ops:
            for _ in range(3):
                if fn():
                    raise RuntimeError(f"{name} {kind} launch failed")
            claimed = far.last_launch_claimed_rows()
            torch.cuda.synchronize()
            k = {"algorithmic_bytes_per_launch": nbytes,
                 "launch_plan": far.describe_launch(T, H, x.dtype, wt.dtype, residual),
                 "row_schedule": row_schedule_text(far, claimed, T, H, x.dtype, wt.dtype, residual, "rmsnorm", sms)}
            for cond in ("flushed", "back_to_back", "stream"):
                if cond == "stream":
                    ms = time_stream(fn, stream, max(2, launches // 3))
                else:
                    ms = time_launches(fn, stream, launches, flush if cond == "flushed" else None)
                st = launch_stats(ms)
                gbs = nbytes / (st["mean_ms"] * 1e-3) / 1e9
                k[cond] = {"gbs": round(gbs, 1), "tokens_per_s": round(T / (st["mean_ms"] * 1e-3), 1),
                           "frac": round(gbs / peak, 4), **st}
                if cond == "stream":
                    k[cond]["launches"] = f"{len(ms)} blocks of {max(2, launches // 3)}"
            e[kind] = k
        if far.device_status() != 0:
            raise RuntimeError(f"device status after the {name} launches")
        entries.append(e)
        del out, res, out2
    return entries


def run_reference(args):
    """--impl reference: the CPU oracle timed on the host cores, each step a bounded row sample."""
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    import far_gen
    import oracle

    w = far_gen.WORKLOADS[args.workload]
    threads = oracle.default_threads()
    probe = far_gen.make_inputs(w, rows=threads * 2)
    probe["b"] = far_gen.ln_beta(probe)
    t0 = time.perf_counter()
    oracle_step(args.op, probe, probe["x"], probe["r"], threads)
    per_row = (time.perf_counter() - t0) / (threads * 2)
    budget = 120.0  # seconds for all steps
    rows = int(max(threads, min(w.tokens, budget / max(1, args.steps + args.warmup) / max(per_row, 1e-9))))
    d = far_gen.make_inputs(w, rows=rows)
    d["b"] = far_gen.ln_beta(d)
    for _ in range(args.warmup):
        oracle_step(args.op, d, d["x"], d["r"], threads)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_step(args.op, d, d["x"], d["r"], threads)
    el = time.perf_counter() - t0
    tdt = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}
    od = "f32" if "f32" in (w.act, w.wd) else w.act
    fb, nb = step_bytes(rows, w.hidden, tdt[w.act], tdt[w.wd], tdt[od], args.op)
    value = (fb + nb) * args.steps / el / 1e9
    sample = (f"{rows} of {w.tokens} rows of the {w.name} batch per step ({OP_STEP[args.op]}), "
              f"oracle on {threads} host threads")
    line = {"impl": "reference", "metric": OP_METRIC[args.op], "value": round(value, 4), "unit": "GB/s",
            "n_gpus": args.gpus, "compute": "host cores (the oracle; no GPU work)",
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(el / args.steps * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": w.act,
            "data": "synthetic (seeded Philox4x32-10 generator)",
            "config": {"workload": f"{w.name}: {w.note}", "tokens": w.tokens, "hidden": w.hidden,
                       "act_dtype": w.act, "weight_dtype": w.wd, "eps": w.eps, "rows_per_step": rows},
            "tokens_per_s": round(rows * args.steps / el, 1),
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def gemm_shape(args):
    M, N, K = (int(v) for v in args.gemm_shape.lower().split("x"))
    return M, N, K


def gemm_oracle_sample(d, seconds, threads=None):
    """The GEMM oracle, as it stands, on the first rows of x (all of N and K): TFLOP/s."""
    import oracle

    threads = threads or oracle.default_threads()
    N, K = d["N"], d["K"]
    rows, t0 = 0, time.perf_counter()
    step = max(1, threads)
    while time.perf_counter() - t0 < seconds and rows < d["M"]:
        oracle.gemm_f16(d["x"][rows:rows + step], d["wt"], d["bias"], "f16", threads=threads)
        rows += step
    el = time.perf_counter() - t0
    return rows, el, threads


def run_gemm_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    import far_gen

    M, N, K = gemm_shape(args)
    d = far_gen.gemm_inputs(M, N, K, seed=0)
    per_step = 120.0 / max(1, args.steps + args.warmup)
    for _ in range(args.warmup):
        gemm_oracle_sample(d, per_step)
    total_rows, total_s, threads = 0, 0.0, 1
    for _ in range(args.steps):
        rows, el, threads = gemm_oracle_sample(d, per_step)
        total_rows, total_s = total_rows + rows, total_s + el
    value = 2.0 * total_rows * N * K / total_s / 1e12
    sample = f"the first rows of x (all {N} columns, K = {K}) per step, about {per_step:.1f} s each, oracle on {threads} host threads"
    line = {"impl": "reference", "metric": OP_METRIC["gemm"], "value": round(value, 8), "unit": "TFLOP/s",
            "n_gpus": args.gpus, "compute": "host cores (the oracle; no GPU work)",
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(total_s / args.steps * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f16",
            "data": "synthetic (seeded Philox4x32-10 generator)",
            "config": {"workload": f"gemm {M}x{N}x{K}", "M": M, "N": N, "K": K, "op": "gemm"},
            "cpu_baseline": {"value": round(value, 8), "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(value, 8), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def run_gemm_bench(args):
    """--op gemm: one GEMM launch per step on resident fp16 operands."""
    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group(backend="nccl", device_id=torch.device("cuda", local))
    else:
        dist = None
    import __graft_entry__

    __graft_entry__.build()
    import far_gen
    import mixed_precision_residual_gb300 as far

    M, N, K = gemm_shape(args)
    d = far_gen.gemm_inputs(M, N, K, seed=rank)
    dev = torch.device("cuda", local)
    x, wt, b = d["x"].to(dev), d["wt"].to(dev), d["bias"].to(dev)
    out = torch.empty((M, N), dtype=torch.float16, device=dev)
    stream = torch.cuda.current_stream()
    sh = stream.cuda_stream
    L = far.lib
    xp, wp, bp, op = x.data_ptr(), wt.data_ptr(), b.data_ptr(), out.data_ptr()
    # operands and output are larger than the 129 MB L2 from 4096^3 up; smaller shapes are
    # flushed by a read sweep of a 512 MB buffer before each step (outside the kernel's events)
    flush = torch.ones(128 << 20, dtype=torch.float32, device=dev)
    needs_flush = (M * K + N * K + M * N) * 2 < 3 * (129 << 20)

    def step():
        if L.gemm_f16_f32acc(xp, wp, bp, op, M, N, K, 1, sh):
            raise RuntimeError("gemm launch failed")

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    assert far.device_status() == 0
    ev0 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ev1 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    clocks = ClockSampler(local)
    clocks.start()
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for k in range(args.steps):
        if needs_flush:
            flush.sum()
        ev0[k].record(stream)
        step()
        ev1[k].record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    if dist is not None:
        dist.barrier()
    clk = clocks.stop()
    if far.device_status() != 0:
        raise RuntimeError("device status after the timed region")
    kernel_ms = sum(a.elapsed_time(c) for a, c in zip(ev0, ev1)) / args.steps
    kernel_ms = max_over_ranks(kernel_ms, dist, dev)
    flops = 2.0 * M * N * K
    value = flops * world / (kernel_ms * 1e-3) / 1e12
    peaks = {}
    if os.path.exists(os.path.join(ROOT, "MEASURED_PEAKS.json")):
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            peaks = json.load(f)
    peak = float(peaks.get("bf16_tflops", 1900.0))
    plan = far.plan_gemm_for_sms(M, N, K, True, torch.float16, torch.cuda.get_device_properties(dev).multi_processor_count)
    line = {
        "metric": OP_METRIC["gemm"], "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": max(3, args.warmup), "ms_per_step": round(kernel_ms, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f16",
        "data": "synthetic (seeded Philox4x32-10 generator)",
        "config": {"workload": f"gemm {M}x{N}x{K}", "M": M, "N": N, "K": K, "op": "gemm",
                   "l2": "flushed by a read sweep before each step" if needs_flush else
                         "no flush: operands and output exceed the 129 MB L2",
                   "parallelism": f"replicas x{world}"},
        "gpu_launches": args.steps,
        "roofline": {"bound": "tensor", "achieved": round(flops / (kernel_ms * 1e-3) / 1e12, 2), "peak": peak,
                     "unit": "TFLOP/s", "frac": round(flops / (kernel_ms * 1e-3) / 1e12 / peak, 4), "traffic": None,
                     "kernel": {0: "tc_gemm_kernel", 1: "generic_gemm_kernel", 2: "tc2_gemm_kernel"}.get(plan["kind"], "?"),
                     "peak_source": "measured bf16_tflops (fp16 runs at the bf16 tensor rate)",
                     "algorithmic_flops_per_launch": flops, "avg_launch_ms": round(kernel_ms, 5), "launch_plan": plan},
        "clocks": clk,
        "e2e": None,
        "wall_s": round(wall, 3),
    }
    if rank == 0 and not args.no_cpu_baseline:
        rows, el, threads = gemm_oracle_sample(d, args.cpu_seconds)
        line["cpu_baseline"] = {"value": round(2.0 * rows * N * K / el / 1e12, 8), "unit": "TFLOP/s", "cores": threads,
                                "kind": "oracle", "seconds": round(el, 2),
                                "sample": f"the first {rows} rows of x (all {N} columns, K = {K}), oracle on {threads} host threads"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()
    return 0


def main():
    args = parse_args()
    if args.op == "gemm":
        return run_gemm_reference(args) if args.impl == "reference" else run_gemm_bench(args)
    if args.impl == "reference":
        return run_reference(args)
    rank, world, local = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (there is no CPU fallback)")
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group(backend="nccl", device_id=torch.device("cuda", local))
    else:
        dist = None

    import __graft_entry__

    __graft_entry__.build()
    import far_gen
    import mixed_precision_residual_gb300 as far

    w = far_gen.WORKLOADS[args.workload]
    d = far_gen.make_inputs(w, seed=rank, rows=args.tokens or None)  # each rank its own batch (replica)
    d["b"] = far_gen.ln_beta(d, seed=rank)
    dev = torch.device("cuda", local)
    x, r, wt, bt = d["x"].to(dev), d["r"].to(dev), d["w"].to(dev), d["b"].to(dev)
    od = far.output_dtype(x.dtype, wt.dtype)
    quant = args.op.startswith("rmsnorm_")
    out_dtype = torch.uint8 if quant else od
    out = torch.empty(x.shape, dtype=out_dtype, device=dev)
    res = torch.empty_like(x)
    out2 = torch.empty(x.shape, dtype=out_dtype, device=dev)
    T, H = x.shape
    sc1 = torch.empty(T, dtype=torch.float32, device=dev)
    sc2 = torch.empty(T, dtype=torch.float32, device=dev)
    eps = d["eps"]
    stream = torch.cuda.current_stream()
    sh = stream.cuda_stream
    code = far.dtypes(x.dtype, wt.dtype)
    L = far.lib
    xp, rp, wp, bp, op, rop, o2p = (t.data_ptr() for t in (x, r, wt, bt, out, res, out2))
    s1p, s2p = sc1.data_ptr(), sc2.data_ptr()
    qt = {"rmsnorm_int8": 1, "rmsnorm_fp8": 2}.get(args.op, 0)
    if args.op == "rmsnorm":
        def fused():
            return L.fused_add_rmsnorm(xp, rp, wp, eps, op, rop, T, H, code, sh)

        def variant():
            return L.rmsnorm(xp, wp, eps, o2p, T, H, code, sh)
    elif args.op == "layernorm":
        def fused():
            return L.fused_add_layernorm(xp, rp, wp, bp, eps, op, rop, T, H, code, sh)

        def variant():
            return L.layernorm(xp, wp, bp, eps, o2p, T, H, code, sh)
    else:
        def fused():
            return L.fused_add_rmsnorm_quant(xp, rp, wp, eps, op, s1p, rop, T, H, code, qt, sh)

        def variant():
            return L.rmsnorm_quant(xp, wp, eps, o2p, s2p, T, H, code, qt, sh)

    def step():
        s1 = fused()
        s2 = variant()
        if s1 or s2:
            raise RuntimeError(f"launch failed: {s1} {s2}")

    far.set_row_schedule(ROW_SCHEDULE_MODE[args.row_schedule])
    for _ in range(max(3, args.warmup)):
        step()
    # the row schedule of each kernel (the flag of this thread's last launch), outside the
    # timed region
    if fused():
        raise RuntimeError("fused launch failed")
    rows_fused = far.last_launch_claimed_rows()
    if variant():
        raise RuntimeError("variant launch failed")
    rows_variant = far.last_launch_claimed_rows()
    torch.cuda.synchronize()
    assert far.device_status() == 0

    ev_f0 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ev_f1 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ev_start, ev_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    clocks.start()
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    ev_start.record(stream)
    for k in range(args.steps):
        ev_f0[k].record(stream)
        if fused():
            raise RuntimeError("fused launch failed")
        ev_f1[k].record(stream)
        if variant():
            raise RuntimeError("variant launch failed")
    ev_end.record(stream)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    status = far.device_status()
    if status != 0:
        raise RuntimeError(f"device status {status} after the timed region")
    total_ms = max_over_ranks(ev_start.elapsed_time(ev_end), dist, dev)
    fused_launch_ms = [a.elapsed_time(b) for a, b in zip(ev_f0, ev_f1)]
    fused_ms = sum(fused_launch_ms) / args.steps
    ms_per_step = total_ms / args.steps
    fb, nb = step_bytes(T, H, x.dtype, wt.dtype, od, args.op)
    value = job_rate(fb + nb, world, ms_per_step) / 1e9
    tokens_per_s = job_rate(T, world, ms_per_step)
    peak, peak_kind = measured_peaks()
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    # every workload, fused and variant, flushed and back to back (the RMSNorm op only);
    # the clock sampler keeps running through these launches, so its window is long enough
    # for nvidia-smi's 100 ms samples
    configs = None
    if args.op == "rmsnorm" and args.config_launches > 0 and not args.tokens:
        flush = torch.ones(128 << 20, dtype=torch.float32, device=dev)  # 512 MB read sweep
        configs = measure_configs(far, dev, stream, args.config_launches, flush, peak, sms,
                                  resident={args.workload: (x, r, wt, eps)})
        del flush
    clk = clocks.stop()
    clk["window"] = ("the timed steps" + (" and the per-workload launches after them" if configs else ""))

    # end to end through the host-buffer entry points: copies inside the timed region
    e2e = None
    if args.e2e_steps > 0:
        xh, rh, wh, bh = (t.pin_memory() for t in (d["x"], d["r"], d["w"], d["b"]))
        roh = torch.empty(x.shape, dtype=x.dtype, pin_memory=True)
        chunk = args.e2e_chunk
        host_op = {"rmsnorm": "rmsnorm", "layernorm": "layernorm"}.get(args.op, "quant")
        ws = torch.empty(far.host_workspace_bytes_op(chunk, H, x.dtype, wt.dtype, True, host_op), dtype=torch.uint8,
                         device=dev)
        wsb = ws.numel()
        if quant:
            oh = torch.empty(x.shape, dtype=torch.uint8, pin_memory=True)
            o2h = torch.empty(x.shape, dtype=torch.uint8, pin_memory=True)
            s1h = torch.empty(T, dtype=torch.float32, pin_memory=True)
            s2h = torch.empty(T, dtype=torch.float32, pin_memory=True)
        else:
            oh = torch.empty(x.shape, dtype=od, pin_memory=True)
            o2h = torch.empty(x.shape, dtype=od, pin_memory=True)
        hp = {n: t.data_ptr() for n, t in (("x", xh), ("r", rh), ("w", wh), ("b", bh), ("o", oh), ("ro", roh),
                                             ("o2", o2h), ("ws", ws))}
        if args.op == "rmsnorm":
            path = "fused_add_rmsnorm_host + rmsnorm_host"

            def e2e_calls():
                return (L.fused_add_rmsnorm_host(hp["x"], hp["r"], hp["w"], eps, hp["o"], hp["ro"], T, H, code,
                                                 hp["ws"], wsb, sh),
                        L.rmsnorm_host(hp["x"], hp["w"], eps, hp["o2"], T, H, code, hp["ws"], wsb, sh))
        elif args.op == "layernorm":
            path = "fused_add_layernorm_host + layernorm_host"

            def e2e_calls():
                return (L.fused_add_layernorm_host(hp["x"], hp["r"], hp["w"], hp["b"], eps, hp["o"], hp["ro"], T, H,
                                                   code, hp["ws"], wsb, sh),
                        L.layernorm_host(hp["x"], hp["w"], hp["b"], eps, hp["o2"], T, H, code, hp["ws"], wsb, sh))
        else:
            path = "fused_add_rmsnorm_quant_host + rmsnorm_quant_host"

            def e2e_calls():
                return (L.fused_add_rmsnorm_quant_host(hp["x"], hp["r"], hp["w"], eps, hp["o"], s1h.data_ptr(),
                                                       hp["ro"], T, H, code, qt, hp["ws"], wsb, sh),
                        L.rmsnorm_quant_host(hp["x"], hp["w"], eps, hp["o2"], s2h.data_ptr(), T, H, code, qt,
                                             hp["ws"], wsb, sh))

        def e2e_step():
            s1, s2 = e2e_calls()
            if s1 or s2:
                raise RuntimeError(f"host-buffer launch failed: {s1} {s2}")
        e2e_step()
        torch.cuda.synchronize()
        if dist is not None:
            dist.barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.e2e_steps):
            e2e_step()
        e1.record(stream)
        torch.cuda.synchronize()
        e2e_ms = max_over_ranks(e0.elapsed_time(e1) / args.e2e_steps, dist, dev)
        sa, sw = DSIZE[x.dtype], DSIZE[wt.dtype]
        so = 1 if quant else DSIZE[od]
        nw = 2 if args.op == "layernorm" else 1  # weight rows copied per call (LayerNorm: gamma and beta)
        h2d = T * H * sa * 2 + nw * H * sw + T * H * sa + nw * H * sw
        d2h = T * H * so + T * H * sa + T * H * so + (2 * T * 4 if quant else 0)
        e2e = {"value": round(job_rate(fb + nb, world, e2e_ms) / 1e9, 3), "unit": "GB/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 3),
               "tokens_per_s": round(job_rate(T, world, e2e_ms), 1),
               "path": f"{path} (pinned host buffers, {chunk}-row chunks, two internal streams)"}
        assert far.device_status() == 0

    achieved = fb / (fused_ms * 1e-3) / 1e9
    if args.op == "rmsnorm":
        plan = far.describe_launch(T, H, x.dtype, wt.dtype, True)
    elif args.op == "layernorm":
        plan = far.plan_ln_for_sms(T, H, x.dtype, wt.dtype, True, torch.cuda.get_device_properties(dev).multi_processor_count)
    else:
        plan = far.plan_quant_for_sms(T, H, x.dtype, wt.dtype, True, args.op.split("_")[1],
                                      torch.cuda.get_device_properties(dev).multi_processor_count)
    traffic = traffic_from_profile(args.workload, args.op, plan, T)
    kernel_name = {"rmsnorm": "fused add+RMSNorm", "layernorm": "fused add+LayerNorm",
                   "rmsnorm_int8": "fused add+RMSNorm, int8 output",
                   "rmsnorm_fp8": "fused add+RMSNorm, FP8 output"}[args.op]
    line = {
        "metric": OP_METRIC[args.op], "value": round(value, 3), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": max(3, args.warmup), "ms_per_step": round(ms_per_step, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f16" if x.dtype == torch.float16 else str(x.dtype),
        "data": "synthetic (seeded Philox4x32-10 generator, per-row log-uniform scales)",
        "config": {"workload": f"{w.name}: {w.note}", "tokens": T, "hidden": H,
                   "act_dtype": w.act, "weight_dtype": w.wd, "out_dtype": {"rmsnorm_int8": "int8 + f32 scale per row",
                                 "rmsnorm_fp8": "e4m3 + f32 scale per row"}.get(
                       args.op, w.act if od == x.dtype else "f32"),
                   "eps": eps, "step": OP_STEP[args.op],
                   "l2": "no flush: every tensor (1 GiB) is larger than the 129 MB L2",
                   "parallelism": f"replicas x{world} (rows are independent; no collective)",
                   "op": args.op, "row_schedule": ROW_SCHEDULE_TEXT[args.row_schedule],
                   "launch": ("programmatic dependent launches (the library default)" if far.get_programmatic_launch()
                              else "plain launches")},
        "tokens_per_s": round(tokens_per_s, 1),
        "value_covers": (f"the whole step: both kernels ({OP_STEP[args.op]}), their algorithmic bytes over the "
                         f"step time; the fused kernel alone is `roofline`"),
        "pct_of_hbm_peak": round(100 * value / world / peak, 2),
        "gpu_launches": 2 * args.steps,
        "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": traffic,
                     "kernel": f"staged_kernel ({kernel_name})", "peak_source": f"{peak_kind} hbm_gbs",
                     "algorithmic_bytes_per_launch": fb, "avg_launch_ms": round(fused_ms, 5),
                     "median_launch_ms": round(statistics.median(fused_launch_ms), 5),
                     "min_launch_ms": round(min(fused_launch_ms), 5),
                     "max_launch_ms": round(max(fused_launch_ms), 5),
                     "launch_plan": plan,
                     "row_schedule": {k: row_schedule_text(far, claimed, T, H, x.dtype, wt.dtype, residual, args.op,
                                                           torch.cuda.get_device_properties(dev).multi_processor_count)
                                      for k, claimed, residual in (("fused", rows_fused, True),
                                                                   ("variant", rows_variant, False))}},
        "clocks": clk,
        "e2e": e2e,
    }
    if configs is not None:
        line["configs"] = configs
        line["configs_note"] = (f"per workload: the fused op and the no-residual variant, {args.config_launches} "
                                f"launches each after a 512 MB L2 read sweep (flushed) and {args.config_launches} "
                                f"back to back, each launch between its own CUDA events on the launching stream "
                                f"(on the small workloads these include the host's time to issue the launch); "
                                f"stream: blocks of launches back to back with events only around each block, "
                                f"spread over the block means (programmatic launch lets each launch be "
                                f"dispatched while the one ahead finishes); GB/s and tokens/s from the mean launch "
                                f"time; frac against the measured copy rate {peak} GB/s; row schedule and launch "
                                f"mode as the line's config")
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(d, args.cpu_seconds, args.op)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
