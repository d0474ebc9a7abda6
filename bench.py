#!/usr/bin/env python3
"""RMSNorm forward + backward throughput on GB300: GB/s of logical bytes and
the fraction of the HBM roofline.

One step = one forward (x, w -> y, rstd) and one backward (x, w, dy, rstd ->
dx, dw) over the whole workload, both through the C ABI of librmsnorm.so.
Timing rules:
  * every call is validated (against a float32 PyTorch reference on the GPU)
    before anything is timed;
  * inputs rotate through clone sets whose total size is >= 3x L2, and a
    buffer of 2x L2 is overwritten before every timed call (outside the
    events), so no call is served from L2;
  * each call is bracketed by CUDA events on the stream it is launched on;
  * the HBM roofline is measured in the same run (best of copy, pure write
    and 2-read-1-write probes over 4 GiB, 20 samples each) at the start and
    again after every timed cell, and a closing / opening ratio below 0.98
    is flagged as drift; the measured copy bandwidth
    (MEASURED_PEAKS.json) is the reported `roofline.peak`, and a copy timed
    under the cells' own flush-then-events protocol is reported beside it;
  * `steady` times the same calls back to back with no flush, as in a
    training step, where each call also pays for writing back what the call
    before left dirty in L2;
  * SM clocks and throttle reasons are sampled with nvidia-smi during the
    timed region; before the first launch a read-only nvidia-smi query
    checks that no other process is using the GPU (flagged in `idle_gate`,
    or refused with --require-idle).

The default run also times the width sweep and the other named workloads
(256 x 1024, 32768 x 8192 with outliers, QK-norm 1048576 x 128) under the
same rules, and records the run environment in `env`.

`--impl reference` times the fp64 CPU oracle (the slow, obviously correct
restatement of the method) on the host cores, on a bounded sample of rows of
the same workload.

Multi-GPU (torchrun): RMSNorm rows are independent and every rank runs its
own replica of the workload (weak scaling, no collective on the data path);
the slowest rank's time is reported.
"""
from __future__ import annotations

import argparse
import csv
import dataclasses
import io
import json
import os
import platform
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "RMSNorm fwd+bwd GB/s and % of measured HBM roofline, bf16 M×N sweep"
DEFAULT_WORKLOAD = "hidden4096_16384x4096"
FALLBACK_HBM_GBS = 6800.0
# closing / opening probe ratio below which the run is flagged as drifting
DRIFT_LIMIT = 0.98


# --------------------------------------------------------------------- setup

def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=2000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default=DEFAULT_WORKLOAD)
    p.add_argument("--shape", default=None,
                   help="M,N,dtype (bf16|f16|f32, or bf16_wf32|f16_wf32 for an fp32 weight): "
                        "an ad-hoc workload drawn like the width sweep's, in place of --workload")
    p.add_argument("--op", choices=["norm", "residual", "naive"], default="norm",
                   help="norm: rmsnorm_fwd + rmsnorm_bwd; residual: rmsnorm_add_fwd + "
                        "rmsnorm_add_bwd with dres (residual and dres drawn like x and dy); "
                        "naive: rmsnorm_fwd + the naive three-kernel rmsnorm_bwd_naive "
                        "(ablation)")
    p.add_argument("--e2e-steps", type=int, default=20)
    p.add_argument("--ref-seconds", type=float, default=120.0,
                   help="host time the reference arm (the fp64 oracle) spends over all its "
                        "warm-up and timed steps")
    p.add_argument("--cpu-seconds", type=float, default=10.0,
                   help="CPU oracle budget for the cpu_baseline sample")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-sweep", action="store_true",
                   help="skip the width sweep (every bf16 and fp32 sweep cell, validated and "
                        "timed like the main workload with --sweep-steps steps)")
    p.add_argument("--sweep-steps", type=int, default=30)
    p.add_argument("--no-small-m", action="store_true",
                   help="skip the small-M eager vs CUDA-graph latency table")
    p.add_argument("--no-configs", action="store_true",
                   help="skip the other named workloads (256 x 1024, 32768 x 8192 with "
                        "outliers, QK-norm 1048576 x 128), each validated and timed like the "
                        "main workload with --config-steps steps")
    p.add_argument("--config-steps", type=int, default=100)
    p.add_argument("--steady-steps", type=int, default=500,
                   help="back-to-back forward + backward steps of the steady-state block "
                        "(no flush between calls); 0 skips it")
    p.add_argument("--probe-gib", type=float, default=4.0,
                   help="buffer size of each in-run roofline probe, GiB")
    p.add_argument("--probe-samples", type=int, default=20)
    p.add_argument("--require-idle", action="store_true",
                   help="exit with an error instead of flagging the line when the GPU is "
                        "busy (memory in use or utilisation) before the first launch")
    p.add_argument("--profile", action="store_true",
                   help="lean run for profilers: no probes, validation, e2e or CPU baseline")
    p.add_argument("--json-out", default=None, help="also write the JSON line to this file")
    p.add_argument("--results-dir", default=None,
                   help="write env.json and one JSON line per timed cell (cells.jsonl) here")
    p.add_argument("--resume", action="store_true",
                   help="with --results-dir: take the sweep and workload cells already in "
                        "cells.jsonl instead of timing them again (the main cell is always "
                        "timed)")
    return p.parse_args(argv)


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def read_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def read_profiled_traffic(kernel_tag: str, workload: str, source_hash: str):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the current sources; else None."""
    path = os.path.join(ROOT, "profiles", f"{kernel_tag}_{workload}.md")
    try:
        text = open(path).read()
    except OSError:
        return None
    h = re.search(r"source_hash:\s*([0-9a-f]+)", text)
    t = re.search(r"traffic_bytes_per_launch:\s*([0-9]+)", text)
    if not h or not t or h.group(1) != source_hash:
        return None
    return int(t.group(1))


# ------------------------------------------------------- run environment

def smi_index(local: int) -> str:
    """nvidia-smi's index of this process's GPU `local`: the entry of
    CUDA_VISIBLE_DEVICES when that lists indices, else `local` itself."""
    vis = os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",")
    if local < len(vis) and vis[local].strip().isdigit():
        return vis[local].strip()
    return str(local)


def smi_query(fields: str, index: str) -> list[str] | None:
    """One read-only nvidia-smi query of this GPU; None if it cannot run."""
    try:
        out = subprocess.run(["nvidia-smi", f"--query-gpu={fields}", "--format=csv,noheader,nounits",
                              "-i", index], capture_output=True, text=True, timeout=20)
    except (OSError, subprocess.TimeoutExpired):
        return None
    if out.returncode != 0 or not out.stdout.strip():
        return None
    return [f.strip() for f in out.stdout.strip().splitlines()[0].split(",")]


# A GPU counts as busy when another process holds more memory than a
# driver's idle reservation, or the GPU is computing, before our first launch.
IDLE_MAX_MIB = 1024
IDLE_MAX_UTIL = 5


def assess_idle(samples: list[tuple[float, float]]) -> dict:
    """Whether the GPU was idle over (memory used MiB, utilisation %) samples."""
    if not samples:
        return {"checked": False, "busy": None}
    mem = max(s[0] for s in samples)
    util = max(s[1] for s in samples)
    return {"checked": True, "busy": mem > IDLE_MAX_MIB or util > IDLE_MAX_UTIL,
            "memory_used_mib_max": mem, "utilization_pct_max": util, "samples": len(samples),
            "limits": {"memory_used_mib": IDLE_MAX_MIB, "utilization_pct": IDLE_MAX_UTIL}}


def idle_gate(local: int) -> dict:
    """Reads memory used and utilisation of this GPU three times, 0.2 s
    apart, before this process creates its CUDA context ("What a tuned
    RMSNorm kernel actually costs on Hopper", section 02: the sweep starts
    only on an idle GPU). Read-only: nothing is changed on the device."""
    samples = []
    for k in range(3):
        rec = smi_query("memory.used,utilization.gpu", smi_index(local))
        if rec is not None:
            try:
                samples.append((float(rec[0]), float(rec[1])))
            except (ValueError, IndexError):
                pass
        if k < 2:
            time.sleep(0.2)
    return assess_idle(samples)


def env_record(torch, local: int, l2: int) -> dict:
    """What the numbers were measured on: GPU, driver, toolkit, PyTorch,
    host and the library's sources."""
    from memory_bound_normalization_gb300 import build as libbuild

    props = torch.cuda.get_device_properties(local)
    drv = smi_query("driver_version", smi_index(local))
    nvcc = None
    try:
        out = subprocess.run([libbuild._nvcc(), "--version"], capture_output=True, text=True,
                             timeout=20)
        m = re.search(r"release ([0-9.]+), V([0-9.]+)", out.stdout)
        nvcc = m.group(2) if m else None
    except (OSError, RuntimeError, subprocess.TimeoutExpired):
        pass
    git = None
    try:
        out = subprocess.run(["git", "-C", ROOT, "rev-parse", "HEAD"], capture_output=True,
                             text=True, timeout=10)
        git = out.stdout.strip() or None if out.returncode == 0 else None
    except (OSError, subprocess.TimeoutExpired):
        pass
    return {"gpu": props.name, "sm_count": props.multi_processor_count,
            "compute_capability": f"{props.major}.{props.minor}", "l2_bytes": l2,
            "hbm_bytes": int(props.total_memory), "driver": drv[0] if drv else None,
            "nvcc": nvcc, "cuda_runtime": torch.version.cuda, "torch": torch.__version__,
            "python": platform.python_version(), "host_arch": platform.machine(),
            "host_cores": os.cpu_count(), "git_head": git,
            "library_source_hash": libbuild.source_hash()}


# ------------------------------------------------------------ result files

class ResultsLog:
    """Per-run record: env.json and cells.jsonl (one JSON object a timed
    cell) in a directory, so that an interrupted run can be resumed without
    timing its finished cells again. Without a directory it records nothing."""

    def __init__(self, directory: str | None, resume: bool = False):
        self.dir = directory
        self.cells: dict[tuple[str, str], dict] = {}
        if directory is None:
            return
        os.makedirs(directory, exist_ok=True)
        path = os.path.join(directory, "cells.jsonl")
        if resume and os.path.exists(path):
            with open(path) as f:
                for line in f:
                    line = line.strip()
                    if not line:
                        continue
                    try:
                        rec = json.loads(line)
                    except ValueError:
                        continue  # a line cut off by the interruption
                    self.cells[(rec.get("kind", ""), rec.get("workload", ""))] = rec
        elif os.path.exists(path):
            os.remove(path)

    def done(self, kind: str, workload: str) -> dict | None:
        rec = self.cells.get((kind, workload))
        if rec is None:
            return None
        return {k: v for k, v in rec.items() if k != "kind"}

    def add(self, kind: str, cell: dict) -> None:
        if self.dir is None:
            return
        rec = {"kind": kind, **cell}
        self.cells[(kind, cell.get("workload", ""))] = rec
        with open(os.path.join(self.dir, "cells.jsonl"), "a") as f:
            f.write(json.dumps(rec) + "\n")

    def env(self, env: dict) -> None:
        if self.dir is None:
            return
        with open(os.path.join(self.dir, "env.json"), "w") as f:
            json.dump(env, f, indent=1)


# ------------------------------------------------------------ multi-rank

def slowest_rank(dist, values, device):
    """Elementwise maximum of `values` (floats) over all ranks; the values
    themselves when not distributed. Timing reports the slowest replica."""
    if dist is None:
        return [float(v) for v in values]
    import torch

    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def replica_throughput(world: int, logical_bytes_per_replica: int, step_ms: float) -> float:
    """Whole-job GB/s: every rank runs one replica of the workload (weak
    scaling), so the job moves world x the logical bytes per step, in the
    slowest rank's step time."""
    return world * logical_bytes_per_replica / (step_ms * 1e-3) / 1e9


# ------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi clock / throttle-reason sampler around the timed region."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu_index = gpu_index
        self.proc = None
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", smi_index(self.gpu_index)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def mark_start(self):
        self.t0 = time.time()

    def mark_end(self):
        self.t1 = time.time()

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = []
        for rec in csv.reader(io.StringIO(out)):
            if len(rec) < 10:
                continue
            rec = [r.strip() for r in rec]
            try:
                ts = time.mktime(time.strptime(rec[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                frac = float("0." + rec[0].split(".")[1]) if "." in rec[0] else 0.0
                rows.append({"t": ts + frac, "sm": float(rec[2]), "max": float(rec[3]),
                             "power": float(rec[4]) if rec[4] not in ("[N/A]", "N/A") else None,
                             "active": rec[5], "hw": rec[6], "hw_thermal": rec[7],
                             "sw_thermal": rec[8], "sw_power": rec[9]})
            except (ValueError, IndexError):
                continue
        if not rows:
            return None
        inside = [r for r in rows if self.t0 and self.t1 and self.t0 - 0.15 <= r["t"] <= self.t1 + 0.15]
        window = "timed_region"
        if len(inside) < 2:
            inside, window = rows, "whole_run"
        reasons = []
        for key, name in (("hw", "hw_slowdown"), ("hw_thermal", "hw_thermal_slowdown"),
                          ("sw_thermal", "sw_thermal_slowdown"), ("sw_power", "sw_power_cap")):
            if any(r[key].lower() == "active" for r in inside):
                reasons.append(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in inside),
                "sm_max_mhz": max(r["max"] for r in inside),
                "reasons": reasons, "samples": len(inside), "window": window,
                "power_w_max": max((r["power"] for r in inside if r["power"] is not None),
                                   default=None)}


# ------------------------------------------------------------ GPU helpers

def event_ms(a, b) -> float:
    return a.elapsed_time(b)


def by_set(xs, nsets: int) -> list:
    """Median time of the calls on each clone set (step k uses set k % nsets)."""
    return [round(statistics.median(xs[i::nsets]), 5) for i in range(nsets) if xs[i::nsets]]


def p90(xs) -> float:
    """90th percentile (nearest rank)."""
    ys = sorted(xs)
    return ys[min(len(ys) - 1, max(0, -(-9 * len(ys) // 10) - 1))]


def make_flush(torch, l2: int, device):
    """The clean-cold-L2 step run before every timed call: write a 2x L2
    buffer, then read another 2x L2 buffer, so the written dirty lines are
    written back here (outside the events) and the timed call starts from a
    clean, cold L2."""
    flush_w = torch.empty(2 * l2, dtype=torch.uint8, device=device)
    flush_r = torch.ones(2 * l2 // 4, dtype=torch.float32, device=device)
    flush_sink = torch.empty((), dtype=torch.float32, device=device)

    def flush():
        flush_w.zero_()
        torch.sum(flush_r, dim=0, out=flush_sink)

    return flush


def run_cold_copy(pkg, torch, nbytes: int, l2: int, samples: int = 20):
    """The copy probe under the cells' protocol: the clean-cold-L2 flush
    before each sample, CUDA events around the copy alone. Copying nbytes
    moves what a forward over an nbytes activation moves (read x, write y),
    and the copy's dirty output lines left in L2 at its end escape its
    events exactly as the cells' outputs do, so this is the like-for-like
    denominator of the cold-cell fractions."""
    dev = torch.cuda.current_device()
    a = torch.ones(nbytes // 4, dtype=torch.float32, device=dev)
    c = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    flush = make_flush(torch, l2, dev)
    stream = torch.cuda.current_stream()
    for _ in range(3):
        flush()
        pkg.check(pkg.rmsnorm_probe(pkg.PROBE_COPY, c, a, None, nbytes, 4, stream), "probe")
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(samples)]
    for e0, e1 in ev:
        flush()
        e0.record(stream)
        pkg.check(pkg.rmsnorm_probe(pkg.PROBE_COPY, c, a, None, nbytes, 4, stream), "probe")
        e1.record(stream)
    torch.cuda.synchronize()
    gbs = [2 * nbytes / (event_ms(e0, e1) * 1e-3) / 1e9 for e0, e1 in ev]
    del a, c
    torch.cuda.empty_cache()
    return {"bytes": nbytes, "moved_bytes": 2 * nbytes, "samples": samples,
            "median_gbs": round(statistics.median(gbs), 1), "best_gbs": round(max(gbs), 1),
            "protocol": "clean cold L2 before each sample, events around the copy only"}


def run_probes(pkg, torch, nbytes: int, samples: int = 10):
    """Best-of GB/s for copy, pure write and 2R1W over nbytes-sized buffers,
    timed back to back (steady state: each sample pays the write-back of the
    one before)."""
    dev = torch.cuda.current_device()
    a = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    b = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    c = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    a.fill_(1)
    b.fill_(2)
    res = {}
    moved = {pkg.PROBE_COPY: 2 * nbytes, pkg.PROBE_WRITE: nbytes, pkg.PROBE_2R1W: 3 * nbytes}
    names = {pkg.PROBE_COPY: "copy", pkg.PROBE_WRITE: "write", pkg.PROBE_2R1W: "2r1w"}
    for kind in (pkg.PROBE_COPY, pkg.PROBE_WRITE, pkg.PROBE_2R1W):
        best = 0.0
        for bps in (2, 4):
            for _ in range(2):
                pkg.check(pkg.rmsnorm_probe(kind, c, a, b, nbytes, bps), "probe")
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            for _ in range(samples):
                e0.record()
                pkg.check(pkg.rmsnorm_probe(kind, c, a, b, nbytes, bps), "probe")
                e1.record()
                e1.synchronize()
                best = max(best, moved[kind] / (event_ms(e0, e1) * 1e-3) / 1e9)
        res[names[kind]] = round(best, 1)
    del a, b, c
    torch.cuda.empty_cache()
    res["best"] = max(res.values())
    res["bytes"] = nbytes
    res["samples"] = samples
    return res


def validate(torch, x, w, dy, eps, y, rstd, dx, dw, dres=None, dw_tol=1e-3):
    """Compare against a float32 PyTorch reference on the GPU (the check
    happens before timing; the tests' rule for each dtype, with the fp32
    margins widened tenfold for a reference that is itself fp32)."""
    import torch.nn.functional as F

    N = x.shape[-1]
    x32 = x.float().requires_grad_(True)
    w32 = w.float().requires_grad_(True)
    y32 = F.rms_norm(x32, (N,), w32, eps)
    y32.backward(dy.float())
    errs = {}
    dx_ref = x32.grad if dres is None else x32.grad + dres.float()
    for name, got, ref in (("y", y, y32.detach()), ("dx", dx, dx_ref)):
        err = (got.float() - ref).abs()
        if x.dtype == torch.bfloat16:
            bad = (err > 1e-2 * ref.abs() + 1e-3).sum().item()
        elif x.dtype == torch.float16:
            rms = ref.pow(2).mean(-1, keepdim=True).sqrt()
            bad = (err > 2.0 ** -10 * ref.abs() + 1e-4 * rms + 2.0 ** -24).sum().item()
        else:
            rms = ref.pow(2).mean(-1, keepdim=True).sqrt()
            bad = (err > 1e-4 * ref.abs() + 1e-4 * rms).sum().item()
        errs[name] = {"max_abs_err": float(err.max().item()), "bad": int(bad)}
    r_ref = torch.rsqrt(x.float().pow(2).mean(-1) + eps)
    errs["rstd"] = {"max_rel_err": float(((rstd - r_ref).abs() / r_ref).max().item())}
    dwr = w32.grad
    errs["dw"] = {"rel_l2": float(((dw - dwr).norm() / dwr.norm()).item())}
    ok = errs["y"]["bad"] == 0 and errs["dx"]["bad"] == 0 and errs["rstd"]["max_rel_err"] < 1e-4 \
        and errs["dw"]["rel_l2"] < dw_tol
    return ok, errs


# ------------------------------------------------------------- CPU baseline

def cpu_baseline(wl, budget_s: float):
    """Times the fp64 CPU oracle, as it stands (single thread), on the
    workload's own rows: all of them when one pass fits the budget (then
    repeated until the budget is used), else the first rows that fit."""
    import torch

    import oracle  # the one place bench.py's own arm uses the oracle
    from memory_bound_normalization_gb300 import synth

    oracle.build()
    elem = torch.empty(0, dtype=wl.dtype).element_size()
    w_elem = torch.empty(0, dtype=wl.weight_dtype).element_size()
    probe_rows = min(wl.M, 64)
    inp = synth.make_inputs(wl, device="cpu", M=probe_rows)

    def one(x, w, dy):
        t0 = time.perf_counter()
        oracle.fwd(x, w, wl.eps)
        oracle.bwd_dx(x, w, dy, wl.eps)
        oracle.bwd_dw(x, dy, wl.eps)
        return time.perf_counter() - t0

    per_row = one(inp["x"], inp["w"], inp["dy"]) / probe_rows
    rows = int(max(1, min(wl.M, budget_s / max(per_row, 1e-12))))
    inp = synth.make_inputs(wl, device="cpu", M=rows)
    passes, total = 0, 0.0
    while True:
        total += one(inp["x"], inp["w"], inp["dy"])
        passes += 1
        if total >= budget_s or passes >= 64:
            break
    fb, bb = synth.logical_bytes(rows, wl.N, elem, w_elem)
    what = "all" if rows == wl.M else f"the first {rows} of"
    out = {"value": round(passes * (fb + bb) / total / 1e9, 4), "unit": "GB/s", "cores": 1,
           "kind": "oracle",
           "sample": f"{what} {wl.M} rows x {wl.N} ({wl.dtype_name}), fwd + dx + dw in fp64 on "
                     f"one host thread, {passes} pass(es), {total:.1f} s"}
    cores = os.cpu_count() or 1
    if cores > 1:
        out["all_cores"] = cpu_baseline_all_cores(oracle, synth, wl, rows, cores, budget_s,
                                                  elem, w_elem)
    return out


def cpu_baseline_all_cores(oracle, synth, wl, rows_one, cores, budget_s, elem, w_elem):
    """The same oracle calls on every host core: the rows are cut into one
    contiguous shard per thread (the oracle's C entry points run without the
    interpreter lock), each thread computes its shard's y, dx and partial dw,
    and the partial dw are added in shard order. The sample is about what one
    thread did alone, times the number of threads, up to all rows."""
    from concurrent.futures import ThreadPoolExecutor

    rows = int(min(wl.M, max(cores, rows_one * cores)))
    inp = synth.make_inputs(wl, device="cpu", M=rows)
    x, w, dy = inp["x"], inp["w"], inp["dy"]
    cuts = [rows * k // cores for k in range(cores + 1)]

    def shard(k):
        a, b = cuts[k], cuts[k + 1]
        if a == b:
            return None
        oracle.fwd(x[a:b], w, wl.eps)
        oracle.bwd_dx(x[a:b], w, dy[a:b], wl.eps)
        return oracle.bwd_dw(x[a:b], dy[a:b], wl.eps)

    passes, total = 0, 0.0
    with ThreadPoolExecutor(max_workers=cores) as pool:
        while True:
            t0 = time.perf_counter()
            dw = None
            for part in pool.map(shard, range(cores)):
                if part is not None:
                    dw = part if dw is None else dw + part
            total += time.perf_counter() - t0
            passes += 1
            if total >= budget_s or passes >= 64:
                break
    fb, bb = synth.logical_bytes(rows, wl.N, elem, w_elem)
    what = "all" if rows == wl.M else f"the first {rows} of"
    return {"value": round(passes * (fb + bb) / total / 1e9, 4), "unit": "GB/s", "cores": cores,
            "sample": f"{what} {wl.M} rows in {cores} row shards, one thread each; "
                      f"{passes} pass(es), {total:.1f} s"}


def pick_workload(synth, args):
    """--shape M,N,dtype (x, dy ~ N(0,1), w = 1 + 0.1 N(0,1), eps 1e-5, fixed
    seeds), else the named workload."""
    if not args.shape:
        return synth.WORKLOADS[args.workload]
    import torch

    m, n, dt = args.shape.split(",")
    act, _, wt = dt.partition("_w")  # e.g. bf16_wf32: bf16 activations, fp32 weight
    types = {"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32}
    return synth.Workload(f"shape_{m}x{n}_{dt}", int(m), int(n), types[act], 1e-5, 51, 52, 53,
                          about="ad-hoc shape", w_dtype=types[wt] if wt else None)


# ------------------------------------------------------------------ our arm

def time_cell(pkg, torch, synth, wl, op, code, steps, warmup, local, l2, check_first=True,
              sample_clocks=False, dist=None, steady_steps=0):
    """Validates (unless check_first is False) and times `steps` forward +
    backward calls of one workload: inputs rotated over clone sets covering
    >= 3x L2, a clean cold L2 before every call, CUDA events on the calling
    stream around each call; the backward is re-run once at the end and must
    give the same dw bits."""
    M, N, eps = wl.M, wl.N, wl.eps
    residual = op == "residual"
    naive = op == "naive"
    elem = torch.empty(0, dtype=wl.dtype).element_size()
    # inputs, rotated over clone sets covering >= 3x L2
    base = synth.make_inputs(wl, device=f"cuda:{local}")
    if residual:
        more = synth.make_inputs(dataclasses.replace(wl, seed_x=wl.seed_x + 1000,
                                                     seed_dy=wl.seed_dy + 1000),
                                 device=f"cuda:{local}")
        base["res"], base["dres"] = more["x"], more["dy"]
    set_bytes = sum(v.numel() for k, v in base.items() if k != "w") * elem
    nsets = max(2, -(-3 * l2 // set_bytes))
    sets = [base] + [{k: v.clone() for k, v in base.items()} for _ in range(nsets - 1)]
    outs = []
    for _ in range(nsets):
        outs.append({"y": torch.empty_like(base["x"]), "dx": torch.empty_like(base["x"]),
                     "h": torch.empty_like(base["x"]) if residual else None,
                     "rstd": torch.empty(M, dtype=torch.float32, device=base["x"].device),
                     "dw": torch.empty(N, dtype=torch.float32, device=base["x"].device)})
    # L2 flush between timed calls (outside the events)
    flush = make_flush(torch, l2, base["x"].device)

    stream = torch.cuda.current_stream()

    def fwd(i):
        s, o = sets[i], outs[i]
        if residual:
            return pkg.rmsnorm_add_fwd(s["x"], s["res"], s["w"], o["h"], o["y"], o["rstd"], M, N,
                                       eps, code, stream)
        return pkg.rmsnorm_fwd(s["x"], s["w"], o["y"], o["rstd"], M, N, eps, code, stream)

    def bwd(i):
        s, o = sets[i], outs[i]
        if residual:
            return pkg.rmsnorm_add_bwd(o["h"], s["w"], s["dy"], o["rstd"], s["dres"], o["dx"],
                                       o["dw"], M, N, code, stream)
        if naive:
            return pkg.rmsnorm_bwd_naive(s["x"], s["w"], s["dy"], o["dx"], o["dw"], M, N, eps,
                                         code, stream)
        return pkg.rmsnorm_bwd(s["x"], s["w"], s["dy"], o["rstd"], o["dx"], o["dw"], M, N, code,
                               stream)

    # validate every clone set before timing
    errs = None
    if check_first:
        for i in range(nsets):
            pkg.check(fwd(i), "rmsnorm_fwd")
            pkg.check(bwd(i), "rmsnorm_bwd")
        st = pkg.rmsnorm_get_last_device_error(stream)
        pkg.check(st, "device status")
        for i in range(nsets):
            xin = sets[i]["x"]
            if residual:
                h_ref = sets[i]["x"] + sets[i]["res"]  # added in the activation type
                if not torch.equal(outs[i]["h"], h_ref):
                    raise SystemExit("validation failed before timing: h != x + residual")
                xin = h_ref
            ok, errs_i = validate(torch, xin, sets[i]["w"], sets[i]["dy"], eps,
                                  outs[i]["y"], outs[i]["rstd"], outs[i]["dx"], outs[i]["dw"],
                                  sets[i]["dres"] if residual else None,
                                  # the naive chain rounds every dw term to the
                                  # activation type (about 1e-3 relative in bf16)
                                  dw_tol=5e-3 if naive else 1e-3)
            if not ok:
                raise SystemExit(f"validation failed before timing: {json.dumps(errs_i)}")
            errs = errs if errs is not None else errs_i
    dw0 = None

    for k in range(warmup):
        i = k % nsets
        flush()
        pkg.check(fwd(i))
        flush()
        pkg.check(bwd(i))
    torch.cuda.synchronize()

    K = steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(K)]
    region0, region1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local) if sample_clocks else None
    if clocks is not None:
        clocks.start()
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    if clocks is not None:
        clocks.mark_start()
    region0.record(stream)
    for k in range(K):
        i = k % nsets
        e = ev[k]
        flush()
        e[0].record(stream)
        fwd(i)
        e[1].record(stream)
        flush()
        e[2].record(stream)
        bwd(i)
        e[3].record(stream)
    region1.record(stream)
    torch.cuda.synchronize()
    if clocks is not None:
        clocks.mark_end()
    if dist is not None:
        dist.barrier()
    clock_info = clocks.stop() if clocks is not None else None
    st = pkg.rmsnorm_get_last_device_error(stream)
    pkg.check(st, "device status after timing")
    if dw0 is None:
        dw0 = outs[0]["dw"].clone()
        pkg.check(bwd(0))
        torch.cuda.synchronize()
    if not torch.equal(outs[0]["dw"], dw0):
        raise SystemExit("dw changed between identical backward calls")

    fwd_ms = [event_ms(e[0], e[1]) for e in ev]
    bwd_ms = [event_ms(e[2], e[3]) for e in ev]
    # throughput is total bytes over total time: the means; the median, the
    # minimum and the 90th percentile are reported beside them
    fwd_mean = sum(fwd_ms) / K
    bwd_mean = sum(bwd_ms) / K
    step_ms = fwd_mean + bwd_mean
    region_ms = event_ms(region0, region1)
    steady = None
    if steady_steps > 0:
        steady = time_steady(torch, fwd, bwd, nsets, steady_steps, stream)
        if not torch.equal(outs[0]["dw"], dw0):
            raise SystemExit("dw changed between the cold and the steady-state calls")
    return {"fwd_ms": fwd_ms, "bwd_ms": bwd_ms, "fwd_mean": fwd_mean, "bwd_mean": bwd_mean,
            "step_ms": step_ms, "region_ms": region_ms, "nsets": nsets, "set_bytes": set_bytes,
            "errs": errs, "base": base, "clock_info": clock_info, "dw0": outs[0]["dw"],
            "steady": steady}


def time_steady(torch, fwd, bwd, nsets: int, steps: int, stream):
    """Steady state, as inside a training step: forward and backward calls
    back to back over the rotating clone sets (>= 3x L2 of inputs, so no
    call finds its inputs in L2), with no flush, so every call also pays for
    writing back the outputs the call before left dirty in L2. One event pair
    brackets all `steps` steps; a second pass records events between the
    calls for the forward / backward split."""
    for k in range(2 * nsets):
        fwd(k % nsets)
        bwd(k % nsets)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for k in range(steps):
        fwd(k % nsets)
        bwd(k % nsets)
    e1.record(stream)
    torch.cuda.synchronize()
    step_ms = event_ms(e0, e1) / steps
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2 * steps + 1)]
    ev[0].record(stream)
    for k in range(steps):
        fwd(k % nsets)
        ev[2 * k + 1].record(stream)
        bwd(k % nsets)
        ev[2 * k + 2].record(stream)
    torch.cuda.synchronize()
    f = [event_ms(ev[2 * k], ev[2 * k + 1]) for k in range(steps)]
    b = [event_ms(ev[2 * k + 1], ev[2 * k + 2]) for k in range(steps)]
    return {"steps": steps, "step_ms": step_ms, "fwd_ms": sum(f) / steps, "bwd_ms": sum(b) / steps}


def run_ours(args):
    import torch

    import memory_bound_normalization_gb300 as pkg
    from memory_bound_normalization_gb300 import build as libbuild
    from memory_bound_normalization_gb300 import synth

    rank, world, local = dist_env()
    # before this process touches the GPU: is anyone else using it?
    idle = idle_gate(local)
    if idle.get("busy") and args.require_idle:
        raise SystemExit(f"GPU {smi_index(local)} is busy before the first launch: {json.dumps(idle)}")
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")

    pkg.load_library()  # raises if librmsnorm.so is missing
    wl = pick_workload(synth, args)
    M, N, eps = wl.M, wl.N, wl.eps
    residual = args.op == "residual"
    naive = args.op == "naive"
    code = pkg.dtype_code(wl.dtype, wl.weight_dtype)
    elem = torch.empty(0, dtype=wl.dtype).element_size()
    w_elem = torch.empty(0, dtype=wl.weight_dtype).element_size()
    fwd_bytes, bwd_bytes = synth.logical_bytes(M, N, elem, w_elem)
    if residual:
        # the residual is read and h written in the forward; dres is read in
        # the backward
        fwd_bytes += 2 * M * N * elem
        bwd_bytes += M * N * elem
    props = torch.cuda.get_device_properties(local)
    l2 = int(getattr(props, "L2_cache_size", 126 * 2 ** 20))

    peak, peak_src = read_peaks()
    probe_bytes = int(args.probe_gib * (1 << 30)) // 16 * 16
    probes_open = None if args.profile else run_probes(pkg, torch, probe_bytes,
                                                       args.probe_samples)

    cell = time_cell(pkg, torch, synth, wl, args.op, code, args.steps, args.warmup, local, l2,
                     check_first=not args.profile, sample_clocks=True, dist=dist,
                     steady_steps=0 if args.profile else args.steady_steps)
    fwd_ms, bwd_ms = cell["fwd_ms"], cell["bwd_ms"]
    fwd_mean, bwd_mean, step_ms = cell["fwd_mean"], cell["bwd_mean"], cell["step_ms"]
    region_ms, nsets, set_bytes = cell["region_ms"], cell["nsets"], cell["set_bytes"]
    errs, base, clock_info = cell["errs"], cell["base"], cell["clock_info"]
    K = args.steps
    stream = torch.cuda.current_stream()
    step_ms, fwd_mean, bwd_mean = slowest_rank(dist, [step_ms, fwd_mean, bwd_mean],
                                               base["x"].device)

    if args.profile:
        line = {"profile": True, "workload": wl.name, "fwd_ms": round(fwd_mean, 5),
                "bwd_ms": round(bwd_mean, 5), "steps": K}
        if dist is not None:
            dist.destroy_process_group()
        return line if rank == 0 else None
    # end to end through pinned host buffers
    e2e = run_e2e(pkg, torch, wl, base, code, stream, args.e2e_steps, fwd_bytes + bwd_bytes,
                  args.op, ref_dw=cell["dw0"])
    if dist is not None:
        e2e["step_ms"] = slowest_rank(dist, [e2e["step_ms"]], base["x"].device)[0]
        e2e["value"] = round(replica_throughput(world, fwd_bytes + bwd_bytes, e2e["step_ms"]), 2)

    small_m = None if args.no_small_m else run_small_m(pkg, torch)
    plan_f = pkg.rmsnorm_plan(M, N, code, pkg.PASS_FWD_ADD if residual else pkg.PASS_FWD,
                              local).as_dict()
    plan_b = pkg.rmsnorm_plan(M, N, code, pkg.PASS_BWD_RES if residual else pkg.PASS_BWD,
                              local).as_dict()
    value = replica_throughput(world, fwd_bytes + bwd_bytes, step_ms)
    bwd_gbs = bwd_bytes / (bwd_mean * 1e-3) / 1e9
    fwd_gbs = fwd_bytes / (fwd_mean * 1e-3) / 1e9
    # the copy probe under the cells' own protocol, sized to move what the
    # forward and the backward call move
    cold = {"fwd_sized": run_cold_copy(pkg, torch, fwd_bytes // 32 * 16, l2),
            "bwd_sized": run_cold_copy(pkg, torch, bwd_bytes // 32 * 16, l2)}
    steady = None
    if cell["steady"] is not None:
        sd = cell["steady"]
        sd_ms = slowest_rank(dist, [sd["step_ms"]], base["x"].device)[0]
        sd_gbs = replica_throughput(world, fwd_bytes + bwd_bytes, sd_ms)
        sf = fwd_bytes / (sd["fwd_ms"] * 1e-3) / 1e9
        sb = bwd_bytes / (sd["bwd_ms"] * 1e-3) / 1e9
        steady = {
            "steps": sd["steps"], "ms_per_step": round(sd_ms, 5), "gbs": round(sd_gbs, 1),
            "frac": round(sd_gbs / world / peak, 4),
            "frac_of_probe": round(sd_gbs / world / probes_open["best"], 4),
            "fwd_gbs": round(sf, 1), "fwd_frac": round(sf / peak, 4),
            "bwd_gbs": round(sb, 1), "bwd_frac": round(sb / peak, 4),
            "protocol": "forward + backward calls back to back over the rotating clone sets, "
                        "no flush: each call pays the write-back of the outputs the call "
                        "before left dirty in L2; one event pair around all steps (the "
                        "fwd/bwd split from a second pass with events between the calls); "
                        "frac of MEASURED_PEAKS, frac_of_probe of the in-run probes, which "
                        "run back to back as well"}
    traffic = read_profiled_traffic("rmsnorm_add_bwd" if residual else "rmsnorm_bwd", wl.name,
                                    libbuild.kernel_source_hash())
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": round(step_ms, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": wl.dtype_name,
        "data": "synthetic",
        "config": {
            "workload": wl.name,
            "op": {"norm": "rmsnorm", "residual": "residual add + rmsnorm",
                   "naive": "rmsnorm, naive three-kernel backward (ablation)"}[args.op],
            "M": M, "N": N, "eps": eps, "io_dtype": wl.dtype_name,
            "accumulate": "f32", "rstd_dw_dtype": "f32", "about": wl.about,
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
            "l2": f"inputs rotated over {nsets} clone sets ({nsets * set_bytes >> 20} MiB, "
                  f">= 3x L2 of {l2 >> 20} MiB); before every timed call, outside the events, "
                  f"a {2 * l2 >> 20} MiB write then a {2 * l2 >> 20} MiB read (cold, clean L2)",
            "logical_bytes": {"fwd": fwd_bytes, "bwd": bwd_bytes},
        },
        "fwd": {"ms": round(fwd_mean, 5), "median_ms": round(statistics.median(fwd_ms), 5),
                "min_ms": round(min(fwd_ms), 5), "p90_ms": round(p90(fwd_ms), 5),
                "median_ms_by_clone_set": by_set(fwd_ms, nsets),
                "gbs": round(fwd_gbs, 1),
                "frac_of_peak": round(fwd_gbs / peak, 4),
                "frac_of_probe": round(fwd_gbs / probes_open["best"], 4),
                "frac_of_cold_copy": round(fwd_gbs / cold["fwd_sized"]["median_gbs"], 4),
                "plan": plan_f},
        "bwd": {"ms": round(bwd_mean, 5), "median_ms": round(statistics.median(bwd_ms), 5),
                "min_ms": round(min(bwd_ms), 5), "p90_ms": round(p90(bwd_ms), 5),
                "median_ms_by_clone_set": by_set(bwd_ms, nsets),
                "gbs": round(bwd_gbs, 1),
                "frac_of_peak": round(bwd_gbs / peak, 4),
                "frac_of_probe": round(bwd_gbs / probes_open["best"], 4),
                "frac_of_cold_copy": round(bwd_gbs / cold["bwd_sized"]["median_gbs"], 4),
                "plan": plan_b,
                "workspace_bytes_overhead": 2 * plan_b["workspace_bytes"]},
        "steady": steady,
        "cold_copy": cold,
        "frac_of_peak": round(value / world / peak, 4),
        "roofline": {
            "bound": "hbm",
            "kernel": "rmsnorm_bwd_naive (row kernel + two column sums, one call)" if naive
            else ("rmsnorm_add_bwd" if residual else "rmsnorm_bwd")
            + " (persistent kernel + fixed-order column sum, one call)",
            "achieved": round(bwd_gbs, 1),
            "peak": peak,
            "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)" if peak_src == "measured"
            else "fallback 6800 GB/s",
            "unit": "GB/s",
            "frac": round(bwd_gbs / peak, 4),
            "traffic": traffic,
        },
        "timed_region_ms": round(region_ms, 3),
        "clocks": clock_info,
        "e2e": e2e,
        "small_m": small_m,
        # ours only: fwd, main bwd and its column sum (none with one partial row);
        # the naive chain is three kernels behind the forward
        "gpu_launches": (4 if naive else 2 + (plan_b["partial_rows"] > 1)) * K,
        "validation": errs,
        "library": {"path": pkg.library_path(), "source_hash": libbuild.source_hash(),
                    "bwd_kernel_hash": libbuild.kernel_source_hash(),
                    "version": pkg.rmsnorm_version()},
        "idle_gate": idle,
        "env": env_record(torch, local, l2),
    }
    log = ResultsLog(args.results_dir if rank == 0 else None, args.resume)
    log.env(line["env"])
    log.add("main", {"workload": wl.name, "op": args.op, "fwd_frac": line["fwd"]["frac_of_peak"],
                     "bwd_frac": line["bwd"]["frac_of_peak"], "value": line["value"],
                     "steady_frac": steady["frac"] if steady else None})
    if world == 1 and args.op == "norm" and not args.no_sweep:
        line["sweep"] = run_sweep(pkg, torch, synth, args, local, l2, peak, log)
    if world == 1 and args.op == "norm" and not args.no_configs:
        line["configs"] = run_configs(pkg, torch, synth, args, local, l2, peak,
                                      skip=wl.name, log=log)
    # the closing probe comes after every timed cell, so a drift across the
    # whole run shows ("What a tuned RMSNorm kernel actually costs on Hopper",
    # sections 02 and 08: opening and closing probes)
    probes_close = run_probes(pkg, torch, probe_bytes, args.probe_samples)
    ratio = probes_close["best"] / probes_open["best"]
    line["probes"] = {"open": probes_open, "close": probes_close,
                      "close_over_open": round(ratio, 4), "drift_flag": ratio < DRIFT_LIMIT,
                      "drift_limit": DRIFT_LIMIT,
                      "note": "closing probe taken after the main cell, the sweep and the "
                              "other workloads"}
    if rank == 0 and not args.no_cpu_baseline and args.op == "norm":
        line["cpu_baseline"] = cpu_baseline(wl, args.cpu_seconds)
    if dist is not None:
        dist.destroy_process_group()
    return line if rank == 0 else None


def steady_fields(cell, step_bytes: int, peak: float) -> dict:
    """The steady-state step of a cell (back to back, no flush) as GB/s and
    a fraction of the measured copy bandwidth; empty when not timed."""
    sd = cell.get("steady")
    if not sd:
        return {}
    gbs = step_bytes / (sd["step_ms"] * 1e-3) / 1e9
    return {"steady_gbs": round(gbs, 1), "steady_frac": round(gbs / peak, 4)}


def run_sweep(pkg, torch, synth, args, local, l2, peak, log=None):
    """The width sweep (fixed M*N = 2^27, bf16 and fp32): each cell validated
    against PyTorch, then forward and backward timed after a clean cold L2,
    as for the main workload. Fractions are of the measured copy bandwidth.
    Cells `log` already holds (a resumed run) are taken from it."""
    log = log or ResultsLog(None)
    cells = []
    for dt in (torch.bfloat16, torch.float32):
        for wl in synth.width_sweep(dt):
            prev = log.done("sweep", wl.name)
            if prev is not None:
                cells.append({**prev, "resumed": True})
                continue
            code = pkg.dtype_code(wl.dtype, wl.weight_dtype)
            elem = torch.empty(0, dtype=wl.dtype).element_size()
            fb, bb = synth.logical_bytes(wl.M, wl.N, elem)
            c = time_cell(pkg, torch, synth, wl, "norm", code, args.sweep_steps, 3, local, l2,
                          steady_steps=min(args.steady_steps, 100))
            fg = fb / (c["fwd_mean"] * 1e-3) / 1e9
            bg = bb / (c["bwd_mean"] * 1e-3) / 1e9
            cells.append({"workload": wl.name, "dtype": wl.dtype_name, "M": wl.M, "N": wl.N,
                          "fwd_gbs": round(fg, 1), "bwd_gbs": round(bg, 1),
                          "fwd_frac": round(fg / peak, 4), "bwd_frac": round(bg / peak, 4),
                          "fwd_bwd_gbs": round((fb + bb) / (c["step_ms"] * 1e-3) / 1e9, 1),
                          **steady_fields(c, fb + bb, peak)})
            log.add("sweep", cells[-1])
            del c
    return {"steps": args.sweep_steps, "peak_gbs": peak, "cells": cells}


CONFIG_WORKLOADS = ("small_256x1024", "hidden8192_32768x8192_outliers", "qknorm_1048576x128")


def run_configs(pkg, torch, synth, args, local, l2, peak, skip=None, log=None):
    """The other named workloads (256 x 1024, which fits in L2 and is bound
    by latency; 32768 x 8192 with 0.1% outliers; QK-norm 1048576 x 128),
    each validated against PyTorch and timed like the main workload: clone
    sets >= 3x L2, a clean cold L2 before every call, events per call.
    Cells `log` already holds (a resumed run) are taken from it."""
    log = log or ResultsLog(None)
    cells = []
    for name in CONFIG_WORKLOADS:
        if name == skip:
            continue
        prev = log.done("config", name)
        if prev is not None:
            cells.append({**prev, "resumed": True})
            continue
        wl = synth.WORKLOADS[name]
        code = pkg.dtype_code(wl.dtype, wl.weight_dtype)
        elem = torch.empty(0, dtype=wl.dtype).element_size()
        fb, bb = synth.logical_bytes(wl.M, wl.N, elem)
        c = time_cell(pkg, torch, synth, wl, "norm", code, args.config_steps, 5, local, l2,
                      steady_steps=min(args.steady_steps, 100))
        fg = fb / (c["fwd_mean"] * 1e-3) / 1e9
        bg = bb / (c["bwd_mean"] * 1e-3) / 1e9
        plan_b = pkg.rmsnorm_plan(wl.M, wl.N, code, pkg.PASS_BWD, local).as_dict()
        cells.append({"workload": wl.name, "dtype": wl.dtype_name, "M": wl.M, "N": wl.N,
                      "fwd_us": round(c["fwd_mean"] * 1e3, 2),
                      "bwd_us": round(c["bwd_mean"] * 1e3, 2),
                      "fwd_gbs": round(fg, 1), "bwd_gbs": round(bg, 1),
                      "fwd_frac": round(fg / peak, 4), "bwd_frac": round(bg / peak, 4),
                      "fwd_bwd_gbs": round((fb + bb) / (c["step_ms"] * 1e-3) / 1e9, 1),
                      "bwd_variant": plan_b["variant_name"],
                      **steady_fields(c, fb + bb, peak),
                      "validation": c["errs"]})
        log.add("config", cells[-1])
        del c
    return {"steps": args.config_steps, "peak_gbs": peak, "cells": cells}


def run_small_m(pkg, torch, steps: int = 200, per_graph: int = 20):
    """Launch-bound shapes: microseconds per forward+backward step, back to
    back (inputs stay in L2 here; this measures latency, not HBM): called
    eagerly through the C ABI, replayed as a captured CUDA graph of one step,
    and replayed as a graph of `per_graph` steps. The first two pay the
    host's cost of a call or a replay every step, which for these shapes is
    about as long as the device's work; the last shows the device's time."""
    from memory_bound_normalization_gb300 import synth

    out = []
    for M, N in ((1, 4096), (16, 4096), (256, 4096), (256, 1024)):
        wl = synth.Workload(f"small{M}x{N}", M, N, torch.bfloat16, 1e-6, 71, 72, 73)
        inp = synth.make_inputs(wl, device=torch.cuda.current_device())
        x, w, dy = inp["x"], inp["w"], inp["dy"]
        y, dx = torch.empty_like(x), torch.empty_like(x)
        rstd = torch.empty(M, dtype=torch.float32, device=x.device)
        dw = torch.empty(N, dtype=torch.float32, device=x.device)
        side = torch.cuda.Stream()

        def step():
            pkg.check(pkg.rmsnorm_fwd(x, w, y, rstd, M, N, wl.eps, pkg.BF16, side))
            pkg.check(pkg.rmsnorm_bwd(x, w, dy, rstd, dx, dw, M, N, pkg.BF16, side))

        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            for _ in range(10):
                step()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(side)
            for _ in range(steps):
                step()
            e1.record(side)
        e1.synchronize()
        eager_us = event_ms(e0, e1) * 1e3 / steps
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=side):
            step()
        with torch.cuda.stream(side):
            for _ in range(10):
                graph.replay()
            e0.record(side)
            for _ in range(steps):
                graph.replay()
            e1.record(side)
        e1.synchronize()
        graph_us = event_ms(e0, e1) * 1e3 / steps
        many = torch.cuda.CUDAGraph()
        with torch.cuda.graph(many, stream=side):
            for _ in range(per_graph):
                step()
        reps = max(1, steps // per_graph)
        with torch.cuda.stream(side):
            for _ in range(3):
                many.replay()
            e0.record(side)
            for _ in range(reps):
                many.replay()
            e1.record(side)
        e1.synchronize()
        many_us = event_ms(e0, e1) * 1e3 / (reps * per_graph)
        torch.cuda.current_stream().wait_stream(side)
        out.append({"M": M, "N": N, "eager_us_per_step": round(eager_us, 2),
                    "graph_us_per_step": round(graph_us, 2),
                    f"graph_of_{per_graph}_steps_us_per_step": round(many_us, 2)})
    return out


def run_e2e(pkg, torch, wl, base, code, stream, steps, logical, op="norm", ref_dw=None):
    """Same work through the C ABI with the inputs in pinned host memory:
    every step copies x, w, dy (and the residual and dres) to the device,
    runs forward and backward, and copies y, rstd, dx, dw (and h) back.
    Steps are independent batches, so they are pipelined over two device
    buffer slots: the inputs of a step go in on one copy stream while the
    previous step's results come out on another and the GPU computes in
    between, using both directions of the host link at once. The timed
    region runs from the first input copy to the last result copy."""
    M, N, eps = wl.M, wl.N, wl.eps
    residual = op == "residual"
    names = ["x", "w", "dy"] + (["res", "dres"] if residual else [])
    outn = ["y", "rstd", "dx", "dw"] + (["h"] if residual else [])
    host = {k: base[k].cpu().pin_memory() for k in names}
    dev_in = [{k: torch.empty_like(base[k]) for k in names} for _ in range(2)]
    x0 = base["x"]

    def outs():
        o = {"y": torch.empty_like(x0), "dx": torch.empty_like(x0),
             "rstd": torch.empty(M, dtype=torch.float32, device=x0.device),
             "dw": torch.empty(N, dtype=torch.float32, device=x0.device)}
        if residual:
            o["h"] = torch.empty_like(x0)
        return o

    dev_out = [outs(), outs()]
    host_out = {k: torch.empty(v.shape, dtype=v.dtype).pin_memory() for k, v in dev_out[0].items()}
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    in_done = [torch.cuda.Event() for _ in range(2)]
    cmp_done = [torch.cuda.Event() for _ in range(2)]
    out_done = [torch.cuda.Event() for _ in range(2)]

    def compute(d, o):
        if residual:
            pkg.check(pkg.rmsnorm_add_fwd(d["x"], d["res"], d["w"], o["h"], o["y"], o["rstd"], M,
                                          N, eps, code, stream))
            pkg.check(pkg.rmsnorm_add_bwd(o["h"], d["w"], d["dy"], o["rstd"], d["dres"], o["dx"],
                                          o["dw"], M, N, code, stream))
        elif op == "naive":
            pkg.check(pkg.rmsnorm_fwd(d["x"], d["w"], o["y"], o["rstd"], M, N, eps, code, stream))
            pkg.check(pkg.rmsnorm_bwd_naive(d["x"], d["w"], d["dy"], o["dx"], o["dw"], M, N, eps,
                                            code, stream))
        else:
            pkg.check(pkg.rmsnorm_fwd(d["x"], d["w"], o["y"], o["rstd"], M, N, eps, code, stream))
            pkg.check(pkg.rmsnorm_bwd(d["x"], d["w"], d["dy"], o["rstd"], o["dx"], o["dw"], M, N,
                                      code, stream))

    def step(k):
        b = k % 2
        s_in.wait_event(cmp_done[b])  # the compute that read this input slot is done
        with torch.cuda.stream(s_in):
            for n in names:
                dev_in[b][n].copy_(host[n], non_blocking=True)
        in_done[b].record(s_in)
        stream.wait_event(in_done[b])
        stream.wait_event(out_done[b])  # the copy-out of this output slot is done
        compute(dev_in[b], dev_out[b])
        cmp_done[b].record(stream)
        s_out.wait_event(cmp_done[b])
        with torch.cuda.stream(s_out):
            for n in outn:
                host_out[n].copy_(dev_out[b][n], non_blocking=True)
        out_done[b].record(s_out)

    for k in range(3):
        step(k)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    for k in range(steps):
        step(k)
    e1.record(s_out)  # every step's copy-out is ordered before it on s_out
    torch.cuda.synchronize()
    ms = event_ms(e0, e1) / steps
    if ref_dw is not None and not torch.equal(host_out["dw"], ref_dw.cpu()):
        raise SystemExit("end-to-end dw differs from the device-resident run on the same inputs")
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = sum(t.numel() * t.element_size() for t in host_out.values())
    return {"value": round(logical / (ms * 1e-3) / 1e9, 2), "unit": "GB/s",
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "step_ms": round(ms, 4), "steps": steps,
            "pipeline": "two buffer slots; copies in and out on their own streams"}


# ------------------------------------------------------------ reference arm

def run_reference(args):
    """The fp64 CPU oracle timed on the host cores, one bounded sample of rows
    per step, sized so that warm-up plus timed steps end within minutes."""
    rank, world, _ = dist_env()
    if rank != 0:
        return None
    import torch

    import oracle
    from memory_bound_normalization_gb300 import synth

    oracle.build()
    wl = pick_workload(synth, args)
    elem = torch.empty(0, dtype=wl.dtype).element_size()
    w_elem = torch.empty(0, dtype=wl.weight_dtype).element_size()
    rows_avail = min(wl.M, 2048)
    inp = synth.make_inputs(wl, device="cpu", M=rows_avail)
    x, w, dy = inp["x"], inp["w"], inp["dy"]

    def one(rows):
        t0 = time.perf_counter()
        oracle.fwd(x[:rows], w, wl.eps)
        oracle.bwd_dx(x[:rows], w, dy[:rows], wl.eps)
        oracle.bwd_dw(x[:rows], dy[:rows], wl.eps)
        return time.perf_counter() - t0

    t = one(4)
    per_row = t / 4
    total_budget = args.ref_seconds
    rows = int(max(1, min(rows_avail, total_budget / max(1, args.steps + args.warmup) / per_row)))
    for _ in range(args.warmup):
        one(rows)
    times = [one(rows) for _ in range(args.steps)]
    med = statistics.median(times)
    fb, bb = synth.logical_bytes(rows, wl.N, elem, w_elem)
    value = (fb + bb) / med / 1e9
    sample = (f"first {rows} of {wl.M} rows x {wl.N} ({wl.dtype_name}) per step; fp64 oracle "
              "fwd + dx + dw, single thread")
    return {
        "impl": "reference",
        "metric": METRIC,
        "value": round(value, 4),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(med * 1e3, 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": wl.dtype_name,
        "data": "synthetic",
        "config": {"workload": wl.name, "M": wl.M, "N": wl.N, "eps": wl.eps,
                   "sample_rows": rows},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main(argv=None):
    args = parse_args(argv)
    line = run_reference(args) if args.impl == "reference" else run_ours(args)
    if line is not None:
        s = json.dumps(line)
        print(s, flush=True)
        if args.json_out:
            with open(args.json_out, "w") as f:
                f.write(s + "\n")


if __name__ == "__main__":
    main()
