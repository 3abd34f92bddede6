#!/usr/bin/env python3
"""Benchmark of the Purlin copy/reduce datapath on GB300.

One step = one pass of the hot path over the headline workload: ReduceScatter
then AllGather over R=8 virtual ranks, bf16, 64 MiB per rank input (8
partitions of 8 MiB), N(0,1) values, binary32 accumulation in rank order.  The
inputs (512 MiB) are larger than L2, so no flush is needed between steps.

Prints ONE JSON line (rank 0).  ``value`` is effective GB/s: the algorithmic
bytes (read + written) of all ranks' steps divided by the max-over-ranks device
time.  Also reported: per-collective GB/s and roofline fraction, the AllReduce
latency at 4 KiB per rank, the end-to-end figure through host buffers, the CPU
oracle as a baseline, clocks sampled during the timed region.

``--impl reference`` times the CPU oracle instead (the reference arm: the
pages publish no code, so the oracle written from them stands in).
Under torchrun, every rank runs an independent replica on its own GPU
(the collective does not shard across GPUs).
"""
from __future__ import annotations

import argparse
import ctypes
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "effective HBM GB/s (% of GB300 peak) per collective @R=8; µs at 4 KiB/rank"
UNIT = "GB/s"
WORKLOAD = "rs_ag_r8_bf16"
WORKLOAD_SHORT = "RS+AG, R=8, bf16, 64 MiB/rank, N(0,1)"
R = 8
BYTES_PER_RANK = 64 << 20
ELEMS_PER_RANK = BYTES_PER_RANK // 2
PART = ELEMS_PER_RANK // R
FALLBACK_HBM_GBS = 6800.0


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["purlin", "reference"], default="purlin")
    ap.add_argument("--variant", choices=["zs", "staged", "staged_y"], default="zs")
    ap.add_argument("--chunk", type=int, default=0, help="SNAC chunk bytes (0 = auto)")
    ap.add_argument("--depth", type=int, default=0, help="SNAC ring depth (0 = auto)")
    ap.add_argument("--ctas", type=int, default=0, help="CTAs / channels (0 = auto)")
    ap.add_argument("--staging", type=int, default=0,
                    help="SNAC staging ring bytes of the handle (0 = library default)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--quick", action="store_true",
                    help="only the timed step, its split and the end-to-end figure "
                         "(no side studies, no CPU baseline)")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--studies-out", default=None,
                    help="write the side studies to this JSON file instead of an earlier "
                         "stdout line")
    ap.add_argument("--only", choices=["rs", "ag", "ar", "a2av"], default=None,
                    help="time one collective alone (profiling runs); prints a short line")
    ap.add_argument("--ranks", type=int, default=R, choices=range(1, R + 1), metavar="R",
                    help="virtual ranks of an --only run (1..8; default 8)")
    ap.add_argument("--bytes-per-rank", type=int, default=BYTES_PER_RANK,
                    help="with --only: input bytes per rank")
    ap.add_argument("--atom", choices=["auto", "vector", "bulk", "copy_engine"], default="auto",
                    help="with --only: copy Atom of the zero-staging path")
    ap.add_argument("--trim", type=int, default=0,
                    help="with --only: elements taken off every partition (rs, ag) or every "
                         "non-empty block (a2av), which puts partitions off the vector grid")
    return ap.parse_args()


# ---------------------------------------------------------------- environment

def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def bench_config(world):
    """The workload both arms measure (the reference arm reports the same)."""
    return {"workload": WORKLOAD_SHORT, "parallelism": f"replicas x{world}",
            "l2": "inputs>L2"}


def cpu_model():
    """The host CPU's model name (lscpu's on Arm, where /proc/cpuinfo gives
    only a part number)."""
    part = None
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                key = line.lower()
                if key.startswith("model name"):
                    return line.split(":", 1)[1].strip()
                if key.startswith("cpu part") and part is None:
                    part = line.split(":", 1)[1].strip()
    except OSError:
        pass
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name:"):
                name = line.split(":", 1)[1].strip()
                return f"{name} ({part})" if part else name
    except (OSError, subprocess.SubprocessError):
        pass
    return part or os.uname().machine


class ClockSampler:
    """SM clock and clock-event reasons during the timed region (NVML via
    ctypes every few ms; nvidia-smi as a fallback).  Read-only."""

    REASONS = {0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap",
               0x8: "hw_slowdown", 0x10: "sync_boost", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown",
               0x100: "display_clock_setting"}

    def __init__(self, torch_device):
        self.samples = []
        self.max_mhz = None
        self._stop = threading.Event()
        self._thread = None
        self._proc = None
        self._nvml = None
        self._h = ctypes.c_void_p()
        try:
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() != 0:
                raise OSError("nvmlInit failed")
            got = False
            bus = self._pci_bus_id(torch_device)
            if bus:
                got = nv.nvmlDeviceGetHandleByPciBusId_v2(bus.encode(), ctypes.byref(self._h)) == 0
            if not got and nv.nvmlDeviceGetHandleByIndex_v2(0, ctypes.byref(self._h)) != 0:
                raise OSError("no NVML handle")
            mx = ctypes.c_uint()
            if nv.nvmlDeviceGetMaxClockInfo(self._h, 1, ctypes.byref(mx)) == 0:
                self.max_mhz = mx.value
            self._reasons_fn = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                getattr(nv, "nvmlDeviceGetCurrentClocksThrottleReasons")
            self._nvml = nv
        except (OSError, AttributeError):
            self._nvml = None

    @staticmethod
    def _pci_bus_id(dev):
        try:
            import torch
            p = torch.cuda.get_device_properties(dev)
            return "%08x:%02x:%02x.0" % (p.pci_domain_id, p.pci_bus_id, p.pci_device_id)
        except Exception:
            return None

    def _loop(self):
        mhz = ctypes.c_uint()
        reasons = ctypes.c_ulonglong()
        while not self._stop.is_set():
            if self._nvml.nvmlDeviceGetClockInfo(self._h, 1, ctypes.byref(mhz)) == 0 and \
                    self._reasons_fn(self._h, ctypes.byref(reasons)) == 0:
                self.samples.append((mhz.value, reasons.value))
            self._stop.wait(0.005)

    def start(self):
        if self._nvml is not None:
            self._thread = threading.Thread(target=self._loop, daemon=True)
            self._thread.start()
        else:
            try:
                self._proc = subprocess.Popen(
                    ["nvidia-smi", "--query-gpu=clocks.sm,clocks.max.sm,clocks_event_reasons.active",
                     "--format=csv,noheader,nounits", "-lms", "100"],
                    stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            except OSError:
                self._proc = None

    def stop(self):
        if self._thread is not None:
            self._stop.set()
            self._thread.join()
        if self._proc is not None:
            self._proc.terminate()
            out, _ = self._proc.communicate()
            for line in out.splitlines():
                try:
                    sm, mx, rs = [v.strip() for v in line.split(",")]
                    self.samples.append((int(sm), int(rs, 16)))
                    self.max_mhz = int(mx)
                except ValueError:
                    pass

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": [], "samples": 0}
        seen = 0
        for _, rs in self.samples:
            seen |= rs
        names = [n for bit, n in self.REASONS.items() if seen & bit and n != "gpu_idle"]
        return {"sm_mhz": statistics.median(m for m, _ in self.samples),
                "sm_max_mhz": self.max_mhz, "reasons": names, "samples": len(self.samples)}


# ------------------------------------------------------------------ distributed

def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def dist_init(world, local, backend):
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group(backend=backend)


def barrier(world, device=None):
    if world > 1:
        import torch.distributed as dist
        if device is not None:
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


def max_over_ranks(world, value, device=None):
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device if device is not None else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_value(world, steps, bytes_per_step, local_ms, device=None):
    """Replicas: every rank moved steps * bytes_per_step; the job took the
    slowest rank's time.  Returns (GB/s of the whole job, max ms)."""
    max_ms = max_over_ranks(world, local_ms, device)
    return world * steps * bytes_per_step / (max_ms / 1e3) / 1e9, max_ms


# ----------------------------------------------------------------- the workload

def step_bytes():
    """Algorithmic bytes of one step: RS reads R*N*e, writes N*e; AG reads N*e,
    writes R*N*e (N*e = 64 MiB summed over the 8 partitions)."""
    rs = (R + 1) * BYTES_PER_RANK
    ag = (R + 1) * BYTES_PER_RANK
    return rs, ag


def host_bits(t):
    import numpy as np
    import torch
    t = t.detach().cpu().contiguous()
    return t.view(torch.int16).numpy().view(np.uint16)


def run_cpu_oracle(xh, budget_s, max_reps=20):
    """The oracle as it stands (single-threaded C) on full steps of the
    workload; repeated until `budget_s` seconds of CPU work."""
    import oracle
    counts = [PART] * R
    reps, t0, y, z = 0, time.perf_counter(), None, None
    while True:
        y = oracle.reduce_scatter(xh, counts, dtype="bf16")
        z = oracle.all_gather(y)
        reps += 1
        el = time.perf_counter() - t0
        if el >= budget_s or reps >= max_reps:
            break
    rs, ag = step_bytes()
    return {"value": reps * (rs + ag) / el / 1e9, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"{reps} full step(s) of the workload (RS then AG, R=8, 8 x 64 MiB bf16) "
                      f"in {el:.1f} s, single-threaded C, {cpu_model()}",
            "short": f"{reps} full steps, {el:.1f} s, {cpu_model().split(' (')[0][:24]}",
            "seconds": el}, y, z


def run_cpu_oracle_threads(xh, budget_s, max_reps=20):
    """The same oracle calls split by output partition over up to R host
    threads: thread k sums partition k (ReduceScatter restricted to one
    partition), then thread j builds output j (the AllGather's block placement
    for one destination, through the oracle's AllToAllV with only column j
    non-zero).  Each element's rank order is unchanged, so the results are
    bit-identical to the single-threaded step; the oracle's own code is not
    changed.  ctypes releases the interpreter lock during each C call.  A finer
    split (sub-ranges of each partition over all 16 cores of a Grace host) needs
    the oracle's separately returned pieces copied together, and that memory-
    bound step then ran slower (10.6 GB/s against 12.3-13.4 GB/s)."""
    import numpy as np
    from concurrent.futures import ThreadPoolExecutor
    import oracle
    threads = max(1, min(R, os.cpu_count() or 1))

    def rs_part(k):
        counts = [0] * R
        counts[k] = PART
        return oracle.reduce_scatter(xh, counts, [k * PART] * R, dtype="bf16")[k]

    def ag_dest(j, y):
        C = np.zeros((R, R), dtype=np.uint64)
        C[:, j] = PART
        return oracle.all_to_all_v(y, C)[j]

    reps, t0 = 0, time.perf_counter()
    with ThreadPoolExecutor(max_workers=threads) as pool:
        while True:
            y = list(pool.map(rs_part, range(R)))
            z = list(pool.map(lambda j: ag_dest(j, y), range(R)))
            reps += 1
            el = time.perf_counter() - t0
            if el >= budget_s or reps >= max_reps:
                break
    rs, ag = step_bytes()
    return {"value": reps * (rs + ag) / el / 1e9, "unit": UNIT, "cores": threads,
            "kind": "oracle, split by output partition",
            "sample": f"{reps} full step(s) of the workload in {el:.1f} s, {threads} threads, "
                      f"{cpu_model()}"}, y, z


def bench_reference(args):
    """The reference arm: the CPU oracle timed on the host cores."""
    world, rank, local = dist_setup(args)
    if rank != 0:
        return
    import numpy as np
    import workloads
    import torch
    x = workloads.rank_buffers(WORKLOAD, R, ELEMS_PER_RANK, "bf16", device="cpu")
    xh = [host_bits(t) for t in x]
    warm = max(0, args.warmup)
    import oracle
    oracle.build()
    for _ in range(min(warm, 1)):
        run_cpu_oracle(xh, 0.0, max_reps=1)
    steps = max(1, args.steps)
    # each timed step is one full step of the workload; bounded to a few minutes
    steps = min(steps, 60)
    t0 = time.perf_counter()
    for _ in range(steps):
        run_cpu_oracle(xh, 0.0, max_reps=1)
    el = time.perf_counter() - t0
    rs, ag = step_bytes()
    value = steps * (rs + ag) / el / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": steps, "warmup": warm, "ms_per_step": el / steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": bench_config(args.gpus),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": f"{steps} full step(s), single-threaded C, {cpu_model()}"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "note": "the pages publish no code; the CPU oracle written from them is the reference arm",
    }
    print(json.dumps(line), flush=True)


# Source files whose content determines each kernel family's device code.
KERNEL_SOURCES = {
    "zs": ["atom.cuh", "plan.h", "zs_kernels.cuh"],
    "snac": ["atom.cuh", "plan.h", "snac.h", "snac_kernels.cu", "zs_kernels.cuh"],
}


def product_source(text):
    """The source as the product build compiles it: the checked build's parts
    left out -- blocks under `#if defined(PURLIN_CHECKED)` (their `#else`
    branch is kept), and the PURLIN_CHECK_* macros, which the product build
    defines to nothing."""
    out = []
    stack = []   # per open #if: "checked" (inside the checked branch), "else" or "other"
    for line in text.splitlines():
        t = line.strip()
        in_checked = "checked" in stack
        if t.startswith("#if"):
            stack.append("checked" if t.startswith("#if defined(PURLIN_CHECKED)") else "other")
            if stack[-1] == "other" and not in_checked:
                out.append(line)
            continue
        if t.startswith("#else") and stack:
            if stack[-1] == "checked":
                stack[-1] = "else"
            elif not in_checked:
                out.append(line)
            continue
        if t.startswith("#endif") and stack:
            kind = stack.pop()
            if kind == "other" and "checked" not in stack:
                out.append(line)
            continue
        if in_checked:
            continue
        if t.startswith("PURLIN_CHECK_") or t.startswith("#define PURLIN_CHECK_"):
            continue
        out.append(line)
    return "\n".join(out)


def code_tokens(text):
    """C/C++ source with comments removed and whitespace runs collapsed (string
    and character literals kept as written): what the compiler sees."""
    text = product_source(text)
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
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


def sources_digest(family, read=None):
    """Digest of a kernel family's sources as compiled (comments and layout do
    not count), which ties an ncu summary's traffic to the code it measured."""
    import hashlib
    src = os.path.join(ROOT, "reduce_datapath_gb300", "csrc")
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[family]:
        if read is None:
            with open(os.path.join(src, f), encoding="utf-8") as fh:
                text = fh.read()
        else:
            text = read(f)
        h.update(code_tokens(text).encode())
        h.update(b"\0")
    return h.hexdigest()[:16]


def traffic_from_profiles(kernel_key):
    """Per-launch DRAM bytes of a kernel from the committed ncu summaries, if
    taken on the current sources of that kernel family: (bytes, kind, digest),
    bytes None if there is none.  A summary line reads
    "traffic: <kernel_key> <bytes per launch> sources=<digest>" (one launch
    captured alone, caches flushed) or "traffic-in-step: ..." (one launch of the
    benchmark step, caches as the step leaves them), which is preferred."""
    family = "snac" if kernel_key.startswith("snac") else "zs"
    digest = sources_digest(family)
    pdir = os.path.join(ROOT, "profiles")
    found = {}
    if os.path.isdir(pdir):
        for f in sorted(os.listdir(pdir)):
            if not f.endswith((".md", ".txt")):
                continue
            with open(os.path.join(pdir, f)) as fh:
                for line in fh:
                    parts = line.strip().strip("`").split()
                    if len(parts) == 4 and parts[0] in ("traffic:", "traffic-in-step:") \
                            and parts[1] == kernel_key and parts[3] == f"sources={digest}":
                        found[parts[0]] = int(parts[2])
    if "traffic-in-step:" in found:
        return found["traffic-in-step:"], "in step", digest
    if "traffic:" in found:
        return found["traffic:"], "alone, cold L2", digest
    return None, None, digest


def roofline_entry(coll, peak, peak_kind, name, traffic, traffic_kind):
    """The roofline object of the dominant kernel: algorithmic bytes per launch
    over its event-timed duration, against the measured copy peak; beside it
    the DRAM bytes ncu counted for one launch over the same duration
    (dram_frac), which tells bytes served by HBM from bytes served by L2."""
    dur_s = coll["us"] / 1e6
    out = {"bound": "hbm", "achieved": coll["gbs"], "peak": peak, "unit": "GB/s",
           "frac": coll["gbs"] / peak, "traffic": traffic, "kernel": name,
           "algorithmic_bytes_per_launch": coll["bytes"],
           "peak_kind": "of measured" if peak_kind == "measured" else "of fallback"}
    if traffic is not None:
        out["dram_frac"] = traffic / dur_s / 1e9 / peak
        out["traffic_kind"] = traffic_kind
    return out


def _r(v, nd=4):
    return round(v, nd) if isinstance(v, float) else v


def compact_line(*, world, steps, warmup, value, ms_per_step, variant, roofline, per, e2e,
                 cpu, parity, lat, launches, clocks, peak, step_traffic):
    """The benchmark's result line: the contract keys and the figures that
    back them, short enough to be read whole from the end of a log."""
    rf = {k: roofline.get(k) for k in ("bound", "achieved", "peak", "unit", "frac", "traffic",
                                       "dram_frac", "kernel", "algorithmic_bytes_per_launch")}
    for k in ("achieved", "peak"):
        rf[k] = _r(rf[k], 1)
    for k in ("frac", "dram_frac"):
        rf[k] = _r(rf[k], 4)
    line = {
        "metric": METRIC, "value": _r(value, 1), "unit": UNIT, "n_gpus": world, "steps": steps,
        "warmup": warmup, "ms_per_step": _r(ms_per_step, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": bench_config(world) | {"variant": variant},
        "roofline": rf,
        "e2e": {"value": _r(e2e["value"], 1), "unit": e2e["unit"],
                "h2d_bytes_per_step": e2e["h2d_bytes_per_step"],
                "d2h_bytes_per_step": e2e["d2h_bytes_per_step"],
                "ms_per_step": _r(e2e.get("ms_per_step"), 2),
                "link_frac": _r(e2e.get("link_frac"), 2)},
        "cpu_baseline": None if cpu is None else
        {"value": _r(cpu["value"], 3), "unit": cpu["unit"], "cores": cpu["cores"],
         "kind": cpu["kind"], "sample": cpu.get("short", "full steps")},
        "allreduce_4KiB_us": None if lat is None else _r(lat.get("us_graph_per_launch"), 3),
        "parity_vs_oracle": parity,
        "gpu_launches": launches,
        "clocks": {"sm_mhz": clocks.get("sm_mhz"), "sm_max_mhz": clocks.get("sm_max_mhz"),
                   "reasons": clocks.get("reasons", [])},
    }
    if step_traffic is not None:
        line["step_dram_frac"] = _r(step_traffic / (ms_per_step / 1e3) / 1e9 / peak)
    return line


def emit(line, studies, studies_out=None):
    """Side studies go to a file (or an earlier stdout line); the result line
    is always the last line on stdout."""
    if studies_out:
        with open(studies_out, "w") as f:
            json.dump(studies, f)
    else:
        print(json.dumps({"studies": studies}), flush=True)
    print(json.dumps(line, separators=(",", ":")), flush=True)


def bench_purlin(args):
    import numpy as np
    import torch

    import reduce_datapath_gb300 as rd
    import workloads

    world, rank, local = dist_setup(args)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist_init(world, local, "nccl")
    rd.build() if rank == 0 else None
    barrier(world, dev)
    rd.lib()

    peak, peak_kind = measured_peaks()
    stream = torch.cuda.Stream(device=dev)
    h = rd.purlin_create(R, args.staging, local)
    variant = {"zs": rd.VARIANT_ZS, "staged": rd.VARIANT_STAGED,
               "staged_y": rd.VARIANT_STAGED_Y}[args.variant]
    rd.purlin_set_policy(h, args.chunk, args.depth, args.ctas, variant)

    x = workloads.rank_buffers(WORKLOAD, R, ELEMS_PER_RANK, "bf16", device=dev)
    y = [torch.empty(PART, dtype=torch.bfloat16, device=dev) for _ in range(R)]
    z = [torch.empty(ELEMS_PER_RANK, dtype=torch.bfloat16, device=dev) for _ in range(R)]
    counts = [PART] * R
    torch.cuda.synchronize()

    # marshalled once: each repeat is one C call that plans and launches (the
    # side studies change the handle's policy between calls)
    rs = rd.prepare(rd.purlin_reduce_scatter, h, x, y, counts, None, "bf16", stream=stream)
    ag = rd.prepare(rd.purlin_all_gather, h, y, z, counts, None, "bf16", stream=stream)
    # planned once: each timed repeat is one launch of the kept plan
    rs_plan = rd.plan(rd.purlin_reduce_scatter, h, x, y, counts, None, "bf16", stream=stream)
    ag_plan = rd.plan(rd.purlin_all_gather, h, y, z, counts, None, "bf16", stream=stream)

    with torch.cuda.stream(stream):
        for _ in range(max(3, args.warmup)):
            rs()
            ag()
    torch.cuda.synchronize()
    rs_info = None
    rs()
    rs_info = rd.purlin_last_launch(h)
    ag()
    ag_info = rd.purlin_last_launch(h)
    torch.cuda.synchronize()

    # The timed region: K steps back to back, events only at its two ends, so
    # that nothing sits between the kernels (an event between two launches
    # stops the second one's programmatic early launch).
    K = max(1, args.steps)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(dev)
    barrier(world, dev)
    torch.cuda.synchronize()
    clocks.start()
    t0.record(stream)
    for i in range(K):
        rs_plan()
        ag_plan()
    t1.record(stream)
    torch.cuda.synchronize()
    clocks.stop()
    barrier(world, dev)
    total_ms = t0.elapsed_time(t1)
    # The split between the two collectives, from a second run of the same
    # steps with an event around each launch.
    Kb = min(K, 100)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(Kb)]
    for i in range(Kb):
        ev[i][0].record(stream)
        rs_plan()
        ev[i][1].record(stream)
        ag_plan()
        ev[i][2].record(stream)
    torch.cuda.synchronize()
    rs_ms = [ev[i][0].elapsed_time(ev[i][1]) for i in range(Kb)]
    ag_ms = [ev[i][1].elapsed_time(ev[i][2]) for i in range(Kb)]
    split_ms = sum(rs_ms) + sum(ag_ms)
    status = rd.purlin_query_status(h)
    if status != rd.OK:
        raise RuntimeError("device status: " + rd.purlin_status_string(status))
    launches = K * (rs_info["kernels"] + ag_info["kernels"])
    rs_b, ag_b = step_bytes()
    value, max_ms = whole_job_value(world, K, rs_b + ag_b, total_ms, dev)

    rs_avg = sum(rs_ms) / Kb
    ag_avg = sum(ag_ms) / Kb
    per = {
        "reduce_scatter": {"us": rs_avg * 1e3, "gbs": rs_b / (rs_avg / 1e3) / 1e9,
                           "bytes": rs_b, "grid": rs_info["grid"]},
        "all_gather": {"us": ag_avg * 1e3, "gbs": ag_b / (ag_avg / 1e3) / 1e9,
                       "bytes": ag_b, "grid": ag_info["grid"]},
    }
    for v in per.values():
        v["frac_of_peak"] = v["gbs"] / peak
        v["sm_bound"] = min(v["grid"], rs_info["sms"])
    dom = "reduce_scatter" if rs_avg >= ag_avg else "all_gather"
    family = "zs" if args.variant == "zs" else "snac"
    keys = {"reduce_scatter": ("zs_reduce" if family == "zs" else "snac") + ":" + WORKLOAD,
            "all_gather": ("zs_copy" if family == "zs" else "snac_ag") + ":" + WORKLOAD}
    # DRAM bytes per launch from the committed ncu summaries: the in-step
    # capture (caches as the step leaves them) where there is one, else the
    # cold one-launch capture; None once the kernel sources have changed.
    traffic = {}
    digest = None
    for coll, key in keys.items():
        t, kind, digest = traffic_from_profiles(key)
        traffic[coll] = (t, kind)
    roofline = roofline_entry(per[dom], peak, peak_kind, "rs" if dom == "reduce_scatter" else "ag",
                              *traffic[dom])
    step_traffic = None
    if all(t is not None for t, _ in traffic.values()):
        step_traffic = sum(t for t, _ in traffic.values())
    per["split_run_step_us"] = split_ms / Kb * 1e3

    lat = staged = frugal = tree = configs = sweep = None
    if not args.quick:
        # ---- AllReduce latency at 4 KiB per rank (R=8 bf16, 2048 elements)
        lat = allreduce_latency(rd, torch, dev, stream, variant)
        lat["c_caller"] = c_caller_cost(rd)

        # ---- the same step through the staged (SNAC) path, default policy
        staged = staged_step(rd, torch, h, rs, ag, stream, rs_b + ag_b, peak)

        # ---- bandwidth vs CTAs launched, per Atom, and the copy-engine AllGather
        frugal = cta_study(rd, torch, h, rs, ag, stream, rs_b, peak)

        # ---- the pairwise rank order, reported beside the fixed order
        tree = tree_order_report(rd, torch, h, x, y, counts, stream, rs_b, peak)

        # ---- the other workload configurations, zero staging (default policy)
        configs = other_configs(rd, torch, dev, stream, peak)
        configs["zs_by_rank_count"] = rank_scaling(rd, torch, dev, stream, peak)
        configs["off_grid_partitions"] = off_grid_partitions(rd, torch, dev, stream, peak)
        configs["layout_fuzz"] = layout_fuzz(rd, torch, dev, stream, peak)

        # ---- AllReduce size sweep: zero staging vs SNAC (default policy)
        sweep = allreduce_sweep(rd, torch, dev, stream, peak)
        configs["allreduce_noalloc"] = noalloc_allreduce(rd, torch, dev, stream, peak)

    # ---- end to end: inputs from pinned host memory, outputs back to it; with
    # several ranks the job's figure is all ranks' bytes over the slowest rank
    barrier(world, dev)
    e2e = bench_e2e(args, rd, torch, h, x, y, z, counts, stream)
    e2e["value"], e2e_ms = whole_job_value(world, e2e["steps"], rs_b + ag_b,
                                           e2e["ms_per_step"] * e2e["steps"], dev)
    e2e["ms_per_step"] = e2e_ms / e2e["steps"]

    # ---- CPU oracle baseline and a bit-exact check of this run's result
    cpu = None
    cpu_threads = None
    parity = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline and not args.quick:
        xh = [host_bits(t) for t in x]
        cpu, want_y, want_z = run_cpu_oracle(xh, args.cpu_seconds)
        cpu.pop("seconds", None)
        rs()
        ag()
        torch.cuda.synchronize()
        parity = all(np.array_equal(host_bits(y[k]), want_y[k]) for k in range(R)) and \
            all(np.array_equal(host_bits(z[k]), want_z[k]) for k in range(R))
        cpu_threads, ty, tz = run_cpu_oracle_threads(xh, args.cpu_seconds / 2)
        cpu_threads["bit_identical_to_single_thread"] = bool(
            all(np.array_equal(ty[k], want_y[k]) for k in range(R)) and
            all(np.array_equal(tz[k], want_z[k]) for k in range(R)))

    rd.purlin_destroy(h)
    if rank != 0:
        return
    line = compact_line(
        world=world, steps=K, warmup=max(3, args.warmup), value=value, ms_per_step=max_ms / K,
        variant=args.variant, roofline=roofline, per=per, e2e=e2e, cpu=cpu, parity=parity,
        lat=lat, launches=launches, clocks=clocks.summary(), peak=peak,
        step_traffic=step_traffic)
    studies = {
        "per_collective": per,
        "allreduce_4KiB": lat,
        "staged_step": staged,
        "cta_study": frugal,
        "configs": configs,
        "tree_order": tree,
        "allreduce_sweep": sweep,
        "e2e": e2e,
        "cpu_baseline": cpu,
        "cpu_baseline_threads": cpu_threads,
        "roofline": roofline,
        "sources": digest,
    }
    emit(line, studies, args.studies_out)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def _graph_us(torch, stream, fn, per_graph=50, replays=4):
    """Device time per launch: `per_graph` launches captured in one CUDA graph,
    replayed; None if the launch cannot be captured."""
    try:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for _ in range(per_graph):
                fn()
    except Exception:
        torch.cuda.synchronize()
        return None
    with torch.cuda.stream(stream):
        g.replay()
        torch.cuda.synchronize()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(replays):
            g.replay()
        b.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(b) * 1e3 / (per_graph * replays)


def _cold_l2_us(torch, stream, fn, flush, reps=20):
    """Median device time of one call right after a write of twice the L2
    size, so that its buffers come from HBM."""
    ts = []
    with torch.cuda.stream(stream):
        for _ in range(reps):
            flush.fill_(1.0)
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            b.synchronize()
            ts.append(a.elapsed_time(b) * 1e3)
    return statistics.median(ts)


def _events_us(torch, stream, fn, iters):
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(iters):
        fn()
    b.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(b) * 1e3 / iters


def staged_step(rd, torch, h, rs, ag, stream, step_b, peak):
    """The benchmark step (RS then AG) through SNAC staging (default policy):
    sums staging the R input chunks (the top-level figures) and, under
    `staged_y`, sums staging the reduced chunk."""
    def one(variant):
        rd.purlin_set_policy(h, 0, 0, 0, variant)
        try:
            for _ in range(3):
                rs()
                ag()
            torch.cuda.synchronize()
            rs_us = _events_us(torch, stream, rs, 20)
            rs_info = rd.purlin_last_launch(h)
            ag_us = _events_us(torch, stream, ag, 20)
            info = rd.purlin_last_launch(h)
            if rd.purlin_query_status(h) != rd.OK:
                raise RuntimeError("staged step: device status not ok")
        finally:
            rd.purlin_set_policy(h, 0, 0, 0, rd.VARIANT_ZS)
        us = rs_us + ag_us
        return {"us": us, "gbs": step_b / (us / 1e6) / 1e9,
                "frac_of_peak": step_b / (us / 1e6) / 1e9 / peak,
                "reduce_scatter_us": rs_us, "all_gather_us": ag_us,
                "reduce_scatter_chunk_bytes": rs_info["chunk_bytes"],
                "chunk_bytes": info["chunk_bytes"], "depth": info["depth"], "grid": info["grid"]}

    out = one(rd.VARIANT_STAGED)
    out["staged_y"] = one(rd.VARIANT_STAGED_Y)
    return out


def cta_study(rd, torch, h, rs, ag, stream, coll_b, peak):
    """Bandwidth of the AllGather (copy) and ReduceScatter (sum) of the step as
    a function of the CTAs launched, for the vector and TMA-bulk Atoms, plus the
    AllGather on the copy engines (no kernel).  Concurrent SM use is bounded by
    min(CTAs launched, SMs); beyond the resident CTAs (2 per SM for the vector
    kernels, 1 for the bulk one) extra CTAs queue and are handed to SMs as they
    drain.  ctas 0 = the library's default grid (reported in `grid`)."""
    rows = []

    def row(coll, fn, atom_name, ctas, **extra):
        rd.purlin_set_policy(h, 0, 0, ctas, rd.VARIANT_ZS)
        fn()
        us = _events_us(torch, stream, fn, 10)
        rows.append({"collective": coll, "atom": atom_name, **extra, "ctas": ctas,
                     "grid": rd.purlin_last_launch(h)["grid"], "us": round(us, 1),
                     "gbs": round(coll_b / (us / 1e6) / 1e9, 1),
                     "frac_of_peak": round(coll_b / (us / 1e6) / 1e9 / peak, 3)})

    try:
        for atom_name, atom, ctas_list in (
                ("vector", rd.ATOM_VECTOR, (8, 16, 38, 76, 152, 304, 608, 1216, 0)),
                ("bulk", rd.ATOM_BULK, (8, 16, 38, 76, 152, 608, 0))):
            rd.purlin_set_atom(h, atom)
            for ctas in ctas_list:
                row("all_gather", ag, atom_name, ctas)
        rd.purlin_set_atom(h, rd.ATOM_VECTOR)
        for ctas in (8, 16, 38, 76, 152, 304, 1216, 0):
            row("reduce_scatter", rs, "vector", ctas)
        rd.purlin_set_atom(h, rd.ATOM_VECTOR)
        rd.purlin_set_direction(h, rd.DIRECTION_PULL)
        for ctas in (152, 304, 0):
            row("all_gather", ag, "vector", ctas, direction="pull")
        rd.purlin_set_direction(h, rd.DIRECTION_AUTO)
        rd.purlin_set_atom(h, rd.ATOM_COPY_ENGINE)
        row("all_gather", ag, "copy_engine", 0)
        if rd.purlin_query_status(h) != rd.OK:
            raise RuntimeError("cta study: device status not ok")
    finally:
        rd.purlin_set_atom(h, rd.ATOM_AUTO)
        rd.purlin_set_direction(h, rd.DIRECTION_AUTO)
        rd.purlin_set_policy(h, 0, 0, 0, rd.VARIANT_ZS)
    return rows


def tree_order_report(rd, torch, h, x, y_fixed, counts, stream, coll_b, peak):
    """The step's ReduceScatter with the pairwise rank order: its bandwidth and
    how far it lands from the fixed order (y_fixed holds the fixed-order result
    of the last timed step)."""
    y = [torch.empty_like(t) for t in y_fixed]
    rs_tree = rd.prepare(rd.purlin_reduce_scatter, h, x, y, counts, None, "bf16", stream=stream)
    rd.purlin_set_reduce_order(h, rd.ORDER_TREE)
    try:
        for _ in range(3):
            rs_tree()
        us = _events_us(torch, stream, rs_tree, 20)
    finally:
        rd.purlin_set_reduce_order(h, rd.ORDER_FIXED)
    c = y_fixed[0].numel()
    differing, max_ulp, max_scaled = 0, 0, 0.0
    for k in range(R):
        a = y[k].view(torch.int16).int()
        b = y_fixed[k].view(torch.int16).int()
        differing += int((a != b).sum())
        same_sign = (a < 0) == (b < 0)
        if bool(same_sign.any()):
            max_ulp = max(max_ulp, int((a - b).abs()[same_sign].max()))
        mag = sum(t[k * c:(k + 1) * c].float().abs() for t in x)
        err = (y[k].float() - y_fixed[k].float()).abs() / mag.clamp_min(1e-30)
        max_scaled = max(max_scaled, float(err.max()))
    gbs = coll_b / (us / 1e6) / 1e9
    return {"collective": "reduce_scatter", "us": round(us, 2), "gbs": round(gbs, 1),
            "frac_of_peak": round(gbs / peak, 3),
            "elements_differing_from_fixed_order": round(differing / (R * c), 4),
            "max_bf16_ulp_vs_fixed_order": max_ulp,
            "max_abs_diff_over_sum_abs": max_scaled}


def rank_scaling(rd, torch, dev, stream, peak):
    """Zero-staging bandwidth against the number of virtual ranks (64 MiB per
    rank): the Atom's R-way loop at R = 2, 4, 8 in bf16 (AllReduce,
    ReduceScatter, AllGather), and the fp32 sums (AllReduce, ReduceScatter)."""
    out = []
    for dtype, colls in (("bf16", ("all_reduce", "reduce_scatter", "all_gather")),
                         ("f32", ("all_reduce", "reduce_scatter"))):
        tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
        esz = 2 if dtype == "bf16" else 4
        n = BYTES_PER_RANK // esz
        for R_ in (2, 4, 8):
            h = rd.purlin_create(R_, 0, dev.index)
            try:
                x = [torch.randn(n, device=dev).to(tdt) for _ in range(R_)]
                o = [torch.empty_like(t) for t in x]
                c = n // R_
                y = [torch.empty(c, dtype=tdt, device=dev) for _ in range(R_)]
                runs = {"all_reduce": (lambda: rd.purlin_all_reduce(h, x, o, n, dtype, stream=stream),
                                       2 * R_ * n * esz),
                        "reduce_scatter": (lambda: rd.purlin_reduce_scatter(
                            h, x, y, [c] * R_, None, dtype, stream=stream), (R_ + 1) * c * R_ * esz),
                        "all_gather": (lambda: rd.purlin_all_gather(
                            h, y, o, [c] * R_, None, dtype, stream=stream), (R_ + 1) * c * R_ * esz)}
                for name in colls:
                    fn, nbytes = runs[name]
                    with torch.cuda.stream(stream):
                        for _ in range(3):
                            fn()
                    torch.cuda.synchronize()
                    us = _events_us(torch, stream, fn, 20)
                    gbs = nbytes / (us / 1e6) / 1e9
                    out.append({"R": R_, "dtype": dtype, "collective": name, "us": round(us, 1),
                                "gbs": round(gbs, 1), "frac_of_peak": round(gbs / peak, 3)})
                del x, o, y
                if rd.purlin_query_status(h) != rd.OK:
                    raise RuntimeError("rank scaling: device status not ok")
            finally:
                rd.purlin_destroy(h)
                torch.cuda.empty_cache()
    return out


def off_grid_partitions(rd, torch, dev, stream, peak):
    """Layouts whose partitions start off the 32-byte grid (64 MiB per rank,
    bf16): 3 ranks (partitions of n/3 elements start 20 bytes past a
    boundary), 8 ranks with partitions 3 elements short, and an AllReduce into
    outputs one element into their allocations.  The plans read the sources
    through shifted vector bodies."""
    out = []
    for R_, trim in ((3, 0), (8, 3)):
        n = BYTES_PER_RANK // 2
        c = n // R_ - trim
        h = rd.purlin_create(R_, 0, dev.index)
        try:
            x = [torch.randn(R_ * c, device=dev).to(torch.bfloat16) for _ in range(R_)]
            y = [torch.empty(c, dtype=torch.bfloat16, device=dev) for _ in range(R_)]
            zf = [torch.empty(R_ * c + 1, dtype=torch.bfloat16, device=dev) for _ in range(R_)]
            z = [t[:R_ * c] for t in zf]
            zo = [t[1:] for t in zf]
            m = R_ * c
            runs = (("reduce_scatter", lambda: rd.purlin_reduce_scatter(
                        h, x, y, [c] * R_, None, "bf16", stream=stream), (R_ + 1) * c * R_ * 2),
                    ("all_gather", lambda: rd.purlin_all_gather(
                        h, y, z, [c] * R_, None, "bf16", stream=stream), (R_ + 1) * c * R_ * 2),
                    ("all_reduce_off_grid_outputs", lambda: rd.purlin_all_reduce(
                        h, x, zo, m, "bf16", stream=stream), 2 * R_ * m * 2))
            for name, fn, nbytes in runs:
                with torch.cuda.stream(stream):
                    for _ in range(3):
                        fn()
                torch.cuda.synchronize()
                us = _events_us(torch, stream, fn, 20)
                gbs = nbytes / (us / 1e6) / 1e9
                out.append({"R": R_, "partition_elems": c, "collective": name, "us": round(us, 1),
                            "gbs": round(gbs, 1), "frac_of_peak": round(gbs / peak, 3)})
            if rd.purlin_query_status(h) != rd.OK:
                raise RuntimeError("off-grid partitions: device status not ok")
            del x, y, zf, z, zo
        finally:
            rd.purlin_destroy(h)
            torch.cuda.empty_cache()
    return out


def layout_fuzz(rd, torch, dev, stream, peak, trials=16, seed=7):
    """Bandwidth over random layouts (seeded): R in 2..8, a random collective
    (ReduceScatterV, AllGatherV, AllReduce, AllToAllV), bf16 / fp32 (and bytes
    for copies), 16-64 MiB per rank, random counts, each rank's input and output
    buffer 0-2 elements into its allocation with probability 0.3.  Reports
    every trial and the minimum and median fraction of the peak."""
    import numpy as np
    rng = np.random.default_rng(seed)
    tdt = {"bf16": torch.bfloat16, "f32": torch.float32, "u8": torch.uint8}
    esz = {"bf16": 2, "f32": 4, "u8": 1}
    out, handles = [], {}
    try:
        for trial in range(trials):
            R_ = int(rng.integers(2, R + 1))
            coll = ("rs", "ag", "ar", "a2av")[int(rng.integers(0, 4))]
            dts = ("bf16", "f32") if coll in ("rs", "ar") else ("bf16", "f32", "u8")
            dtype = dts[int(rng.integers(0, len(dts)))]
            e = esz[dtype]
            n = (int(rng.integers(16, 65)) << 20) // e
            in_off = [int(rng.integers(0, 3)) * int(rng.random() < 0.3) for _ in range(R_)]
            out_off = [int(rng.integers(0, 3)) * int(rng.random() < 0.3) for _ in range(R_)]
            h = handles.setdefault(R_, rd.purlin_create(R_, 0, dev.index))

            def buf(m, off, fill=False):
                t = torch.empty(m + off + 16, dtype=tdt[dtype], device=dev)
                if fill:
                    t.copy_(torch.randn(t.numel(), device=dev).to(tdt[dtype]))
                return t[off:off + m]

            if coll in ("rs", "ag"):
                counts = rng.integers(1, 2 * n // R_, size=R_)
                counts = (counts * (n / counts.sum())).astype(np.int64) + 1
                total = int(counts.sum())
                if coll == "rs":
                    x = [buf(total, in_off[r], True) for r in range(R_)]
                    y = [buf(int(c), out_off[k]) for k, c in enumerate(counts)]
                    fn = lambda: rd.purlin_reduce_scatter(h, x, y, counts, None, dtype, stream=stream)
                else:
                    x = [buf(int(c), in_off[k]) for k, c in enumerate(counts)]
                    y = [buf(total, out_off[j]) for j in range(R_)]
                    fn = lambda: rd.purlin_all_gather(h, x, y, counts, None, dtype, stream=stream)
                nbytes = (R_ + 1) * total * e
            elif coll == "ar":
                x = [buf(n, in_off[r], True) for r in range(R_)]
                y = [buf(n, out_off[r]) for r in range(R_)]
                fn = lambda: rd.purlin_all_reduce(h, x, y, n, dtype, stream=stream)
                nbytes = 2 * R_ * n * e
            else:
                C = rng.integers(1, 2 * n // (R_ * R_), size=(R_, R_))
                x = [buf(int(C[a].sum()), in_off[a]) for a in range(R_)]
                y = [buf(int(C[:, j].sum()), out_off[j]) for j in range(R_)]
                fn = lambda: rd.purlin_all_to_all_v(h, x, y, C, None, None, dtype, stream=stream)
                nbytes = 2 * int(C.sum()) * e
            with torch.cuda.stream(stream):
                for _ in range(2):
                    fn()
            torch.cuda.synchronize()
            us = _events_us(torch, stream, fn, 10)
            if rd.purlin_query_status(h) != rd.OK:
                raise RuntimeError("layout fuzz: device status not ok")
            gbs = nbytes / (us / 1e6) / 1e9
            out.append({"R": R_, "collective": coll, "dtype": dtype, "mbytes_moved": round(nbytes / 1e6, 1),
                        "in_off": in_off, "out_off": out_off, "us": round(us, 1),
                        "frac_of_peak": round(gbs / peak, 3)})
            del x, y
            torch.cuda.empty_cache()
    finally:
        for h in handles.values():
            rd.purlin_destroy(h)
    fr = sorted(r["frac_of_peak"] for r in out)
    return {"trials": out, "min_frac": fr[0], "median_frac": fr[len(fr) // 2],
            "timing": "events over 10 launches from Python (small calls include host time)"}


def other_configs(rd, torch, dev, stream, peak):
    """The remaining workload configurations, each timed with CUDA events:
    AllReduce R=2 fp32 4096 elements (latency); MoE AllToAllV dispatch and its
    inverse (R=8, 4096 tokens x 7168 bf16 per source, Zipf(1.2)); data-parallel
    attention AllGatherV + ReduceScatterV (token counts uniform in [1, 2048]);
    AllGather with 1 GiB out per rank; AllReduce with 1 GiB per rank."""
    import workloads
    H = workloads.HIDDEN
    out = {}

    def entry(us, nbytes):
        gbs = nbytes / (us / 1e6) / 1e9
        return {"us": round(us, 2), "gbs": round(gbs, 1), "frac_of_peak": round(gbs / peak, 3),
                "algorithmic_bytes": nbytes}

    # AllReduce R=2 fp32 4096 integers: a latency point
    h2 = rd.purlin_create(2, 0, dev.index)
    try:
        x = workloads.rank_buffers("allreduce_r2_f32", 2, 4096, "f32", device=dev, values="int")
        o = [torch.empty_like(t) for t in x]
        fn = lambda: rd.purlin_all_reduce(h2, x, o, 4096, "f32", stream=stream)
        fn()
        us = _graph_us(torch, stream, fn) or _events_us(torch, stream, fn, 200)
        out["allreduce_r2_f32_4096"] = entry(us, 2 * 2 * 4096 * 4) | {"timing": "cuda graph"}
    finally:
        rd.purlin_destroy(h2)

    h = rd.purlin_create(R, 0, dev.index)
    try:
        # MoE dispatch and inverse
        T = 4096
        C = workloads.zipf_pair_counts(R, T, workloads.ZIPF_S, workloads.seed_for("moe_a2av_r8", 9))
        x = workloads.rank_buffers("moe_a2av_r8", R, T * H, "bf16", device=dev)
        recv = [torch.empty(int(C[:, j].sum()) * H, dtype=torch.bfloat16, device=dev)
                for j in range(R)]
        back = [torch.empty_like(t) for t in x]
        fwd = lambda: rd.purlin_all_to_all_v(h, x, recv, C * H, None, None, "bf16", stream=stream)
        inv = lambda: rd.purlin_all_to_all_v(h, recv, back, C.T * H, None, None, "bf16",
                                             stream=stream)
        for _ in range(3):
            fwd()
            inv()
        nb = 2 * int(C.sum()) * H * 2
        out["moe_a2av_dispatch"] = entry(_events_us(torch, stream, fwd, 20), nb)
        out["moe_a2av_combine"] = entry(_events_us(torch, stream, inv, 20), nb)
        out["moe_a2av_received_tokens"] = [int(v) for v in C.sum(axis=0)]
        del x, recv, back

        # data-parallel attention: AllGatherV + ReduceScatterV
        tok = workloads.uniform_token_counts(R, 1, 2048, workloads.seed_for("dp_attn_agv_rsv_r8", 9))
        counts = [int(t) * H for t in tok]
        Tt = sum(counts)
        ag_in = [torch.randn(c, device=dev).to(torch.bfloat16) for c in counts]
        ag_out = [torch.empty(Tt, dtype=torch.bfloat16, device=dev) for _ in range(R)]
        rs_in = [torch.randn(Tt, device=dev).to(torch.bfloat16) for _ in range(R)]
        rs_out = [torch.empty(c, dtype=torch.bfloat16, device=dev) for c in counts]
        agv = lambda: rd.purlin_all_gather(h, ag_in, ag_out, counts, None, "bf16", stream=stream)
        rsv = lambda: rd.purlin_reduce_scatter(h, rs_in, rs_out, counts, None, "bf16",
                                               stream=stream)
        for _ in range(3):
            agv()
            rsv()
        nb = (R + 1) * Tt * 2
        out["dp_attn_allgatherv"] = entry(_events_us(torch, stream, agv, 20), nb)
        out["dp_attn_reducescatterv"] = entry(_events_us(torch, stream, rsv, 20), nb)
        out["dp_attn_tokens"] = [int(t) for t in tok]
        del ag_in, ag_out, rs_in, rs_out
        torch.cuda.empty_cache()

        # AllGather, 1 GiB out per rank (128 MiB in per rank)
        c = (128 << 20) // 2
        ag_in = [torch.randn(c, device=dev).to(torch.bfloat16) for _ in range(R)]
        ag_out = [torch.empty(R * c, dtype=torch.bfloat16, device=dev) for _ in range(R)]
        ag1 = lambda: rd.purlin_all_gather(h, ag_in, ag_out, [c] * R, None, "bf16", stream=stream)
        for _ in range(3):
            ag1()
        out["allgather_1GiB_out"] = entry(_events_us(torch, stream, ag1, 10), (R + 1) * R * c * 2)
        del ag_in, ag_out
        torch.cuda.empty_cache()

        # AllReduce, 1 GiB per rank
        n = (1 << 30) // 2
        ar_in = [torch.empty(n, dtype=torch.bfloat16, device=dev).normal_() for _ in range(R)]
        ar_out = [torch.empty_like(t) for t in ar_in]
        ar1 = lambda: rd.purlin_all_reduce(h, ar_in, ar_out, n, "bf16", stream=stream)
        for _ in range(3):
            ar1()
        out["allreduce_1GiB"] = entry(_events_us(torch, stream, ar1, 10), 2 * R * n * 2)
        del ar_in, ar_out
        if rd.purlin_query_status(h) != rd.OK:
            raise RuntimeError("configs: device status not ok")
    finally:
        rd.purlin_destroy(h)
        torch.cuda.empty_cache()
    return out


SWEEP_RING = 96 << 20   # SNAC ring of the sweep: two 2 MiB-chunk channels, inside L2


def allreduce_sweep(rd, torch, dev, stream, peak):
    """AllReduce R=8 bf16 at 4 KiB..256 MiB per rank: zero staging, SNAC with
    its default chunk, and SNAC at every chunk of 64 KiB..2 MiB per rank."""
    import workloads
    h = rd.purlin_create(R, SWEEP_RING, dev.index)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(2 * l2 // 4 + 1, dtype=torch.float32, device=dev)
    out = []
    try:
        for nbytes in workloads.SWEEP_BYTES:
            n = nbytes // 2
            x = [torch.randn(n, device=dev).to(torch.bfloat16) for _ in range(R)]
            o = [torch.empty_like(t) for t in x]
            # inputs + outputs that fit in L2 stay there across repeated launches,
            # so their GB/s is not an HBM figure (it can exceed the HBM peak)
            row = {"bytes_per_rank": nbytes, "fits_in_l2": 2 * R * nbytes <= l2}
            runs = [("zs", rd.VARIANT_ZS, 0), ("snac", rd.VARIANT_STAGED, 0),
                    ("snac_y", rd.VARIANT_STAGED_Y, 0)] + \
                [(f"snac_chunk_{c >> 10}KiB", rd.VARIANT_STAGED, c) for c in workloads.SWEEP_CHUNKS] + \
                [(f"snac_y_chunk_{c >> 10}KiB", rd.VARIANT_STAGED_Y, c) for c in workloads.SWEEP_CHUNKS]
            for name, variant, chunk in runs:
                rd.purlin_set_policy(h, chunk, 0, 0, variant)
                fn = lambda: rd.purlin_all_reduce(h, x, o, n, "bf16", stream=stream)
                with torch.cuda.stream(stream):
                    for _ in range(3):
                        fn()
                torch.cuda.synchronize()
                host_us = _events_us(torch, stream, fn, 20 if nbytes >= (1 << 20) else 200)
                # below 16 MiB a Python caller's launch rate hides the device
                # time: take it from a CUDA graph of 50 launches instead
                graph_us = _graph_us(torch, stream, fn) if nbytes < (16 << 20) else None
                us = graph_us if graph_us is not None else host_us
                gbs = 2 * R * nbytes / (us / 1e6) / 1e9
                row[name] = {"us": round(us, 2), "gbs": round(gbs, 1),
                             "frac_of_peak": round(gbs / peak, 3),
                             "timing": "cuda graph" if graph_us is not None else "events",
                             "us_host_launched": round(host_us, 2)}
                if variant != rd.VARIANT_ZS:
                    info = rd.purlin_last_launch(h)
                    row[name]["chunk_bytes"] = info["chunk_bytes"]
                    row[name]["channels"] = info["grid"] // (3 if variant == rd.VARIANT_STAGED else 2)
            if row["fits_in_l2"]:
                # after both warm timings: the flush leaves L2 full of dirty lines
                for name, variant in (("zs", rd.VARIANT_ZS), ("snac", rd.VARIANT_STAGED)):
                    rd.purlin_set_policy(h, 0, 0, 0, variant)
                    fn = lambda: rd.purlin_all_reduce(h, x, o, n, "bf16", stream=stream)
                    cold = _cold_l2_us(torch, stream, fn, flush)
                    row[name]["us_cold_l2"] = round(cold, 2)
                    row[name]["gbs_cold_l2"] = round(2 * R * nbytes / (cold / 1e6) / 1e9, 1)
            for prefix in ("snac_chunk_", "snac_y_chunk_"):
                chunked = {k: v for k, v in row.items() if k.startswith(prefix)}
                row[prefix.replace("chunk_", "best_chunk")] = min(chunked, key=lambda k: chunked[k]["us"])
            out.append(row)
            del x, o
        if rd.purlin_query_status(h) != rd.OK:
            raise RuntimeError("allreduce sweep: device status not ok")
    finally:
        rd.purlin_destroy(h)
        torch.cuda.empty_cache()
    return out


def noalloc_allreduce(rd, torch, dev, stream, peak):
    """The AllReduce that allocates nothing (its staged kernel runs from a
    fixed static device array), R=8, bf16, 64 MiB and 4 KiB per rank."""
    out = []
    for nbytes in (64 << 20, 4096):
        n = nbytes // 2
        x = [torch.randn(n, device=dev).to(torch.bfloat16) for _ in range(R)]
        o = [torch.empty_like(t) for t in x]
        status = torch.zeros(1, dtype=torch.int32, device=dev)
        fn = lambda: rd.purlin_all_reduce_noalloc(x, o, n, "bf16", device_status=status,
                                                  stream=stream)
        with torch.cuda.stream(stream):
            for _ in range(3):
                fn()
        torch.cuda.synchronize()
        us = _events_us(torch, stream, fn, 10 if nbytes > 4096 else 200)
        if int(status.item()) != 0:
            raise RuntimeError("allocation-free AllReduce: device status not ok")
        gbs = 2 * R * nbytes / (us / 1e6) / 1e9
        out.append({"bytes_per_rank": nbytes, "us": round(us, 2), "gbs": round(gbs, 1),
                    "frac_of_peak": round(gbs / peak, 3)})
        del x, o
    return out


def allreduce_latency(rd, torch, dev, stream, variant):
    n = 2048   # 4 KiB of bf16 per rank
    h = rd.purlin_create(R, 0, dev.index)
    rd.purlin_set_policy(h, 0, 0, 0, variant)
    x = [torch.randn(n, device=dev).to(torch.bfloat16) for _ in range(R)]
    o = [torch.empty_like(t) for t in x]
    with torch.cuda.stream(stream):
        for _ in range(20):
            rd.purlin_all_reduce(h, x, o, n, "bf16", stream=stream)
    torch.cuda.synchronize()
    # one launch, device time between two events
    single = []
    for _ in range(200):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        rd.purlin_all_reduce(h, x, o, n, "bf16", stream=stream)
        b.record(stream)
        b.synchronize()
        single.append(a.elapsed_time(b) * 1e3)
    # 1000 launches back to back from the host: a prepared call (one C call
    # that plans and launches) and a plan (one launch of the kept plan)
    b2b = {}
    for name, call in (("prepared", rd.prepare(rd.purlin_all_reduce, h, x, o, n, "bf16",
                                                 stream=stream)),
                       ("plan", rd.plan(rd.purlin_all_reduce, h, x, o, n, "bf16", stream=stream))):
        for _ in range(20):
            call()
        torch.cuda.synchronize()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        t_host = time.perf_counter()
        a.record(stream)
        for _ in range(1000):
            call()
        b.record(stream)
        host_us = (time.perf_counter() - t_host) * 1e6 / 1000
        torch.cuda.synchronize()
        b2b[name] = (a.elapsed_time(b) * 1e3 / 1000, host_us)
    # CUDA graph of 100 launches, replayed 10 times
    graph_us = None
    try:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for _ in range(100):
                rd.purlin_all_reduce(h, x, o, n, "bf16")
        with torch.cuda.stream(stream):   # replay and events on one stream
            g.replay()
            torch.cuda.synchronize()
            a.record(stream)
            for _ in range(10):
                g.replay()
            b.record(stream)
        torch.cuda.synchronize()
        graph_us = a.elapsed_time(b) * 1e3 / 1000
    except Exception as e:  # capture is optional for the latency figure
        graph_us = f"capture failed: {e}"
    torch.cuda.synchronize()
    rd.purlin_destroy(h)
    return {"us_graph_per_launch": graph_us, "us_back_to_back": b2b["plan"][0],
            "us_back_to_back_prepared_call": b2b["prepared"][0],
            "host_us_per_call": {"plan": b2b["plan"][1], "prepared_call": b2b["prepared"][1]},
            "us_single_event_median": statistics.median(single), "R": R, "bytes_per_rank": 4096}


def c_caller_cost(rd):
    """Host time per call of the same AllReduce from a plain C99 caller
    (tests/c_abi/abi_check.c, built here against include/*.h and the library):
    planning alone, recording a plan, a direct call, a plan launch."""
    import shutil
    import tempfile
    from reduce_datapath_gb300 import _build
    gcc = shutil.which("gcc")
    if gcc is None:
        return "unavailable: no C compiler"
    cuda = os.path.dirname(os.path.dirname(_build.nvcc()))
    libdir = os.path.dirname(rd.LIB_PATH)
    with tempfile.TemporaryDirectory() as tmp:
        exe = os.path.join(tmp, "abi_check")
        cmd = [gcc, "-std=c99", "-O1", "-o", exe,
               os.path.join(ROOT, "tests", "c_abi", "abi_check.c"),
               "-I", os.path.join(ROOT, "include"), "-I", os.path.join(cuda, "include"),
               "-L", libdir, "-lpurlin", "-L", os.path.join(cuda, "lib64"), "-lcudart",
               "-Wl,-rpath," + libdir, "-Wl,-rpath," + os.path.join(cuda, "lib64")]
        b = subprocess.run(cmd, capture_output=True, text=True)
        if b.returncode != 0:
            return "unavailable: build failed: " + (b.stderr.strip().splitlines() or ["?"])[-1]
        r = subprocess.run([exe, "cost"], capture_output=True, text=True, timeout=120)
        if r.returncode != 0:
            return f"failed: exit {r.returncode}"
        return json.loads(r.stdout.strip().splitlines()[-1])


def bench_e2e(args, rd, torch, h, x, y, z, counts, stream):
    """End to end through host buffers: every step copies its inputs from pinned
    host memory, runs ReduceScatter then AllGather, and copies the gathered
    outputs back to pinned host memory.  Steps are pipelined over three streams
    (upload, compute, download) with double-buffered device inputs and outputs,
    so step i+1's upload overlaps step i's download (the host link is full
    duplex)."""
    dev = x[0].device
    xh = [torch.empty_like(t, device="cpu").pin_memory() for t in x]
    zh = [torch.empty_like(t, device="cpu").pin_memory() for t in z]
    for a, b in zip(xh, x):
        a.copy_(b)
    xs = [x, [torch.empty_like(t) for t in x]]
    zs = [z, [torch.empty_like(t) for t in z]]
    up = torch.cuda.Stream(device=dev)
    down = torch.cuda.Stream(device=dev)
    torch.cuda.synchronize()

    def run(K):
        rs_done = [None, None]
        d2h_done = [None, None]
        start = torch.cuda.Event(enable_timing=True)
        start.record(up)
        for i in range(K):
            b = i % 2
            with torch.cuda.stream(up):
                if rs_done[b] is not None:
                    up.wait_event(rs_done[b])       # step i-2 no longer reads xs[b]
                for a, src in zip(xs[b], xh):
                    a.copy_(src, non_blocking=True)
                h2d = torch.cuda.Event()
                h2d.record(up)
            stream.wait_event(h2d)
            if d2h_done[b] is not None:
                stream.wait_event(d2h_done[b])      # step i-2's outputs are downloaded
            rd.purlin_reduce_scatter(h, xs[b], y, counts, None, "bf16", stream=stream)
            rs_done[b] = torch.cuda.Event()
            rs_done[b].record(stream)
            rd.purlin_all_gather(h, y, zs[b], counts, None, "bf16", stream=stream)
            ag = torch.cuda.Event()
            ag.record(stream)
            with torch.cuda.stream(down):
                down.wait_event(ag)
                for dst, a in zip(zh, zs[b]):
                    dst.copy_(a, non_blocking=True)
                d2h_done[b] = torch.cuda.Event()
                d2h_done[b].record(down)
        end = torch.cuda.Event(enable_timing=True)
        up.wait_stream(down)
        up.wait_stream(stream)
        end.record(up)
        torch.cuda.synchronize()
        return start.elapsed_time(end)

    def link_gbs(upload, download, reps=3):
        """This machine's host link on the same pinned buffers: the step's uploads,
        its downloads, or both at once on their two streams."""
        nbytes = 0
        torch.cuda.synchronize()
        t = time.perf_counter()
        for _ in range(reps):
            if upload:
                with torch.cuda.stream(up):
                    for a, src in zip(xs[0], xh):
                        a.copy_(src, non_blocking=True)
                nbytes += sum(t_.numel() * t_.element_size() for t_ in xh)
            if download:
                with torch.cuda.stream(down):
                    for dst, a in zip(zh, zs[0]):
                        dst.copy_(a, non_blocking=True)
                nbytes += sum(t_.numel() * t_.element_size() for t_ in zh)
        torch.cuda.synchronize()
        return nbytes / (time.perf_counter() - t) / 1e9

    run(2)
    K = max(1, args.e2e_steps)
    ms = run(K) / K
    rs_b, ag_b = step_bytes()
    h2d = sum(t.numel() * t.element_size() for t in xh)
    d2h = sum(t.numel() * t.element_size() for t in zh)
    link = {"h2d_gbs": round(link_gbs(True, False), 1), "d2h_gbs": round(link_gbs(False, True), 1),
            "both_gbs": round(link_gbs(True, True), 1)}
    return {"value": (rs_b + ag_b) / (ms / 1e3) / 1e9, "unit": UNIT,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "ms_per_step": ms, "steps": K,
            # the step's transfers over the link's rate with both directions busy
            "link_frac": (h2d + d2h) / (ms / 1e3) / 1e9 / link["both_gbs"], "link": link,
            "note": "pinned host buffers; upload, compute and download pipelined across steps"}


def bench_only(args):
    """One collective of the bench workload's shape (R = --ranks virtual ranks),
    K times (for ncu runs)."""
    import torch

    import reduce_datapath_gb300 as rd
    import workloads

    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    rd.build()
    R = args.ranks
    n = args.bytes_per_rank // 2
    c = n // R - args.trim
    h = rd.purlin_create(R, args.staging, 0)
    variant = {"zs": rd.VARIANT_ZS, "staged": rd.VARIANT_STAGED,
               "staged_y": rd.VARIANT_STAGED_Y}[args.variant]
    rd.purlin_set_policy(h, args.chunk, args.depth, args.ctas, variant)
    rd.purlin_set_atom(h, {"auto": rd.ATOM_AUTO, "vector": rd.ATOM_VECTOR, "bulk": rd.ATOM_BULK,
                           "copy_engine": rd.ATOM_COPY_ENGINE}[args.atom])
    stream = torch.cuda.Stream(device=dev)
    if args.only == "rs":
        x = workloads.rank_buffers(WORKLOAD, R, n, "bf16", device=dev)
        y = [torch.empty(c, dtype=torch.bfloat16, device=dev) for _ in range(R)]
        fn = lambda: rd.purlin_reduce_scatter(h, x, y, [c] * R, None, "bf16", stream=stream)
        nbytes = (R + 1) * c * R * 2
    elif args.only == "ag":
        y = workloads.rank_buffers(WORKLOAD, R, c, "bf16", device=dev)
        z = [torch.empty(n, dtype=torch.bfloat16, device=dev) for _ in range(R)]
        fn = lambda: rd.purlin_all_gather(h, y, z, [c] * R, None, "bf16", stream=stream)
        nbytes = (R + 1) * c * R * 2
    elif args.only == "ar":
        x = workloads.rank_buffers(WORKLOAD, R, n, "bf16", device=dev)
        o = [torch.empty_like(t) for t in x]
        fn = lambda: rd.purlin_all_reduce(h, x, o, n, "bf16", stream=stream)
        nbytes = 2 * R * n * 2
    else:
        H = workloads.HIDDEN
        T = max(1, n // H)
        C = workloads.zipf_pair_counts(R, T, workloads.ZIPF_S, workloads.seed_for("moe_a2av_r8", 9))
        E = C * H
        E[E > 0] -= args.trim
        x = workloads.rank_buffers("moe_a2av_r8", R, T * H, "bf16", device=dev)
        o = [torch.empty(int(E[:, j].sum()), dtype=torch.bfloat16, device=dev) for j in range(R)]
        fn = lambda: rd.purlin_all_to_all_v(h, x, o, E, None, None, "bf16", stream=stream)
        nbytes = 2 * int(E.sum()) * 2
    with torch.cuda.stream(stream):
        for _ in range(max(1, args.warmup)):
            fn()
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    K = max(1, args.steps)
    a.record(stream)
    for _ in range(K):
        fn()
    b.record(stream)
    torch.cuda.synchronize()
    assert rd.purlin_query_status(h) == rd.OK
    info = rd.purlin_last_launch(h)
    rd.purlin_destroy(h)
    us = a.elapsed_time(b) * 1e3 / K
    print(json.dumps({"only": args.only, "variant": args.variant, "R": R,
                      "bytes_per_rank": args.bytes_per_rank, "trim": args.trim, "us": us,
                      "gbs": nbytes / (us / 1e6) / 1e9, "algorithmic_bytes": nbytes,
                      "launch": info}), flush=True)


def main():
    args = parse_args()
    if args.only:
        bench_only(args)
        return
    if args.impl == "reference":
        bench_reference(args)
    else:
        bench_purlin(args)


if __name__ == "__main__":
    main()
