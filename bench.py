#!/usr/bin/env python
"""Benchmark: one DWC training step (forward, backward data, backward filter) on GB300.

A step is one pass of the whole hot path over one batch of synthetic input: dwc_fwd,
dwc_bwd_data and dwc_bwd_filter on the same problem.  Default workload: fp32,
N=64, 56x56, C=128, 7x7 filter, stride 1, pad 3 (the ConvNeXt-stage shape), inputs drawn
as described in depthwise_convolution_nhwc_gb300/inputs.py.

Prints ONE JSON line (rank 0).  `value` is device-timed throughput with inputs resident in
HBM (CUDA events on the launching stream around each step, L2 flushed between steps by a
256 MiB write that is not timed, then an untimed device-side spin so that the step's launches
are all enqueued before its first event is reached); `e2e` is the same metric through the C ABI with the inputs
copied from pinned host memory and the outputs copied back inside the timed region.
`--impl reference` times the fp64 CPU oracle on bounded samples of the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "DWC fwd+bwd TFLOP/s and GB/s on 1 GB300, % of roofline, per filter size"
PASSES_ALL = ("fwd", "bwd_data", "bwd_filter")
# Device-side spin (untimed) between the L2 flush and each timed window: the host enqueues the
# timed launches while the GPU is still busy, so no host-side launch gap falls inside the
# window (a pass of a few microseconds is shorter than a call's host-side cost).
HOLD_CYCLES = 400_000


def hold_device(torch):
    torch.cuda._sleep(HOLD_CYCLES)
PASS_CODE = {"fwd": 0, "bwd_data": 1, "bwd_filter": 2, "fwd_bn_act": 3}
DTYPE_CODE = {"f32": 0, "bf16": 1, "f16": 2}
FAMILY = {0: "general", 1: "cuda-core", 2: "tensor-core", 3: "small-map", 4: "tensor-core"}
TENSOR_FAMILIES = (2, 4)   # tcgen05 or warp-level MMA kernels
# kernels per pass and family (the library's dwc_path tells which family serves a call)
KERNEL_NAMES = {
    ("fwd", 0): "general_fwd_kernel", ("bwd_data", 0): "general_bwd_data_kernel",
    ("bwd_filter", 0): "general_bwd_filter_kernel + reduce_slices_kernel",
    ("fwd", 1): "rows_kernel<flip=false>", ("bwd_data", 1): "rows_kernel<flip=true>",
    ("bwd_filter", 1): "fgrad_kernel + reduce_slices_kernel",
    ("fwd", 2): "tc_prep_kernel + tc_rows_kernel", ("bwd_data", 2): "tc_prep_kernel + tc_rows_kernel",
    ("bwd_filter", 2): "tc_stack_pm_kernel + tc_fgrad_kernel",
    ("bwd_filter", 4): "mma_fgrad_kernel + reduce_slices_kernel",
    ("fwd", 4): "mma_rows_kernel<flip=false>", ("bwd_data", 4): "mma_rows_kernel<flip=true>",
    ("fwd", 3): "small_rows_kernel", ("bwd_data", 3): "small_rows_kernel",
    ("bwd_filter", 3): "small_fgrad_kernel + reduce_slices_kernel",
    ("fwd_bn_act", 0): "general_fwd_bnact_kernel", ("fwd_bn_act", 1): "rows_kernel<act>",
}


def launches(dwc, case, pass_name):
    """Launches of this library's kernels in one call of the pass, as the library counts them
    (a filter gradient adds its slice sum; the tcgen05 path its preparation kernel)."""
    return dwc.kernel_launches(pass_name, case.N, case.H, case.W, case.C, case.FH, case.FW,
                               case.stride, case.pad, DTYPE_CODE[case.dtype])


def kernel_name(case, pass_name, family):
    """The kernel(s) serving a pass (the stride-2 backward data has its own kernel; 7x7 maps
    with 3 to 7 taps and "same" padding have their own small-map kernels)."""
    if case.stride == 2 and family == 1 and pass_name == "bwd_data":
        return "s2_bwd_data_kernel"
    if (pass_name == "fwd_bn_act" and family == 1 and case.stride == 1 and case.FH == case.FW == 7
            and case.C % 4 == 0 and case.W >= 28):
        return "bnact_apply_kernel + rows_kernel"
    if (family == 3 and case.stride == 1 and case.H == case.W == 7 and case.FH == case.FW
            and case.FH in (3, 5, 7) and case.pad == (case.FH - 1) // 2):
        if pass_name != "bwd_filter":
            return "tiny_rows_kernel"
        return "tiny_fgrad_cluster_kernel" if case.FH == 3 else "tiny_fgrad_kernel + reduce_slices_kernel"
    return KERNEL_NAMES[(pass_name, family)]


def kernel_family(dwc, case, pass_name):
    """0 general, 1 CUDA-core, 2 tcgen05 tensor-core, 3 small-map, 4 warp-level MMA
    (asked of the library itself)."""
    return dwc.path(pass_name, None, None, None, case.N, case.H, case.W, case.C, case.FH,
                    case.FW, case.stride, case.pad, DTYPE_CODE[case.dtype])


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default="f32_n64_56x56_c128_f7")
    ap.add_argument("--passes", default=",".join(PASSES_ALL))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--record-traffic", metavar="NCU_RAW_CSV",
                    help="write profiles/traffic.json from an ncu raw-page CSV and exit")
    ap.add_argument("--sweep", metavar="DTYPES",
                    help="time every pass of the filter sweep for these input dtypes "
                         "(comma separated, e.g. f32,bf16): one JSON line per sweep point")
    ap.add_argument("--sweep-set", choices=("stride1", "stride2", "large"), default="stride1",
                    help="filter sweep over the stage shapes at stride 1, the stride-2 "
                         "down-sampling shapes, or 41 and 51 taps over the stage shapes")
    ap.add_argument("--sweep-steps", type=int, default=20)
    ap.add_argument("--sweep-md", metavar="FILE", help="also write the sweep as a markdown table")
    ap.add_argument("--no-per-filter", action="store_true",
                    help="skip the per-filter-size table of the default line")
    ap.add_argument("--per-filter-steps", type=int, default=5)
    return ap.parse_args()


def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0")),
            int(os.environ.get("WORLD_SIZE", "1")))


def get_case(name):
    from depthwise_convolution_nhwc_gb300.inputs import (WORKLOADS, large_filter_cases,
                                                         stride2_cases, sweep_cases)
    if name in WORKLOADS:
        return WORKLOADS[name]
    for c in sweep_cases() + stride2_cases() + large_filter_cases():
        if c.name == name:
            return c
    raise SystemExit(f"unknown workload {name!r}")


# ---------------------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.lines = []
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self):
        return time.time()

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0, t1):
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        sm, mx, reasons, n = [], None, set(), 0
        for t, line in self.lines:
            if not (t0 - 0.15 <= t <= t1 + 0.15):
                continue
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            n += 1
            for nm, v in zip(names, parts[3:7]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": n}


# ---------------------------------------------------------------------------- oracle timing
def oracle_sample_run(case, passes, frac, host):
    """Run the oracle on a `frac` sample of every pass's outputs; returns (seconds, flops)."""
    import numpy as np

    import oracle
    rng = np.random.default_rng(12345)
    s, p = case.stride, case.pad
    x, w, dy = host
    flops = 0
    t0 = time.perf_counter()
    for name in passes:
        if name == "fwd":
            n_out = case.N * case.OH * case.OW * case.C
            k = max(1, int(round(frac * n_out)))
            oracle.fwd_at(x, w, rng.integers(0, n_out, k), s, p)
            flops += k * 2 * case.FH * case.FW
        elif name == "bwd_data":
            n_out = case.N * case.H * case.W * case.C
            k = max(1, int(round(frac * n_out)))
            oracle.bwd_data_at(dy, w, (case.H, case.W), rng.integers(0, n_out, k), s, p)
            flops += k * 2 * case.FH * case.FW * (case.N * case.OH * case.OW) // (case.N * case.H * case.W)
        else:
            n_out = case.FH * case.FW * case.C
            k = max(1, int(round(frac * n_out)))
            oracle.bwd_filter_at(x, dy, (case.FH, case.FW), rng.integers(0, n_out, k), s, p)
            flops += k * 2 * case.N * case.OH * case.OW
    return time.perf_counter() - t0, flops


def oracle_host_inputs(case):
    x, w, dy = case.x(), case.w(), case.dy()
    return tuple(t.double().numpy() for t in (x, w, dy))


def calibrate_fraction(case, passes, host, seconds):
    frac = 1e-5
    for _ in range(8):
        dt, _ = oracle_sample_run(case, passes, frac, host)
        if dt > 0.3 or frac >= 1.0:
            break
        frac = min(1.0, frac * 8)
    return min(1.0, frac * seconds / max(dt, 1e-6))


def cpu_baseline(case, passes, seconds):
    import oracle
    host = oracle_host_inputs(case)
    frac = calibrate_fraction(case, passes, host, seconds)
    dt, flops, reps = 0.0, 0, 0
    while reps == 0 or dt < 0.8 * seconds:  # a full step shorter than the budget repeats
        t, f = oracle_sample_run(case, passes, frac, host)
        dt, flops, reps = dt + t, flops + f, reps + 1
    what = (f"{frac:.3g} of the outputs of each pass ({'+'.join(passes)}) at random positions"
            if frac < 1 else f"every output of every pass ({'+'.join(passes)}), the full step")
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": oracle.max_threads(),
            "kind": "oracle",
            "sample": f"{what}, {reps} run(s), fp64 C oracle with OpenMP; {dt:.1f} s"}


def run_reference(args, case, passes):
    rank, _, world = dist_env()
    if rank != 0:
        return
    import oracle
    host = oracle_host_inputs(case)
    budget = 150.0
    per_step = budget / max(1, args.steps + args.warmup)
    frac = calibrate_fraction(case, passes, host, per_step)
    for _ in range(args.warmup):
        oracle_sample_run(case, passes, frac, host)
    tot_t, tot_f = 0.0, 0
    for _ in range(args.steps):
        dt, fl = oracle_sample_run(case, passes, frac, host)
        tot_t += dt
        tot_f += fl
    value = tot_f / tot_t / 1e12
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * tot_t / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_dict(case, passes),
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": oracle.max_threads(),
                             "kind": "oracle",
                             "sample": f"{frac:.3g} of the outputs of each pass per step"},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def config_dict(case, passes):
    return {"workload": f"{case.dtype} N={case.N} {case.H}x{case.W} C={case.C} "
                        f"{case.FH}x{case.FW} stride={case.stride} pad={case.pad}: "
                        + " + ".join(passes),
            "N": case.N, "H": case.H, "W": case.W, "C": case.C, "FH": case.FH, "FW": case.FW,
            "stride": case.stride, "pad": case.pad, "input_dtype": case.dtype,
            "output_dtype": "f32", "layout": "NHWC / FHxFWxC",
            "l2": "flushed between timed steps by an untimed 256 MiB write",
            "hold": f"untimed device spin of {HOLD_CYCLES} cycles before each timed window",
            "timing": "value / ms_per_step: the passes back to back, CUDA events at the step "
                      "boundaries; per_pass: a second set of as many steps with an event after "
                      "every pass",
            "inputs": f"{case.dist} draws, seed {case.seed}"}


def _sources_sha():
    """Hash of every kernel source file: a traffic entry counts only for the exact sources
    it was captured with."""
    import hashlib
    cdir = os.path.join("depthwise_convolution_nhwc_gb300", "csrc")
    rels = sorted(os.path.join(cdir, f) for f in os.listdir(os.path.join(ROOT, cdir))
                  if f.endswith((".cu", ".cuh", ".h")))
    h = hashlib.sha256()
    for rel in rels:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return rels, h.hexdigest()


def traffic_per_pass(raw_csv, passes=PASSES_ALL):
    """DRAM bytes (read + write) of each pass from `ncu -i <report> --page raw --csv` output
    holding the kernels of one step in launch order: a pass's kernels are told apart by name
    and, where the name does not say (the rotation of the small-map and 7x7-map row kernels,
    the tcgen05 main kernel), by the launch order."""
    import csv
    rows = list(csv.reader(open(raw_csv)))
    hdr, units, data = rows[0], rows[1], rows[2:]
    ix = {h: i for i, h in enumerate(hdr)}
    scale = {"byte": 1, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9}

    def dram(d):
        return sum(float(d[ix[k]]) * scale[units[ix[k]]]
                   for k in ("dram__bytes_read.sum", "dram__bytes_write.sum"))
    per = {"fwd": 0.0, "bwd_data": 0.0, "bwd_filter": 0.0}
    small_rows_seen = 0
    tc_flip = False
    for d in data:
        name = d[ix["Kernel Name"]]
        targs = name.split("<", 1)[1].split(",") if "<" in name else []
        if "small_rows_kernel" in name or "tiny_rows_kernel" in name:
            # rotation is a runtime argument: launch order
            which = [p for p in passes if p in ("fwd", "bwd_data")]
            per[which[min(small_rows_seen, len(which) - 1)]] += dram(d)
            small_rows_seen += 1
        elif "tc_prep_kernel" in name:   # <T, FLIP>; its main kernel follows
            tc_flip = targs[1].split(">")[0].strip() in ("1", "true")
            per["bwd_data" if tc_flip else "fwd"] += dram(d)
        elif "tc_rows_kernel" in name:   # the pass of the preparation launched before it
            per["bwd_data" if tc_flip else "fwd"] += dram(d)
        elif "mma_rows_kernel" in name:  # <T, FLIP>
            flip = targs[1].split(">")[0].strip()
            per["bwd_data" if flip in ("1", "true") else "fwd"] += dram(d)
        elif "rows_kernel" in name:      # <T, FH, FW, R, TM, MINB, FLIP, P>
            flip = targs[6].strip()
            per["bwd_data" if flip in ("1", "true") else "fwd"] += dram(d)
        elif ("fgrad" in name or "reduce_slices" in name or "tc_stack_pm_kernel" in name):
            per["bwd_filter"] += dram(d)
    return per


def record_traffic(raw_csv, workload, passes=PASSES_ALL):
    """Write profiles/traffic.json from `ncu -i <report> --page raw --csv` output that holds
    the kernels of one timed step (in launch order, of the passes given): DRAM bytes per
    launch of each pass, with a hash of the kernel sources so that the entry is ignored once
    a kernel changes."""
    case = get_case(workload)
    per = traffic_per_pass(raw_csv, passes)
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        tab = json.load(open(path))
    except (OSError, ValueError):
        tab = {}
    for p_, b in per.items():
        if b > 0:
            rels, sha = _sources_sha()
            tab[f"{p_}:{case.name}"] = {"bytes_per_launch": b, "sources": rels,
                                        "source_sha256": sha,
                                        "from": os.path.basename(raw_csv)}
    with open(path, "w") as f:
        json.dump(tab, f, indent=1, sort_keys=True)
    print(json.dumps(tab, indent=1, sort_keys=True))


def load_traffic(kernel_key):
    """ncu DRAM bytes per launch for a kernel, if captured against the current source."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            tab = json.load(f)
    except (OSError, ValueError):
        return None
    ent = tab.get(kernel_key)
    if not ent:
        return None
    rels, sha = _sources_sha()
    if rels != ent.get("sources") or sha != ent.get("source_sha256"):
        return None
    return ent.get("bytes_per_launch")


def measure_alu_peaks(dev):
    """Multiply-add rates of the CUDA cores measured in this run with the library's
    microbenchmark (dwc_fma_rate_probe): 8 CTAs of 256 threads per SM, 8 independent chains
    per thread, best of 3 launches timed with CUDA events.  TFLOP/s for each instruction kind
    (a multiply-add is 2 FLOPs); "ffma2" (packed fp32x2) is the fp32 peak the CUDA-core
    kernels are measured against."""
    import torch
    import depthwise_convolution_nhwc_gb300 as dwc
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    blocks, iters = 8 * sms, 1024
    out = torch.empty(blocks * 256, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()
    res = {}
    for kind, lanes in (("ffma", 1), ("ffma2", 2), ("hfma2", 2), ("bf16x2", 2)):
        dwc.fma_rate_probe(kind, blocks, iters, out)
        best = None
        for _ in range(3):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            dwc.fma_rate_probe(kind, blocks, iters, out)
            e1.record(stream)
            e1.synchronize()
            t = e0.elapsed_time(e1) * 1e-3
            best = t if best is None else min(best, t)
        res[kind] = 2.0 * blocks * 256 * iters * 8 * lanes / best / 1e12
    return {"tflops": res, "sms": sms, "launch": f"{blocks} CTAs x 256 threads x {iters} "
            "iterations x 8 chains, best of 3, CUDA events"}


def measure_link_rates(dev, nbytes):
    """Standalone pinned host-to-device and device-to-host copy rates (GB/s) of a buffer of
    `nbytes`, best of 3, each direction alone, CUDA events on one stream."""
    import torch
    n = max(1, nbytes // 4)
    h = torch.empty(n, dtype=torch.float32).pin_memory()
    d = torch.empty(n, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()
    rates = {}
    for name, fn in (("h2d_gbs", lambda: d.copy_(h, non_blocking=True)),
                     ("d2h_gbs", lambda: h.copy_(d, non_blocking=True))):
        fn()
        best = None
        for _ in range(3):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            e1.synchronize()
            t = e0.elapsed_time(e1) * 1e-3
            best = t if best is None else min(best, t)
        rates[name] = 4 * n / best / 1e9
    return rates


def gpu_local_cpus(dev):
    """CPUs the kernel lists as local to the GPU's PCI function (None if unknown)."""
    import torch
    p = torch.cuda.get_device_properties(dev)
    try:
        bus = f"{p.pci_domain_id:04x}:{p.pci_bus_id:02x}:{p.pci_device_id:02x}.0"
        txt = open(f"/sys/bus/pci/devices/{bus}/local_cpulist").read().strip()
    except (AttributeError, OSError):
        return None
    cpus = set()
    for part in txt.split(","):
        if "-" in part:
            lo, hi = part.split("-")
            cpus.update(range(int(lo), int(hi) + 1))
        elif part:
            cpus.add(int(part))
    allowed = os.sched_getaffinity(0)
    return sorted(cpus & allowed) or None


def per_filter_table(args, dev, peaks):
    """Every pass of every sweep filter size on the first stage shape (N=64, 56x56, C=128,
    pad (F-1)/2), fp32 and bf16 inputs: mean device time of --per-filter-steps launches
    (L2 flushed before each, 2 warm-up launches) and the roofline fraction of the pass.  x
    and dy are drawn once per dtype (they do not depend on F); W per filter size."""
    import torch
    import depthwise_convolution_nhwc_gb300 as dwc
    from depthwise_convolution_nhwc_gb300 import roofline as rl
    from depthwise_convolution_nhwc_gb300.inputs import SWEEP_FILTERS, SWEEP_SHAPES, Case
    N, H, W, C = SWEEP_SHAPES[0]
    stream = torch.cuda.current_stream()
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    ab = {0: "gen", 1: "cc", 2: "tc", 3: "sm", 4: "mma"}
    points = []
    for dt in ("f32", "bf16"):
        base = Case(N, H, W, C, 3, 3, 1, 1, dt, "normal", 900)
        x, dy = base.x().to(dev), base.dy().to(dev)
        y = torch.empty((N, H, W, C), device=dev, dtype=torch.float32)
        dx = torch.empty_like(y)
        for F in SWEEP_FILTERS:
            case = Case(N, H, W, C, F, F, 1, (F - 1) // 2, dt, "normal", 900)
            w = case.w().to(dev)
            dw = torch.empty((F, F, C), device=dev, dtype=torch.float32)
            ws = dwc.workspace(dwc.bwd_filter_workspace_size(x.shape, (F, F), 1, case.pad,
                                                             x.dtype), dev)
            run = {"fwd": lambda: dwc.fwd(x, w, 1, case.pad, out=y),
                   "bwd_data": lambda: dwc.bwd_data(dy, w, (H, W), 1, case.pad, out=dx),
                   "bwd_filter": lambda: dwc.bwd_filter(x, dy, (F, F), 1, case.pad, out=dw,
                                                        ws=ws)}
            pt = {"dtype": dt, "F": F}
            fams = []
            for name in PASSES_ALL:
                for _ in range(2):
                    run[name]()
                evs = []
                for k in range(args.per_filter_steps):
                    flush.fill_(float(k))
                    hold_device(torch)
                    e0 = torch.cuda.Event(enable_timing=True)
                    e1 = torch.cuda.Event(enable_timing=True)
                    e0.record(stream)
                    run[name]()
                    e1.record(stream)
                    evs.append((e0, e1))
                torch.cuda.synchronize()
                t = statistics.fmean(a.elapsed_time(b) for a, b in evs) * 1e-3
                fam = kernel_family(dwc, case, name)
                tr, bound = rl.roofline_time_s(case, name, peaks, tensor=fam in TENSOR_FAMILIES)
                pt[name] = {"us": round(t * 1e6, 2), "frac": round(tr / t, 3), "bound": bound,
                            "tflops": round(rl.nominal_flops(case) / t / 1e12, 2)}
                fams.append(ab[fam])
            pt["families"] = "/".join(fams)
            points.append(pt)
    if dwc.device_status() != 0:
        raise SystemExit("a kernel reported a timed-out wait in the per-filter table")
    return {"workload": f"N={N} {H}x{W} C={C}, F x F filters, pad (F-1)/2, stride 1",
            "timing": f"mean of {args.per_filter_steps} launches per pass, L2 flushed before "
                      "each (then an untimed device spin), CUDA events",
            "frac": "roofline fraction of the pass (hbm: compulsory bytes at the measured HBM "
                    "copy rate; alu: valid FLOPs at the measured fp32x2 FMA rate; tensor: "
                    "valid FLOPs at the measured bf16 peak)",
            "families": "fwd/bwd_data/bwd_filter kernel family: cc CUDA-core, tc tensor-core "
                        "(tcgen05), mma warp-level MMA, sm small-map, gen general",
            "points": points}


def run_e2e(args, case, passes, x, w, dy, ws, world, flops_step):
    """Same step through the public API with every step's inputs copied from pinned host
    memory and its outputs copied back, inside the timed region.  Steps are pipelined over
    two device buffer sets and three streams (host-to-device copies, kernels, device-to-host
    copies), ordered by events, so that one step's copies overlap another step's kernels;
    every step still moves all of its own bytes."""
    import torch
    import depthwise_convolution_nhwc_gb300 as dwc
    dev = x.device
    # pinned buffers on the GPU's own NUMA node: allocate (first touch) from its local CPUs
    old_aff = os.sched_getaffinity(0)
    local = gpu_local_cpus(dev)
    if local:
        os.sched_setaffinity(0, local)
    try:
        out = _run_e2e_pinned(args, case, passes, x, w, dy, ws, world, flops_step)
    finally:
        os.sched_setaffinity(0, old_aff)
    out[-1]["host_cpus"] = (f"{len(local)} CPUs local to the GPU" if local
                            else "process affinity unchanged (GPU-local CPUs unknown)")
    return out


def _run_e2e_pinned(args, case, passes, x, w, dy, ws, world, flops_step):
    import torch
    import depthwise_convolution_nhwc_gb300 as dwc
    dev = x.device
    hx, hw, hdy = (t.pin_memory() for t in (case.x(), case.w(), case.dy()))
    shapes = {"fwd": (case.N, case.OH, case.OW, case.C), "bwd_data": (case.N, case.H, case.W, case.C),
              "bwd_filter": (case.FH, case.FW, case.C)}
    need = {"x": "fwd" in passes or "bwd_filter" in passes, "w": True,
            "dy": "bwd_data" in passes or "bwd_filter" in passes}
    sets = []
    for _ in range(2):
        sets.append({"x": torch.empty_like(x), "w": torch.empty_like(w), "dy": torch.empty_like(dy),
                     "out": {n: torch.empty(shapes[n], device=dev, dtype=torch.float32) for n in passes},
                     "host": {n: torch.empty(shapes[n], dtype=torch.float32).pin_memory() for n in passes}})
    h2d = sum(t.numel() * t.element_size() for t, nm in ((hx, "x"), (hw, "w"), (hdy, "dy")) if need[nm])
    d2h = sum(sets[0]["host"][n].numel() * 4 for n in passes)
    s_in, s_cmp, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev = lambda: torch.cuda.Event()
    in_ready, cmp_done, out_done = [ev(), ev()], [ev(), ev()], [ev(), ev()]
    used = [False, False]

    def e2e_step(k):
        b = k % 2
        S = sets[b]
        with torch.cuda.stream(s_in):
            if used[b]:
                s_in.wait_event(cmp_done[b])  # the kernels of step k-2 have read this set
            for nm, h in (("x", hx), ("w", hw), ("dy", hdy)):
                if need[nm]:
                    S[nm].copy_(h, non_blocking=True)
            in_ready[b].record(s_in)
        s_cmp.wait_event(in_ready[b])
        if used[b]:
            s_cmp.wait_event(out_done[b])     # step k-2's outputs have left this set
        for name in passes:
            o = S["out"][name]
            if name == "fwd":
                dwc.fwd(S["x"], S["w"], case.stride, case.pad, out=o, stream=s_cmp)
            elif name == "bwd_data":
                dwc.bwd_data(S["dy"], S["w"], (case.H, case.W), case.stride, case.pad, out=o, stream=s_cmp)
            else:
                dwc.bwd_filter(S["x"], S["dy"], (case.FH, case.FW), case.stride, case.pad, out=o,
                               ws=ws, stream=s_cmp)
        cmp_done[b].record(s_cmp)
        s_out.wait_event(cmp_done[b])
        with torch.cuda.stream(s_out):
            for name in passes:
                S["host"][name].copy_(S["out"][name], non_blocking=True)
            out_done[b].record(s_out)
        used[b] = True

    for k in range(4):
        e2e_step(k)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    s_cmp.wait_event(e0)
    s_out.wait_event(e0)
    for k in range(args.e2e_steps):
        e2e_step(k)
    s_out.wait_stream(s_in)
    s_out.wait_stream(s_cmp)
    e1.record(s_out)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1)
    if world > 1:
        t = torch.tensor([e2e_ms], device=dev, dtype=torch.float64)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        e2e_ms = float(t.item())
    e2e_value = world * args.e2e_steps * flops_step / (e2e_ms * 1e-3) / 1e12
    link = measure_link_rates(dev, max(h2d, d2h))
    # the copies of one step cannot take less than the slower direction alone
    link["copy_bound_ms_per_step"] = max(h2d / (link["h2d_gbs"] * 1e9),
                                         d2h / (link["d2h_gbs"] * 1e9)) * 1e3
    return e2e_value, h2d, d2h, e2e_ms / args.e2e_steps, link


def roofline_entry(rl, case, pass_name, family, seconds, peaks):
    """Roofline of one pass: achieved algorithmic bytes or FLOPs per launch over the
    measured time, against the peak of the resource that bounds it."""
    _, bound = rl.roofline_time_s(case, pass_name, peaks, tensor=family in TENSOR_FAMILIES)
    if bound == "hbm":
        achieved = rl.compulsory_bytes(case, pass_name) / seconds / 1e9
        peak, unit = peaks["hbm_gbs"], "GB/s"
        src = ("measured HBM copy (MEASURED_PEAKS.json)" if peaks["source"] == "measured"
               else "fallback HBM figure")
    elif bound == "tensor":
        achieved = rl.valid_flops(case) / seconds / 1e12
        peak, unit = peaks["bf16_tflops"], "TFLOP/s"
        src = ("measured bf16 cuBLAS burst (MEASURED_PEAKS.json)" if peaks["source"] == "measured"
               else "fallback bf16 figure")
    else:
        achieved = rl.valid_flops(case) / seconds / 1e12
        peak, unit = peaks["fp32_tflops"], "TFLOP/s"
        src = ("measured fp32x2 FMA rate (dwc_fma_rate_probe, all SMs, this run)"
               if peaks.get("fp32_source") == "measured"
               else "fp32 FMA peak derived: SMs x 128 lanes x 2 x 2070 MHz")
    return {"bound": bound, "achieved": achieved, "peak": peak, "unit": unit,
            "frac": achieved / peak, "traffic": None,
            "kernel": kernel_name(case, pass_name, family), "pass": pass_name,
            "peak_source": src}


def run_sweep(args):
    """Every pass of every sweep point: mean device time over --sweep-steps launches, L2
    flushed before each, one JSON line per point.  Filters of 3, 5 and 7 taps also time the
    fused BN + ReLU + forward pass."""
    import torch
    import depthwise_convolution_nhwc_gb300 as dwc
    from depthwise_convolution_nhwc_gb300 import roofline as rl
    from depthwise_convolution_nhwc_gb300.inputs import (large_filter_cases, stride2_cases,
                                                         sweep_cases)

    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    dwc.load_library()
    stream = torch.cuda.current_stream()
    alu = measure_alu_peaks(dev)
    peaks = rl.load_peaks(fp32_tflops=alu["tflops"]["ffma2"])
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    rows = []
    cases = {"stride1": sweep_cases, "stride2": stride2_cases,
             "large": large_filter_cases}[args.sweep_set](tuple(args.sweep.split(",")))
    for case in cases:
        s = case.stride
        x, w, dy = (t.to(dev) for t in (case.x(), case.w(), case.dy()))
        y = torch.empty((case.N, case.OH, case.OW, case.C), device=dev, dtype=torch.float32)
        dx = torch.empty((case.N, case.H, case.W, case.C), device=dev, dtype=torch.float32)
        dw = torch.empty((case.FH, case.FW, case.C), device=dev, dtype=torch.float32)
        ws = dwc.workspace(dwc.bwd_filter_workspace_size(x.shape, (case.FH, case.FW), s,
                                                         case.pad, x.dtype), dev)
        bn = [t.to(dev) for t in case.bn()]
        run = {"fwd": lambda: dwc.fwd(x, w, s, case.pad, out=y),
               "bwd_data": lambda: dwc.bwd_data(dy, w, (case.H, case.W), s, case.pad, out=dx),
               "bwd_filter": lambda: dwc.bwd_filter(x, dy, (case.FH, case.FW), s, case.pad,
                                                    out=dw, ws=ws),
               "fwd_bn_act": lambda: dwc.fwd_bn_act(x, w, *bn, 1e-5, "relu", s, case.pad, out=y)}
        line = {"sweep": case.name, "dtype": case.dtype, "N": case.N, "H": case.H, "W": case.W,
                "C": case.C, "F": case.FH, "stride": s}
        names = PASSES_ALL + (("fwd_bn_act",) if case.FH <= 7 else ())
        for name in names:
            for _ in range(3):
                run[name]()
            evs = []
            for k in range(args.sweep_steps):
                flush.fill_(float(k))
                hold_device(torch)
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                run[name]()
                e1.record(stream)
                evs.append((e0, e1))
            torch.cuda.synchronize()
            t = statistics.fmean(a.elapsed_time(b) for a, b in evs) * 1e-3
            fam = kernel_family(dwc, case, name)
            roof = roofline_entry(rl, case, name, fam, t, peaks)
            line[name] = {"us": t * 1e6, "tflops": rl.nominal_flops(case) / t / 1e12,
                          "kernel": kernel_name(case, name, fam),
                          "gbs": rl.compulsory_bytes(case, name) / t / 1e9,
                          "bound": roof["bound"], "roofline_frac": roof["frac"],
                          "family": FAMILY[fam]}
        if dwc.device_status() != 0:
            raise SystemExit(f"a kernel reported a timed-out wait in {case.name}")
        rows.append(line)
        print(json.dumps(line), flush=True)
    if args.sweep_md:
        write_sweep_md(args, rows)


def write_sweep_md(args, rows):
    cmd = " ".join(["python", "bench.py"] + sys.argv[1:])
    out = [f"# Filter sweep, every pass, one GB300\n",
           f"Command: `{cmd}`\n",
           f"Mean device time of {args.sweep_steps} launches per pass (CUDA events on the "
           "launching stream, 256 MiB L2 flush and an untimed device spin before each launch, "
           "3 warm-up launches). "
           "TFLOP/s are nominal (2·N·OH·OW·C·FH·FW); roofline fraction against the bound "
           "named (hbm: compulsory bytes at the measured HBM copy rate; alu: valid FLOPs at "
           "the fp32x2 FMA rate measured in the same run; tensor: valid FLOPs at the measured "
           "bf16 peak). "
           "Kernel family: cc = CUDA-core row / filter-gradient kernels, tc = tensor-core, "
           "sm = small-map kernels.  BN+ReLU: the fused batch-norm + ReLU + forward pass "
           "(filters up to 7 taps).\n",
           "| dtype | N×H×W×C | F | s | fwd µs | fwd TF/s | fwd roof | bwd_data µs | bwd_data roof "
           "| bwd_filter µs | bwd_filter TF/s | bwd_filter roof | families | BN+ReLU+fwd µs |",
           "|---|---|---|---|---|---|---|---|---|---|---|---|---|---|"]
    ab = {"cuda-core": "cc", "tensor-core": "tc", "general": "gen", "small-map": "sm"}
    for r in rows:
        f, d, g = r["fwd"], r["bwd_data"], r["bwd_filter"]
        fz = f"{r['fwd_bn_act']['us']:.1f}" if "fwd_bn_act" in r else "–"
        out.append(f"| {r['dtype']} | {r['N']}×{r['H']}×{r['W']}×{r['C']} | {r['F']} | {r['stride']} "
                   f"| {f['us']:.1f} | {f['tflops']:.1f} | {f['roofline_frac']:.2f} {f['bound']} "
                   f"| {d['us']:.1f} | {d['roofline_frac']:.2f} {d['bound']} "
                   f"| {g['us']:.1f} | {g['tflops']:.1f} | {g['roofline_frac']:.2f} {g['bound']} "
                   f"| {ab[f['family']]}/{ab[d['family']]}/{ab[g['family']]} | {fz} |")
    with open(args.sweep_md, "w") as fh:
        fh.write("\n".join(out) + "\n")


def run_ours(args, case, passes):
    import torch
    import depthwise_convolution_nhwc_gb300 as dwc
    from depthwise_convolution_nhwc_gb300 import roofline as rl

    rank, local_rank, world = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())
    dwc.load_library()
    stream = torch.cuda.current_stream()
    alu = measure_alu_peaks(dev)
    peaks = rl.load_peaks(fp32_tflops=alu["tflops"]["ffma2"])

    x, w, dy = (t.to(dev) for t in (case.x(), case.w(), case.dy()))
    y = torch.empty((case.N, case.OH, case.OW, case.C), device=dev, dtype=torch.float32)
    dx = torch.empty((case.N, case.H, case.W, case.C), device=dev, dtype=torch.float32)
    dw = torch.empty((case.FH, case.FW, case.C), device=dev, dtype=torch.float32)
    ws = dwc.workspace(dwc.bwd_filter_workspace_size(x.shape, (case.FH, case.FW), case.stride,
                                                     case.pad, x.dtype), dev)
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)

    def run_pass(name, xx, ww, dyy):
        if name == "fwd":
            dwc.fwd(xx, ww, case.stride, case.pad, out=y)
        elif name == "bwd_data":
            dwc.bwd_data(dyy, ww, (case.H, case.W), case.stride, case.pad, out=dx)
        else:
            dwc.bwd_filter(xx, dyy, (case.FH, case.FW), case.stride, case.pad, out=dw, ws=ws)

    for _ in range(args.warmup):
        for name in passes:
            run_pass(name, x, w, dy)
    torch.cuda.synchronize()
    if dwc.device_status() != 0:
        raise SystemExit("a kernel reported a timed-out wait during warm-up")

    # The timed steps: the passes back to back, as a caller runs them (events only at the
    # step boundaries, so nothing is enqueued between the passes' kernels).  Then the same
    # number of steps with an event after every pass, for the per-pass split.
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    evp = [[torch.cuda.Event(enable_timing=True) for _ in range(len(passes) + 1)]
           for _ in range(args.steps)]
    with ClockSampler(torch.cuda.current_device()) as clk:
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        t_wall0 = time.time()
        for k in range(args.steps):
            flush.fill_(float(k))
            hold_device(torch)
            ev[k][0].record(stream)
            for name in passes:
                run_pass(name, x, w, dy)
            ev[k][1].record(stream)
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
        t_wall1 = time.time()
        for k in range(args.steps):
            flush.fill_(float(k))
            hold_device(torch)
            evp[k][0].record(stream)
            for j, name in enumerate(passes):
                run_pass(name, x, w, dy)
                evp[k][j + 1].record(stream)
        torch.cuda.synchronize()
    clocks = clk.summary(t_wall0, t_wall1)
    if dwc.device_status() != 0:
        raise SystemExit("a kernel reported a timed-out wait in the timed region")

    per_pass = {name: [] for name in passes}
    step_ms = []
    for k in range(args.steps):
        step_ms.append(ev[k][0].elapsed_time(ev[k][1]))
        for j, name in enumerate(passes):
            per_pass[name].append(evp[k][j].elapsed_time(evp[k][j + 1]))
    total_ms = sum(step_ms)
    if world > 1:
        t = torch.tensor([total_ms], device=dev, dtype=torch.float64)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        total_ms = float(t.item())

    flops_step = rl.nominal_flops(case) * len(passes)
    value = world * args.steps * flops_step / (total_ms * 1e-3) / 1e12

    e2e_value, h2d, d2h, e2e_step_ms, link = None, 0, 0, None, None
    if args.e2e_steps > 0:
        e2e_value, h2d, d2h, e2e_step_ms, link = run_e2e(args, case, passes, x, w, dy, ws, world,
                                                         flops_step)

    if rank != 0:
        if world > 1:
            torch.distributed.destroy_process_group()
        return

    # --- roofline of the dominant kernel ----------------------------------------------
    fam = {n: kernel_family(dwc, case, n) for n in passes}
    mean_ms = {n: statistics.fmean(v) for n, v in per_pass.items()}
    dom = max(mean_ms, key=mean_ms.get)
    roof = roofline_entry(rl, case, dom, fam[dom], mean_ms[dom] * 1e-3, peaks)
    roof["traffic"] = load_traffic(f"{dom}:{case.name or 'default'}")
    passes_out = {}
    for n in passes:
        t = mean_ms[n] * 1e-3
        tr, b = rl.roofline_time_s(case, n, peaks, tensor=fam[n] in TENSOR_FAMILIES)
        passes_out[n] = {"ms": mean_ms[n], "ms_median": statistics.median(per_pass[n]),
                         "kernel": kernel_name(case, n, fam[n]),
                         "tflops_nominal": rl.nominal_flops(case) / t / 1e12,
                         "tflops_valid": rl.valid_flops(case) / t / 1e12,
                         "gbs": rl.compulsory_bytes(case, n) / t / 1e9,
                         "roofline_frac": tr / t, "roofline_bound": b}
    line = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": total_ms / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": case.dtype,
            "data": "synthetic", "config": config_dict(case, passes),
            "gbs": sum(rl.compulsory_bytes(case, n) for n in passes) * args.steps * world
                   / (total_ms * 1e-3) / 1e9,
            "roofline": roof, "per_pass": passes_out,
            "e2e": ({"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                     "d2h_bytes_per_step": d2h, "steps": args.e2e_steps, "ms_per_step": e2e_step_ms,
                     "pipelining": "two buffer sets; host-to-device copies, kernels and "
                                   "device-to-host copies on three streams ordered by events",
                     "link": link}
                    if e2e_value is not None else None),
            "alu_peaks": alu,
            "gpu_launches": args.steps * sum(launches(dwc, case, n) for n in passes),
            "kernels": {n: kernel_name(case, n, fam[n]) for n in passes},
            "clocks": clocks}
    if not args.no_per_filter and world == 1:
        line["per_filter"] = per_filter_table(args, dev, peaks)
    if not args.no_cpu_baseline and world == 1:
        line["cpu_baseline"] = cpu_baseline(case, passes, args.cpu_seconds)
    print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def main():
    args = parse_args()
    if args.record_traffic:
        record_traffic(args.record_traffic, args.workload,
                       tuple(p for p in args.passes.split(",") if p))
        return
    if args.sweep:
        run_sweep(args)
        return
    case = get_case(args.workload)
    passes = tuple(p for p in args.passes.split(",") if p)
    for p in passes:
        if p not in PASSES_ALL:
            raise SystemExit(f"unknown pass {p}")
    if args.impl == "reference":
        run_reference(args, case, passes)
    else:
        run_ours(args, case, passes)


if __name__ == "__main__":
    main()
