#!/usr/bin/env python
"""Benchmark of the S6 selective-scan forward (libsscan) on B300.

One step = one selective-scan forward over the whole workload (softplus, discretisation,
recurrence, readout, skip, gate, h_last): the library's kernels for one sscan_fwd call.

Headline workload (default): the largest single-GPU workload, the long sequence, bf16 io with
fp32 state, batch 1, L 1,048,576, D 1536, N 16, h_last returned. The same JSON line carries, under
"configs", the other full-size workloads with L >= 2048 (fp32 b8 L2048 D1536; bf16 b16 L4096
D2048; bf16 b4 L8192 D5120), each timed over a region of at least 200 ms, with its own roofline.

Rooflines. The HBM bound divides the algorithmic bytes (inputs read once, outputs written once) by
the measured copy bandwidth (MEASURED_PEAKS.json). The compute ("alu") bound counts, per state
update, one SFU exponential and four FP32-pipe operations; its denominators are measured live, at
the start of the run, by the library's own issue-rate probes (libsscan_peaks: ex2.approx and FFMA
throughput per SM and clock), times the SM count and the maximum SM clock. The bound of a workload
is the slower of the two.

Prints ONE JSON line (rank 0). Under torchrun with N ranks every rank runs its own full replica
of the workload on its own GPU (the batch rows and channels are independent; no data-path
collective), the timed region is bracketed by a barrier and a device synchronize, and the
slowest rank's time is used: value = N * units / max_time ("scaling": "weak").

--impl reference times the fp64 CPU oracle (the correctness reference) on a bounded sample of
the same workload per step, on this machine's host cores.

--mode peaks prints the issue-rate probes' results (per SM and clock, and per second at the
maximum clock) as one JSON line.

--mode conv times the causal depthwise Conv1d + SiLU (sscan_conv1d_silu) over the workload's
(batch, L, dim) in its io type; the roofline is HBM on the input read once, the output written
once and the tiles' halos.

--mode bwd times the backward pass (sscan_bwd: checkpoints, adjoint sweep, reductions) on the
workload with random dy and dh_last; its compute roofline counts the FP32-pipe operations of a
recompute plus an adjoint step per update (16) against the measured FFMA rate.

--mode decode times the single-step recurrence (sscan_step) on the workload's batch, channels
and state size instead: one step per token, the state read and written in place, as K
back-to-back launches and as CUDA-graph replays of 64 captured steps; the roofline is HBM on the
state plus the step's inputs and outputs.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "selective-scan fwd GB/s and (B·L·D·N)/s on 1 B300; % of HBM/SFU roofline"
UNIT = "(B*L*D*N)/s"
FALLBACK_HBM_GBS = 6400.0
FP32_OPS_PER_UPDATE = 4  # dt*A, dt*u*B, the state FMA, the readout FMA
MIN_REGION_MS = 200.0    # each extra workload is timed over at least this much device time
EXTRA_WORKLOADS = ("fp32", "bf16", "wide")
L2_BYTES = 126 * 2**20


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["lib", "reference"], default="lib")
    ap.add_argument("--workload", default="long")
    ap.add_argument("--L", type=int, default=0, help="override the workload's L (profiling)")
    ap.add_argument("--dim", type=int, default=0,
                    help="override the workload's channel count D (profiling)")
    ap.add_argument("--no-configs", action="store_true",
                    help="time only the headline workload")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--mode", choices=["scan", "decode", "conv", "bwd", "peaks"], default="scan")
    ap.add_argument("--conv-width", type=int, default=4)
    return ap.parse_args()


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d.get("sm_max_mhz", 2032.0)), "measured"
    return FALLBACK_HBM_GBS, 2032.0, "fallback"


# The sources the forward scan kernel and its launcher are compiled from (the backward and
# convolution kernels live in files of their own and do not change it).
SCAN_SOURCES = ("sscan_kernels.cu", "sscan_device.cuh", "sscan_internal.h")


def kernel_source_sha() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "selective_state_space_158_b300", "csrc")
    for fn in SCAN_SOURCES:
        with open(os.path.join(csrc, fn), "rb") as f:
            h.update(fn.encode() + f.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload_key: str):
    """DRAM bytes per launch from a committed ncu capture, if taken on the current kernel
    source; else None."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f).get(workload_key)
    if not d or d.get("source_sha") != kernel_source_sha():
        return None
    return float(d["dram_bytes_per_launch"])


class ClockSampler:
    """Samples SM clock and clock-event (throttle) reasons while the timed region runs, with
    NVML if the Python bindings import, else by streaming `nvidia-smi -lms`."""

    REASONS = {
        "sw_power_cap": 0x4, "hw_slowdown": 0x8, "sync_boost": 0x10,
        "sw_thermal_slowdown": 0x20, "hw_thermal_slowdown": 0x40, "hw_power_brake": 0x80,
    }

    def __init__(self, index: int, period_ms: int = 20):
        self.index = index
        self.period_ms = period_ms
        self.samples = []
        self.reasons = set()
        self.max_mhz = None
        self.source = None
        self.err = None
        self._stop = threading.Event()
        try:
            import pynvml
            pynvml.nvmlInit()
            self.nv = pynvml
            self.h = pynvml.nvmlDeviceGetHandleByIndex(index)
            self.max_mhz = pynvml.nvmlDeviceGetMaxClockInfo(self.h, pynvml.NVML_CLOCK_SM)
            self.source = "nvml"
        except Exception as e:
            self.err = repr(e)
            self.source = "nvidia-smi"

    def _run_nvml(self):
        while not self._stop.is_set():
            try:
                self.samples.append(self.nv.nvmlDeviceGetClockInfo(self.h, self.nv.NVML_CLOCK_SM))
                r = self.nv.nvmlDeviceGetCurrentClocksEventReasons(self.h)
                for name, bit in self.REASONS.items():
                    if r & bit:
                        self.reasons.add(name)
            except Exception:
                pass
            time.sleep(self.period_ms / 1e3)

    def _run_smi(self):
        import subprocess
        q = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
             "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
             "clocks_event_reasons.sw_power_cap")
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={q}", "--format=csv,noheader,nounits",
                 "-i", str(self.index), f"-lms={self.period_ms}"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception as e:
            self.err = repr(e)
            return
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 6:
                continue
            try:
                self.samples.append(float(parts[0]))
                self.max_mhz = float(parts[1])
            except ValueError:
                continue
            for n, v in zip(names, parts[2:6]):
                if v.lower() == "active":
                    self.reasons.add(n)

    def __enter__(self):
        target = self._run_nvml if self.source == "nvml" else self._run_smi
        self.t = threading.Thread(target=target, daemon=True)
        self.t.start()
        if self.source == "nvidia-smi":
            time.sleep(0.3)  # let nvidia-smi start before the timed region
        return self

    def __exit__(self, *a):
        self._stop.set()
        if getattr(self, "proc", None) is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        self.t.join(timeout=5)

    def summary(self):
        out = {"sm_mhz": statistics.median(self.samples) if self.samples else None,
               "sm_max_mhz": self.max_mhz, "reasons": sorted(self.reasons),
               "samples": len(self.samples), "source": self.source}
        if not self.samples and self.err:
            out["note"] = f"no clock samples: {self.err}"
        return out

    def rejected(self):
        bad = {"hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"}
        if self.reasons & bad:
            return True
        s = self.summary()
        if s["sm_mhz"] and s["sm_max_mhz"] and s["sm_mhz"] < 0.6 * s["sm_max_mhz"] and \
                not (self.reasons - {"sync_boost"}):
            return True
        return False


def dist_setup(n_gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(x: float, world: int, device=None) -> float:
    """The largest of every rank's x (all-reduce MAX over the default process group); x itself
    for a single process. The bench takes the slowest rank's time."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist

    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank: float, world: int, seconds: float) -> float:
    """Units all ranks processed per second of the slowest rank (weak scaling: every rank runs a
    full replica)."""
    return world * units_per_rank / seconds


def cpu_baseline(w, x, seconds: float):
    """The oracle, as it stands, on a bounded sample of the workload: whole batch rows (or the
    first k channels of row 0) over the full sequence, sized for about `seconds` of wall time."""
    import numpy as np
    import torch

    import oracle

    cores = os.cpu_count() or 1

    def io(t):
        if t is None:
            return None
        t = t.cpu().contiguous()
        return t.numpy() if t.dtype == torch.float32 else t.view(torch.int16).numpy().view(np.uint16)

    def run(rows, k):
        sl = lambda name: None if x.get(name) is None else x[name][0:rows, :, :k]  # noqa: E731
        args = (io(sl("u")), io(sl("delta")), x["A"][:k].cpu().numpy(), io(x["B"][0:rows]),
                io(x["C"][0:rows]), None if x.get("D") is None else x["D"][:k].cpu().numpy(),
                io(sl("z")),
                None if x.get("delta_bias") is None else x["delta_bias"][:k].cpu().numpy())
        t0 = time.perf_counter()
        oracle.fwd(*args, io=w.io, threads=cores)
        return time.perf_counter() - t0

    k = min(w.dim, max(4 * cores, 32))
    t = run(1, k)
    target = w.L * k * w.N * seconds / max(t, 1e-3)  # updates that fill the time budget
    row_units = w.L * w.dim * w.N
    if target >= row_units:
        rows, k = int(min(w.batch, max(1, target // row_units))), w.dim
    else:
        rows, k = 1, int(min(w.dim, max(k, target // (w.L * w.N))))
    t2 = run(rows, k)
    units = rows * w.L * k * w.N
    return {"value": units / t2, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"batch rows 0..{rows - 1} of {w.batch}, channels 0..{k - 1} of {w.dim}, "
                      f"full L={w.L}, N={w.N}: {units:.3g} updates in {t2:.2f} s "
                      f"(fp64 C loop, {cores} threads)"}


def run_reference(args, w):
    """--impl reference: the oracle timed per step on a bounded sample (rank 0 only)."""
    world, rank, local = dist_setup(args.gpus)
    if rank != 0:
        return
    import torch

    import oracle
    from selective_state_space_158_b300.inputs import make_inputs

    oracle.build()
    # The sample's inputs come from the same seeded recipe, drawn for one batch row and a
    # channel slice on the CPU (the oracle needs no device).
    cores = os.cpu_count() or 1
    budget = 120.0  # seconds for the whole run
    per_step = budget / max(1, args.steps + args.warmup)
    k = 1
    sub = w.replace(batch=1, dim=max(1, min(w.dim, 64)))
    x = make_inputs(sub, device="cpu")
    import numpy as np

    def io(t):
        if t is None:
            return None
        t = t.contiguous()
        return t.numpy() if t.dtype == torch.float32 else t.view(torch.int16).numpy().view(np.uint16)

    def step(k):
        sl = lambda n: None if x.get(n) is None else x[n][:, :, :k]  # noqa: E731
        oracle.fwd(io(sl("u")), io(sl("delta")), x["A"][:k].numpy(), io(x["B"]), io(x["C"]),
                   None if x.get("D") is None else x["D"][:k].numpy(), io(sl("z")),
                   None if x.get("delta_bias") is None else x["delta_bias"][:k].numpy(),
                   io=w.io, threads=cores)

    t0 = time.perf_counter()
    step(1)
    t1 = time.perf_counter() - t0
    k = int(max(1, min(sub.dim, per_step / max(t1, 1e-5))))
    for _ in range(args.warmup):
        step(k)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step(k)
    el = time.perf_counter() - t0
    units = args.steps * w.L * k * w.N
    val = units / el
    line = {
        "impl": "reference", "metric": METRIC, "value": val, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded)", "config": config_of(w),
        "cpu_baseline": {"value": val, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"per step: batch row 0, channels 0..{k - 1}, full L={w.L}"},
        "e2e": {"value": val, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def config_of(w):
    return {"workload": w.name, "batch": w.batch, "L": w.L, "D": w.dim, "N": w.N, "io": w.io,
            "A": "-(n+1)" if w.A_kind == "neg_n1" else "-exp(U(log1,log16))",
            "step_range": list(w.dt_range), "z_gate": w.has_z, "D_skip": w.has_D,
            "h_last": True, "parallelism": "replica per GPU",
            "l2": f"inputs larger than L2 ({w.io_bytes() / 1e6:.0f} MB footprint vs 126 MiB L2)"}


def run_decode(args, w):
    """Single-step decode (sscan_step) on the workload's (batch, dim, N): JSON line on stdout."""
    import torch

    from selective_state_space_158_b300 import binding
    from selective_state_space_158_b300.inputs import make_inputs

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    binding.load()
    # Enough concurrent sequences that the state (read and written every step) is twice the
    # 126 MiB L2: the step then streams the state from HBM instead of finding it in L2.
    batch = max(w.batch, math.ceil(2 * L2_BYTES / (w.dim * w.N * 4)))
    w = w.replace(L=1, batch=batch)
    x = make_inputs(w, device=dev)
    one = {k: (v[:, 0].contiguous() if v is not None and v.dim() == 3 else v)
           for k, v in x.items()}
    g = torch.Generator(device=dev)
    g.manual_seed(7)
    h = torch.randn((w.batch, w.dim, w.N), generator=g, device=dev, dtype=torch.float32) * 0.1
    y = torch.empty_like(one["u"])

    def step(stream=None):
        binding.step(one["u"], one["delta"], one["A"], one["B"], one["C"], h, D=one.get("D"),
                     z=one.get("z"), delta_bias=one.get("delta_bias"), y=y, stream=stream)

    stream = torch.cuda.Stream(dev)
    K = max(64, args.steps - args.steps % 64)
    for _ in range(max(3, args.warmup)):
        step(stream)
    torch.cuda.synchronize(dev)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(0) as cs:
        ev0.record(stream)
        for _ in range(K):
            step(stream)
        ev1.record(stream)
        torch.cuda.synchronize(dev)
    ms_launch = ev0.elapsed_time(ev1) / K
    # 64 steps captured once, replayed K / 64 times
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for _ in range(64):
            step()
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize(dev)
    ev0.record()
    for _ in range(K // 64):
        graph.replay()
    ev1.record()
    torch.cuda.synchronize(dev)
    ms_graph = ev0.elapsed_time(ev1) / K
    es = 4 if w.io == "f32" else 2
    bdn = w.batch * w.dim * w.N
    bytes_ = (2 * bdn * 4 + w.dim * w.N * 4 + w.dim * 4 * (int(w.has_D) + int(w.has_bias))
              + w.batch * w.dim * es * (3 + int(w.has_z)) + 2 * w.batch * w.N * es)
    hbm_gbs, _, peak_src = peaks()
    gbs = bytes_ / (ms_graph / 1e3) / 1e9
    line = {
        "metric": "selective-scan decode step (sscan_step): (B·D·N)/s and GB/s on 1 B300",
        "value": bdn / (ms_graph / 1e3), "unit": "(B*D*N)/s", "n_gpus": 1, "steps": K,
        "warmup": args.warmup, "ms_per_step": ms_graph, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": w.io, "data": "synthetic (seeded)",
        "config": {"workload": f"decode step, batch {w.batch}, D {w.dim}, N {w.N}, {w.io}",
                   "batch": w.batch, "D": w.dim, "N": w.N, "z_gate": w.has_z,
                   "D_skip": w.has_D, "timing": "CUDA graph of 64 steps, replayed",
                   "l2": f"state {bdn * 4 / 1e6:.0f} MB, twice the 126 MiB L2"},
        "gpu_launches": K,
        "launch_ms_per_step": ms_launch,
        "roofline": {"bound": "hbm", "achieved": gbs, "peak": hbm_gbs, "unit": "GB/s",
                     "frac": gbs / hbm_gbs, "traffic": None, "bytes_per_step": bytes_,
                     "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs, burst)"},
        "clocks": cs.summary(),
    }
    print(json.dumps(line), flush=True)


def run_conv(args, w):
    """Conv1d + SiLU over the workload's x: JSON line on stdout."""
    import torch

    from selective_state_space_158_b300 import binding

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    binding.load()
    g = torch.Generator(device=dev)
    g.manual_seed(11)
    dt = torch.float32 if w.io == "f32" else torch.bfloat16
    W = args.conv_width
    x = torch.randn((w.batch, w.L, w.dim), generator=g, device=dev).to(dt)
    wt = torch.randn((w.dim, W), generator=g, device=dev) * 0.5
    bias = torch.randn((w.dim,), generator=g, device=dev)
    y = torch.empty_like(x)
    stream = torch.cuda.Stream(dev)

    def step():
        binding.conv1d_silu(x, wt, bias, y=y, stream=stream)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize(dev)
    # 16 launches captured once and replayed, so that host-side argument checks do not pace the
    # GPU for this short kernel.
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for _ in range(16):
            binding.conv1d_silu(x, wt, bias, y=y)
    graph.replay()
    torch.cuda.synchronize(dev)
    K = max(16, args.steps - args.steps % 16)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(0) as cs:
        ev0.record()
        for _ in range(K // 16):
            graph.replay()
        ev1.record()
        torch.cuda.synchronize(dev)
    ms = ev0.elapsed_time(ev1) / K
    es = 4 if w.io == "f32" else 2
    bld = w.batch * w.L * w.dim
    bytes_ = 2 * bld * es + w.dim * (W + 1) * 4
    hbm_gbs, _, peak_src = peaks()
    gbs = bytes_ / (ms / 1e3) / 1e9
    line = {
        "metric": "causal depthwise conv1d + SiLU (sscan_conv1d_silu): (B·L·D)/s and GB/s on 1 B300",
        "value": bld / (ms / 1e3), "unit": "(B*L*D)/s", "n_gpus": 1, "steps": K,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": w.io, "data": "synthetic (seeded)",
        "config": {"workload": f"conv1d width {W} + SiLU on {w.name}", "batch": w.batch,
                   "L": w.L, "D": w.dim, "width": W,
                   "timing": "CUDA graph of 16 launches, replayed",
                   "l2": f"input {bld * es / 1e6:.0f} MB vs 126 MiB L2"},
        "gpu_launches": K,
        "roofline": {"bound": "hbm", "achieved": gbs, "peak": hbm_gbs, "unit": "GB/s",
                     "frac": gbs / hbm_gbs, "traffic": None, "bytes_per_step": bytes_,
                     "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs, burst)"},
        "clocks": cs.summary(),
    }
    print(json.dumps(line), flush=True)


BWD_FP32_OPS_PER_UPDATE = 16  # recompute (4) + adjoint (12) FP32-pipe operations per update


def run_bwd(args, w):
    """Backward pass over the workload: JSON line on stdout."""
    import torch

    from selective_state_space_158_b300 import binding
    from selective_state_space_158_b300.inputs import make_inputs

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    binding.load()
    x = make_inputs(w, device=dev)
    g = torch.Generator(device=dev)
    g.manual_seed(13)
    dy = torch.randn(x["u"].shape, generator=g, device=dev).to(x["u"].dtype)
    dh = torch.randn((w.batch, w.dim, w.N), generator=g, device=dev)
    stream = torch.cuda.Stream(dev)

    def step():
        return binding.bwd(x["u"], x["delta"], x["A"], x["B"], x["C"], dy, D=x.get("D"),
                           z=x.get("z"), delta_bias=x.get("delta_bias"), dh_last=dh,
                           stream=stream)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize(dev)
    K = args.steps
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(0) as cs:
        ev0.record(stream)
        for _ in range(K):
            step()
        ev1.record(stream)
        torch.cuda.synchronize(dev)
    ms = ev0.elapsed_time(ev1) / K
    props = torch.cuda.get_device_properties(dev)
    _, sm_max_mhz, _ = peaks()
    fp32_peak = props.multi_processor_count * 128 * sm_max_mhz * 1e6  # lane-ops per second
    ach = w.elems * BWD_FP32_OPS_PER_UPDATE / (ms / 1e3)
    line = {
        "metric": "selective-scan backward (sscan_bwd): (B·L·D·N)/s on 1 B300",
        "value": w.elems / (ms / 1e3), "unit": "(B*L*D*N)/s", "n_gpus": 1, "steps": K,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": w.io, "data": "synthetic (seeded)",
        "config": dict(config_of(w), workload=f"backward of {w.name}"),
        "gpu_launches": 3 * K + (K if (w.io != "f32" or w.N != 16) else 0),
        "roofline": {"bound": "alu", "achieved": ach / 1e9, "peak": fp32_peak / 1e9,
                     "unit": "G FP32 lane-ops/s", "frac": ach / fp32_peak, "traffic": None,
                     "ops_per_update": BWD_FP32_OPS_PER_UPDATE,
                     "peak_source": f"{props.multi_processor_count} SMs x 128 lanes x "
                                    f"{sm_max_mhz:.0f} MHz"},
        "clocks": cs.summary(),
    }
    print(json.dumps(line), flush=True)


def measure_rates(index: int = 0) -> dict:
    """Issue rates of this GPU's SMs from the library's probes (libsscan_peaks): ex2.approx,
    scalar FFMA, packed FFMA2, and the scan's per-update mix (one ex2 + four FP32 operations) in
    both forms; per SM and clock (clock-independent: cycles counted on the SM)."""
    import ctypes

    import numpy as np
    import torch

    from selective_state_space_158_b300 import build

    lib = ctypes.CDLL(build.PEAKS_LIB)
    fn = lib.sscan_peaks_probe
    fn.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
                   ctypes.c_void_p]
    fn.restype = ctypes.c_int
    sms = torch.cuda.get_device_properties(index).multi_processor_count
    blocks, iters = 2 * sms, 4096
    out = {}
    with torch.cuda.device(index):
        for kind, name in enumerate(["ex2", "ffma", "ffma2", "mix_packed", "mix_scalar"]):
            cyc = np.zeros(blocks, dtype=np.int64)
            e, f = ctypes.c_int(), ctypes.c_int()
            rc = fn(kind, blocks, iters, cyc.ctypes.data, ctypes.byref(e), ctypes.byref(f))
            if rc != 0:
                raise RuntimeError(f"rate probe {name} failed: CUDA error {rc}")
            med = float(np.median(cyc))
            out[name] = {"ex2_per_clk_sm": 1024 * iters * e.value / med,
                         "fp32_per_clk_sm": 1024 * iters * f.value / med,
                         "cycles_median": med, "cycles_spread": [int(cyc.min()), int(cyc.max())]}
        out["step_loop"] = step_loop_rates(lib, sms)
    return out


def step_loop_rates(lib, sms: int, chunks: int = 256) -> dict:
    """The scan's step loop alone (libsscan_peaks step-loop probe: states in registers, the
    step's (dt, dt u) and B/C rows from shared memory, no HBM traffic, no prologue or epilogue),
    in state updates per SM and clock, for 16 and 8 states per lane, with and without the readout,
    at 8, 16 and 24 resident warps per SM. Per SM: the updates of its CTAs over the span from the
    first start to the last end on its own clock; the median over SMs."""
    import ctypes

    import numpy as np

    fn = lib.sscan_peaks_step_loop
    fn.argtypes = [ctypes.c_int] * 4 + [ctypes.c_void_p, ctypes.c_void_p]
    fn.restype = ctypes.c_int
    res = {}
    for k in (16, 8):
        for readout in (1, 0):
            for wps in (8, 16, 24):
                blocks = sms * wps // 4
                smid = np.zeros(blocks, dtype=np.uint32)
                clk = np.zeros(2 * blocks, dtype=np.int64)
                rc = fn(k, readout, blocks, chunks, smid.ctypes.data, clk.ctypes.data)
                if rc != 0:
                    raise RuntimeError(f"step-loop probe failed: CUDA error {rc}")
                per_sm = []
                for sm in np.unique(smid):
                    m = smid == sm
                    span = int(clk[1::2][m].max() - clk[0::2][m].min())
                    per_sm.append(int(m.sum()) * 128 * k * 16 * chunks / span)
                name = f"states{k}_{'readout' if readout else 'no_readout'}_warps{wps}"
                res[name] = float(np.median(per_sm))
    return res


def update_peak(rates: dict, sms: int, mhz: float) -> dict:
    """The compute roofline of the scan: per update one SFU ex2 and four FP32-pipe operations,
    at the measured ex2 rate and the better of the measured FFMA / FFMA2 rates."""
    r_ex2 = rates["ex2"]["ex2_per_clk_sm"]
    r_fma = max(rates["ffma"]["fp32_per_clk_sm"], rates["ffma2"]["fp32_per_clk_sm"])
    per_clk = min(r_ex2, r_fma / FP32_OPS_PER_UPDATE)
    return {"updates_per_s": per_clk * sms * mhz * 1e6, "sms": sms, "mhz": mhz,
            "ex2_per_clk_sm": r_ex2,
            "fp32_per_clk_sm": r_fma, "updates_per_clk_sm": per_clk,
            "binding_pipe": "SFU" if r_ex2 <= r_fma / FP32_OPS_PER_UPDATE else "FP32",
            "mix_updates_per_clk_sm": rates["mix_packed"]["ex2_per_clk_sm"],
            "step_loop_updates_per_clk_sm": rates["step_loop"]["states16_readout_warps24"],
            "source": f"libsscan_peaks probes on this GPU x {sms} SMs x {mhz:.0f} MHz (max SM "
                      f"clock)"}


def scan_roofline(w, sec_per_launch: float, peak: dict, hbm_gbs: float, peak_src: str,
                  traffic, clocks=None) -> dict:
    bytes_ = w.io_bytes()
    gbs = bytes_ / sec_per_launch / 1e9
    ups = w.elems / sec_per_launch
    t_hbm = bytes_ / (hbm_gbs * 1e9)
    t_alu = w.elems / peak["updates_per_s"]
    if t_hbm >= t_alu:
        roof = {"bound": "hbm", "achieved": gbs, "peak": hbm_gbs, "unit": "GB/s",
                "frac": gbs / hbm_gbs, "traffic": traffic,
                "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs, burst)"}
    else:
        roof = {"bound": "alu", "achieved": ups / 1e9, "peak": peak["updates_per_s"] / 1e9,
                "unit": "G state updates/s (1 SFU ex2 + 4 FP32 ops each)",
                "frac": ups / peak["updates_per_s"], "traffic": traffic,
                "peak_source": peak["source"]}
    roof["hbm_frac"] = gbs / hbm_gbs
    roof["alu_frac"] = ups / peak["updates_per_s"]
    # the scan's step loop alone (no HBM, no prologue / epilogue), 24 warps per SM: the practical
    # ceiling of this instruction mix, for context
    loop_ups = peak["step_loop_updates_per_clk_sm"] * peak["sms"] * peak["mhz"] * 1e6
    roof["step_loop_frac"] = ups / loop_ups
    roof["algorithmic_bytes"] = bytes_
    roof["t_hbm_ms"] = t_hbm * 1e3
    roof["t_alu_ms"] = t_alu * 1e3
    if clocks and clocks.get("sm_mhz"):
        at_obs = peak["updates_per_clk_sm"] * peak["sms"] * clocks["sm_mhz"] * 1e6
        roof["alu_frac_at_observed_clock"] = ups / at_obs
    return roof


def launches_per_step(w) -> int:
    """The library's kernels per sscan_fwd call: the scan, plus the pass that widens B and C to
    fp32 rows of 16 states when they are bf16 or N < 16."""
    return 1 + (1 if (w.io != "f32" or w.N != 16) else 0)


def run_peaks(args):
    import torch

    torch.cuda.set_device(0)
    rates = measure_rates(0)
    props = torch.cuda.get_device_properties(0)
    _, mhz, _ = peaks()
    pk = update_peak(rates, props.multi_processor_count, mhz)
    line = {"metric": "issue rates per SM and clock (libsscan_peaks)", "gpu": props.name,
            "sms": props.multi_processor_count, "sm_max_mhz": mhz, "rates": rates,
            "scan_update_peak": pk}
    print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    from selective_state_space_158_b300.inputs import WORKLOADS

    w = WORKLOADS[args.workload]
    if args.L:
        w = w.replace(L=args.L)
    if args.dim:
        w = w.replace(dim=args.dim)
    if args.impl == "reference":
        run_reference(args, w)
        return
    if args.mode == "peaks":
        run_peaks(args)
        return
    if args.mode == "decode":
        run_decode(args, w)
        return
    if args.mode == "conv":
        run_conv(args, w)
        return
    if args.mode == "bwd":
        run_bwd(args, w)
        return

    import torch
    import torch.distributed as dist

    from selective_state_space_158_b300 import binding
    from selective_state_space_158_b300.inputs import make_inputs

    world, rank, local = dist_setup(args.gpus)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    binding.load()  # fails loudly if the library is missing

    hbm_gbs, sm_max_mhz, peak_src = peaks()
    props = torch.cuda.get_device_properties(dev)
    sms = props.multi_processor_count
    rates = measure_rates(local)
    upeak = update_peak(rates, sms, sm_max_mhz)
    stream = torch.cuda.Stream(dev)

    def barrier():
        if world > 1:
            dist.barrier()

    def prepare(wk):
        x = make_inputs(wk, device=dev)
        y = torch.empty_like(x["u"])
        h = torch.empty((wk.batch, wk.dim, wk.N), dtype=torch.float32, device=dev)

        def step():
            binding.fwd(x["u"], x["delta"], x["A"], x["B"], x["C"], x.get("D"), x.get("z"),
                        x.get("delta_bias"), y=y, h_last=h, stream=stream)
        return x, y, h, step

    def timed(step, K):
        ev0 = torch.cuda.Event(enable_timing=True)
        ev1 = torch.cuda.Event(enable_timing=True)
        barrier()
        torch.cuda.synchronize(dev)
        with ClockSampler(local) as cs:
            ev0.record(stream)
            for _ in range(K):
                step()
            ev1.record(stream)
            torch.cuda.synchronize(dev)
        barrier()
        return ev0.elapsed_time(ev1), cs

    def measure(step, K):
        ms, cs = timed(step, K)
        remeasured = False
        if cs.rejected():
            ms, cs = timed(step, K)
            remeasured = True
        if binding.device_error(stream) != 0:
            raise RuntimeError("device-side error during the timed region")
        clocks = cs.summary()
        if remeasured:
            clocks["note"] = "first measurement rejected by clock check; re-measured once"
        return max_over_ranks(ms, world, dev), clocks

    def warm(step, n):
        for _ in range(max(3, n)):
            step()
        torch.cuda.synchronize(dev)
        if binding.device_error(stream) != 0:
            raise RuntimeError("device-side error during warm-up")

    # ---- headline workload: exactly --steps steps ----
    x, y, h, step = prepare(w)
    warm(step, args.warmup)
    ms_max, clocks = measure(step, args.steps)
    sec_per_step = ms_max / 1e3 / args.steps
    value = whole_job_rate(w.elems, world, sec_per_step)
    roof = scan_roofline(w, sec_per_step, upeak, hbm_gbs, peak_src,
                         recorded_traffic(args.workload) if not (args.L or args.dim) else None,
                         clocks)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_max / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": w.io, "data": "synthetic (seeded)",
        "config": config_of(w), "gbs": w.io_bytes() / sec_per_step / 1e9 * world,
        "gpu_launches": args.steps * launches_per_step(w),
        "roofline": roof, "clocks": clocks,
        "peaks": {"update_peak": upeak, "probes": rates},
    }

    # ---- end to end through the host-buffer C entry point ----
    if not args.no_e2e:
        xh = {k: (v.cpu().pin_memory() if v is not None else None) for k, v in x.items()}
        yh = torch.empty(y.shape, dtype=y.dtype).pin_memory()
        hh = torch.empty(h.shape, dtype=h.dtype).pin_memory()

        def e2e_step():
            binding.fwd_host(xh["u"], xh["delta"], xh["A"], xh["B"], xh["C"], xh.get("D"),
                             xh.get("z"), xh.get("delta_bias"), y=yh, h_last=hh, device=local,
                             stream=stream)

        e2e_step()
        K2 = max(3, args.e2e_steps)
        barrier()
        t0 = time.perf_counter()
        for _ in range(K2):
            e2e_step()
        el = time.perf_counter() - t0
        el = max_over_ranks(el, world, dev)
        es = 4 if w.io == "f32" else 2
        bld, bln = w.batch * w.L * w.dim, w.batch * w.L * w.N
        h2d = bld * es * (2 + int(w.has_z)) + 2 * bln * es + w.dim * w.N * 4 + \
            w.dim * 4 * (int(w.has_D) + int(w.has_bias))
        d2h = bld * es + w.batch * w.dim * w.N * 4
        line["e2e"] = {"value": whole_job_rate(w.elems * K2, world, el), "unit": UNIT,
                       "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                       "steps": K2, "ms_per_step": el / K2 * 1e3,
                       "api": "sscan_fwd_host (pinned host buffers, copies inside the region)"}
        del xh, yh, hh

    if rank == 0 and world == 1 and not args.no_cpu:
        line["cpu_baseline"] = cpu_baseline(w, x, args.cpu_seconds)
    del x, y, h, step
    torch.cuda.empty_cache()

    # ---- the other full-size workloads, each over >= MIN_REGION_MS of device time ----
    if not args.no_configs:
        line["configs"] = {}
        for key in EXTRA_WORKLOADS:
            if key == args.workload:
                continue
            wk = WORKLOADS[key]
            xk, yk, hk, stepk = prepare(wk)
            warm(stepk, 3)
            t1, _ = timed(stepk, 3)
            K = max(5, math.ceil(MIN_REGION_MS / max(t1 / 3, 1e-3)))
            K = int(max_over_ranks(K, world, dev))
            msk, ck = measure(stepk, K)
            if msk < MIN_REGION_MS:  # the short estimate ran slower per step: time again, longer
                K = math.ceil(K * 1.1 * MIN_REGION_MS / max(msk, 1e-3))
                K = int(max_over_ranks(K, world, dev))
                msk, ck = measure(stepk, K)
            sk = msk / 1e3 / K
            line["configs"][key] = {
                "workload": wk.name, "ms_per_step": msk / K, "steps": K,
                "timed_ms": msk, "value": whole_job_rate(wk.elems, world, sk), "unit": UNIT,
                "gbs": wk.io_bytes() / sk / 1e9 * world, "dtype": wk.io,
                "gpu_launches": K * launches_per_step(wk),
                "roofline": scan_roofline(wk, sk, upeak, hbm_gbs, peak_src,
                                          recorded_traffic(key), ck),
                "clocks": ck, "config": config_of(wk)}
            del xk, yk, hk, stepk
            torch.cuda.empty_cache()

    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
