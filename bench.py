"""Benchmark: fused Command throughput on GB300 (HBM GB/s, fraction of the
HBM roofline, elements/s).

One step = one fused pass of the Command over one batch of synthetic input:
the workload is the largest of the five headline configurations, the int32
wraparound Command out = x*y + z - w over N = 2^28 elements (four 1 GiB
inputs, one 1 GiB output), inputs resident in HBM. The line also carries
per-workload measurements of the other Commands (add, the fp32 chain,
strided bf16 transpose, wide 16-op DAG and the rest) at their full sizes, an
end-to-end figure through the same API with the tensors in pinned host
memory (the kernel reads and writes them across the host link; a copy
pipeline is reported beside it), the roofline of the executor kernel, SM clocks
sampled during the timed region, and the CPU oracle timed on a bounded
sample as a reported baseline.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload NAME] [--headline-only]

Under torchrun (N > 1) every rank runs its own replica of the workload (the
path has no exchange step); value = all ranks' bytes / max-over-ranks time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

from inputgen import workloads as W  # noqa: E402

HEADLINE = "wrap_i32"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
METRIC = "fused Command throughput: HBM GB/s and % of GB300 HBM roofline (elements/s)"
NP_OF = {"f32": np.float32, "f16": np.float16, "bf16": np.int16, "i32": np.int32, "b1": np.uint32}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=HEADLINE, choices=list(W.FULL) + list(W.LAYOUT) + list(W.PROFILE))
    ap.add_argument("--headline-only", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-extras", action="store_true",
                    help="only the device-timed region (no e2e, CPU baseline or other workloads): for profiling")
    ap.add_argument("--size", type=int, default=0,
                    help="override the workload size (elements; rows = cols for the strided workload)")
    return ap.parse_args()


def make_spec(name, size):
    f = W.FULL.get(name) or W.LAYOUT.get(name) or W.PROFILE[name]
    if not size:
        return f()
    if name == "strided_bf16":
        return f(size, size, size + 128)
    if name == "tile4_f32":
        return f(size, size)
    if name == "batched_transpose":
        return f(max(1, size // (1 << 20)))
    if name == "rows_chain_f32":
        return f(size, size)
    return f(size)


def measured_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


KERNEL_SOURCES = {
    "exec_contig": ["exec_contig.cu", "exec_common.cuh", "interp_asm.cuh", "cmd_internal.h"],
    "exec_tile2d": ["exec_tile2d.cu", "exec_tile2d.h", "exec_common.cuh", "exec_pipe.cuh", "interp_asm.cuh",
                    "cmd_internal.h"],
    "exec_generic": ["exec_generic.cu", "exec_common.cuh", "interp_asm.cuh", "cmd_internal.h"],
}


KERNEL_OF_PATH = {"contig": "exec_contig", "tile2d": "exec_tile2d", "generic": "exec_generic"}


def source_hash(kernel: str) -> str:
    """Hash of the sources that make up one executor kernel."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "tensor_command_execution_gb300", "csrc")
    for name in KERNEL_SOURCES[kernel]:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode())
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from a committed ncu summary, if it was taken
    from the current kernel sources (else None)."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.md")
    try:
        text = open(path).read()
    except OSError:
        return None
    m = re.search(r"traffic_bytes_per_launch:\s*([0-9]+)", text)
    s = re.search(r"source_sha256:\s*([0-9a-f]+)", text)
    if not m or not s or s.group(1) != source_hash(kernel):
        return None
    return int(m.group(1))


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons, taken while the
    timed region runs (start before, stop after)."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.samples = []
        self.proc = None
        self.thread = None
        self.window = (0.0, 0.0)

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        time.sleep(0.3)

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), [x.strip() for x in line.split(",")]))

    def mark(self, t0, t1):
        self.window = (t0, t1)

    def stop(self):
        if self.proc:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        t0, t1 = self.window
        inside = [s for t, s in self.samples if t0 <= t <= t1]
        scope = "timed"
        if len(inside) < 2:
            inside = [s for t, s in self.samples]
            scope = "timed+surrounding (timed region shorter than the sampling period)"

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(s[0]) for s in inside if num(s[0]) is not None]
        mx = [num(s[1]) for s in inside if num(s[1]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for s in inside for i in range(4) if len(s) > 4 + i and s[4 + i] == "Active"})
        power = [num(s[2]) for s in inside if num(s[2]) is not None]
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(inside), "scope": scope,
                "power_w_max": max(power) if power else None}


def host_inputs(spec, pinned: bool):
    """Seeded inputs in (pinned) host memory, filled in place by inputgen."""
    import torch

    import inputgen
    dts = W.tensor_dtypes(spec)
    out = {}
    for k, name in enumerate(W.load_names(spec)):
        kind, lo, hi = spec["inputs"][name]
        n = spec["views"][name]["alloc"]
        t = torch.empty(n, dtype=getattr(torch, {"f32": "float32", "f16": "float16", "bf16": "int16",
                                                  "i32": "int32"}[dts[name]]), pin_memory=pinned)
        inputgen.fill_ptr(kind, spec["seed"], k, t.data_ptr(), n, lo, hi)
        out[name] = t
    return out


def torch_dtype(dt):
    import torch
    return {"f32": torch.float32, "f16": torch.float16, "bf16": torch.int16, "i32": torch.int32,
            "b1": torch.int32}[dt]


class Workload:
    """A compiled Command with device buffers and pre-built launch arguments."""

    def __init__(self, spec, device):
        import torch

        import tensor_command_execution_gb300 as T
        self.spec = spec
        self.dts = W.tensor_dtypes(spec)
        self.host = host_inputs(spec, pinned=True)
        self.dev = {n: t.to(device) for n, t in self.host.items()}
        for n in W.store_names(spec):
            self.dev[n] = torch.empty(spec["views"][n]["alloc"], dtype=torch_dtype(self.dts[n]), device=device)
        # a tensor placed `off` elements into its allocation (spec offsets)
        self._alloc = {}
        for n, off in spec.get("offsets", {}).items():
            t = self.dev[n]
            big = torch.empty(t.numel() + off, dtype=t.dtype, device=device)
            big[off:].copy_(t)
            self._alloc[n] = big
            self.dev[n] = big[off:]
        self.cmd, self.tags = T.command_from_spec(spec)
        self.kernel = self.cmd.compile()
        self.views = {self.tags[n]: self.view_of(n, t) for n, t in self.dev.items()}
        self.scal = T.spec_scalars(spec, self.tags)
        self.args = self.kernel.args(self.views, self.scal)
        self.plan = self.kernel.plan(self.views, self.scal)
        self.bytes = self.plan["bytes"]
        self.elements = self.plan["n_elements"]
        info = self.kernel.info()
        # elements per warp chunk of the contiguous executor: 32 x (elements per slot per thread)
        half2 = all(self.dts[n] in ("f16", "bf16") for n in W.load_names(spec))
        per_slot = {0: 16, 3: 2, 4: 4}.get(info["tier"], 16 if (info["tier"] == 1 and not info["extended"] and half2)
                                           else 8)
        chunk = 32 * per_slot
        self.launches_per_step = 1 + (1 if (self.plan["path"] == "contig" and self.elements % chunk != 0) else 0)

    def units(self, name, a, b):
        """Buffer range holding elements [a, b) of a dense 1-D tensor (for a
        packed-bit store, its 32-bit words; a is then a multiple of 32)."""
        if self.dts[name] == "b1":
            return a // 32, (b + 31) // 32
        return a, b

    def view_of(self, name, t, start=0, count=None):
        """The view of tensor `name` over buffer t (optionally elements
        [start, start + count) of a dense 1-D tensor)."""
        import tensor_command_execution_gb300 as T
        if count is None:
            return T.TensorView(t.data_ptr(), self.spec["sizes"], self.spec["views"][name]["strides"])
        u0, _ = self.units(name, start, start + count)
        return T.TensorView(t.data_ptr() + u0 * t.element_size(), (count,), (1,))

    def launch(self, stream_handle):
        self.kernel.launch_args(self.args, stream_handle)


def time_device(wl, stream, steps, warmup):
    """K launches between CUDA events on the launching stream; ms per step."""
    import torch
    h = stream.cuda_stream
    for _ in range(warmup):
        wl.launch(h)
    torch.cuda.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    stop = torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for _ in range(steps):
        wl.launch(h)
    stop.record(stream)
    stop.synchronize()
    return start.elapsed_time(stop) / steps


def time_graph_rotating(wl, device, min_bytes, replays):
    """Per-launch time of wl's kernel from a CUDA graph that launches it once
    on each of R copies of its buffers (R * bytes >= min_bytes)."""
    import math

    import torch
    sets = max(2, math.ceil(min_bytes / wl.bytes))
    arg_sets = []
    keep = []
    for _ in range(sets):
        bufs = {n: t.clone() for n, t in wl.dev.items()}
        keep.append(bufs)
        views = {wl.tags[n]: wl.view_of(n, t) for n, t in bufs.items()}
        arg_sets.append(wl.kernel.args(views, wl.scal))
    s = torch.cuda.Stream(device)
    for a in arg_sets:  # warm-up outside the capture
        wl.kernel.launch_args(a, s.cuda_stream)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for a in arg_sets:
            wl.kernel.launch_args(a, s.cuda_stream)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(s)
    with torch.cuda.stream(s):
        for _ in range(replays):
            g.replay()
    e1.record(s)
    e1.synchronize()
    del keep
    return e0.elapsed_time(e1) / (replays * sets), sets


class E2EPipeline:
    """One end-to-end step through the public API: the inputs are copied in
    from pinned host memory chunk by chunk, each chunk is launched once it has
    landed and its outputs are copied back once computed, on three streams, so
    host-to-device copies, kernels and device-to-host copies overlap. Dense
    1-D workloads are split into chunks; others run as one chunk."""

    def __init__(self, wl, device, chunks):
        import torch
        self.wl = wl
        spec = wl.spec
        names_in = W.load_names(spec)
        names_out = W.store_names(spec)
        dense_1d = len(spec["sizes"]) == 1 and all(spec["views"][k]["strides"] == (1,)
                                                   for k in names_in + names_out)
        n = wl.elements
        c = chunks if dense_1d else 1
        step = -(-n // c)
        step = -(-step // 256) * 256  # keep chunk starts 16-byte aligned for every dtype
        self.bounds = [(a, min(n, a + step)) for a in range(0, n, step)] if dense_1d else [(0, n)]
        self.dense_1d = dense_1d
        self.outs_host = {k: torch.empty_like(wl.dev[k], device="cpu").pin_memory() for k in names_out}
        self.h2d_bytes = sum(t.numel() * t.element_size() for t in wl.host.values())
        self.d2h_bytes = sum(t.numel() * t.element_size() for t in self.outs_host.values())
        self.s_in = torch.cuda.Stream(device)
        self.s_k = torch.cuda.Stream(device)
        self.s_out = torch.cuda.Stream(device)
        self.args = []
        for a, b in self.bounds:
            if dense_1d:
                views = {wl.tags[k]: wl.view_of(k, wl.dev[k], a, b - a) for k in names_in + names_out}
            else:
                views = wl.views
            self.args.append(wl.kernel.args(views, wl.scal))
        m = len(self.bounds)
        self.ev_in = [torch.cuda.Event() for _ in range(m)]
        self.ev_k = [torch.cuda.Event() for _ in range(m)]
        self.ev_out = [torch.cuda.Event() for _ in range(m)]
        self.started = False

    def step(self):
        import torch
        wl = self.wl
        for c, (a, b) in enumerate(self.bounds):
            if self.started:
                self.s_in.wait_event(self.ev_k[c])    # last step's kernel has read this chunk
            with torch.cuda.stream(self.s_in):
                for k, t in wl.host.items():
                    if self.dense_1d:
                        u0, u1 = wl.units(k, a, b)
                        wl.dev[k][u0:u1].copy_(t[u0:u1], non_blocking=True)
                    else:
                        wl.dev[k].copy_(t, non_blocking=True)
            self.ev_in[c].record(self.s_in)
            self.s_k.wait_event(self.ev_in[c])
            if self.started:
                self.s_k.wait_event(self.ev_out[c])   # last step's outputs of this chunk are home
            wl.kernel.launch_args(self.args[c], self.s_k.cuda_stream)
            self.ev_k[c].record(self.s_k)
            self.s_out.wait_event(self.ev_k[c])
            with torch.cuda.stream(self.s_out):
                for k, t in self.outs_host.items():
                    if self.dense_1d:
                        u0, u1 = wl.units(k, a, b)
                        t[u0:u1].copy_(wl.dev[k][u0:u1], non_blocking=True)
                    else:
                        t.copy_(wl.dev[k], non_blocking=True)
            self.ev_out[c].record(self.s_out)
        self.started = True


class E2EHostDirect:
    """One end-to-end step through the public API with the tensors where the
    user holds them: the step's inputs in pinned host memory and its outputs
    written to pinned host memory, by one launch whose kernel reads and
    writes them across the host link (the pointers are valid on the device
    under unified addressing; on a Grace host the link is the coherent
    CPU-GPU one). The host-to-device transfer of the inputs and the
    device-to-host transfer of the result happen inside the launch."""

    def __init__(self, wl, device):
        import torch
        self.wl = wl
        self.outs_host = {k: torch.empty_like(wl.dev[k], device="cpu").pin_memory() for k in W.store_names(wl.spec)}
        views = {wl.tags[n]: wl.view_of(n, t) for n, t in wl.host.items()}
        views.update({wl.tags[n]: wl.view_of(n, t) for n, t in self.outs_host.items()})
        self.args = wl.kernel.args(views, wl.scal)
        self.plan = wl.kernel.plan(views, wl.scal)
        self.stream = torch.cuda.Stream(device)
        self.h2d_bytes = sum(t.numel() * t.element_size() for t in wl.host.values())
        self.d2h_bytes = sum(t.numel() * t.element_size() for t in self.outs_host.values())

    def step(self):
        self.wl.kernel.launch_args(self.args, self.stream.cuda_stream)


def time_e2e(stepper, first_stream, last_stream, steps, world, device):
    """ms per end-to-end step: a few untimed steps, then `steps` between
    events (the last one's completion waited for), max over ranks."""
    import torch
    import torch.distributed as dist
    for _ in range(3):
        stepper.step()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(first_stream)
    for _ in range(steps):
        stepper.step()
    e1.record(last_stream)
    e1.synchronize()
    torch.cuda.synchronize()
    return max_over_ranks(e0.elapsed_time(e1) / steps, world, device)


def per_launch_times(wl, stream, n: int) -> dict:
    """Median and best of n launches, each between its own pair of events
    (a pass of its own after the headline region: an event recorded between
    two launches keeps the second from starting early, so the headline
    times the launches back to back)."""
    import torch
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    for a, b in evs:
        a.record(stream)
        wl.launch(stream.cuda_stream)
        b.record(stream)
    torch.cuda.synchronize()
    us = sorted(a.elapsed_time(b) * 1e3 for a, b in evs)
    if not us:
        return {"n": 0}
    med = statistics.median(us)
    return {"n": n, "median_us": round(med, 2), "best_us": round(us[0], 2),
            "median_gbs": round(wl.bytes / (med * 1e-6) / 1e9, 1), "best_gbs": round(wl.bytes / (us[0] * 1e-6) / 1e9, 1)}


def max_over_ranks(x: float, world: int, device=None) -> float:
    """The largest value of x over all ranks (the job's time is its slowest
    rank's); x itself on one rank. Uses the default process group (NCCL on
    GPUs, gloo on CPU)."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device if device is not None else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbs(bytes_per_rank: int, world: int, ms_max: float) -> float:
    """Whole-job throughput: the bytes every rank moved over the slowest
    rank's time (each rank runs its own replica of the workload)."""
    return bytes_per_rank * world / (ms_max * 1e-3) / 1e9


DTYPE_OF = {"chain_f32": "f32", "add_f32": "f32", "wrap_i32": "int32", "strided_bf16": "f32 (bf16 io)",
            "tile4_f32": "f32", "wide32_f32": "f32",
            "wide_dag": "f32 (f32+f16 out)", "batched_transpose": "f32", "div_clamp_i32": "f32 (int32 out)",
            "threshold_u32": "u32 (int32 out)", "threshold_bits": "u32 (packed-bit out)",
            "chain_bf16": "f32 (bf16 io)", "rows_chain_f32": "f32", "stencil_f32": "f32"}


def run_ours(args):
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl", init_method="env://")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    stream = torch.cuda.Stream(device)
    peak, peak_kind = measured_peak()

    spec = make_spec(args.workload, args.size)
    wl = Workload(spec, device)
    torch.cuda.synchronize()

    # ---- device-timed region -------------------------------------------------
    clocks = ClockSampler(local)
    clocks.start()
    for _ in range(args.warmup):
        wl.launch(stream.cuda_stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    stop = torch.cuda.Event(enable_timing=True)
    t0 = time.time()
    start.record(stream)
    for _ in range(args.steps):
        wl.launch(stream.cuda_stream)
    stop.record(stream)
    stop.synchronize()
    torch.cuda.synchronize()
    t1 = time.time()
    if world > 1:
        dist.barrier()
    clocks.mark(t0, t1)
    clocks.stop()
    ms = max_over_ranks(start.elapsed_time(stop) / args.steps, world, device)
    gbs = wl.bytes / (ms * 1e-3) / 1e9
    value = whole_job_gbs(wl.bytes, world, ms)
    per_launch = per_launch_times(wl, stream, min(args.steps, 200))

    if args.no_extras:
        if rank == 0:
            print(json.dumps({"workload": args.workload, "elements": wl.elements, "ms_per_step": ms,
                              "gbs": round(gbs, 1), "frac": round(gbs / peak, 4), "path": wl.plan["path"]}))
        if world > 1:
            dist.destroy_process_group()
        return

    # ---- end to end: pinned host inputs -> the kernel -> pinned host outputs ----
    # (the public call on the user's host buffers; the copy pipeline beside it)
    direct = E2EHostDirect(wl, device)
    h2d, d2h = direct.h2d_bytes, direct.d2h_bytes
    e2e_ms = time_e2e(direct, direct.stream, direct.stream, args.e2e_steps, world, device)
    e2e_gbs = whole_job_gbs(wl.bytes, world, e2e_ms)
    pipe = E2EPipeline(wl, device, chunks=8)
    pipe_ms = time_e2e(pipe, pipe.s_in, pipe.s_out, args.e2e_steps, world, device)
    pipe_gbs = whole_job_gbs(wl.bytes, world, pipe_ms)
    del direct, pipe

    # ---- other workloads, same kernels, full sizes (per-rank, informative) ---
    per = {}
    if not args.headline_only and rank == 0:
        for name, f in list(W.FULL.items()) + list(W.LAYOUT.items()):
            if name == args.workload:
                continue
            other = Workload(f(), device)
            l2 = torch.cuda.get_device_properties(device).L2_cache_size
            if other.bytes < 4 * l2:
                # smaller than L2: a CUDA graph of launches over rotating
                # buffer sets (together > 4x L2), so neither launch overhead
                # nor L2 reuse is timed
                oms, sets = time_graph_rotating(other, device, 4 * l2, 50)
                steps, how = sets * 50, f"CUDA graph of {sets} launches over {sets} buffer sets, replayed 50x"
            else:
                steps = max(20, min(2000, int(0.5 / max(1e-6, other.bytes / (peak * 1e9)))))
                oms, how = time_device(other, stream, steps, 10), "stream launches"
            ogbs = other.bytes / (oms * 1e-3) / 1e9
            per[name] = {"path": other.plan["path"], "elements": other.elements, "bytes_per_launch": other.bytes,
                         "us_per_launch": round(oms * 1e3, 2), "gbs": round(ogbs, 1),
                         "frac_of_measured_peak": round(ogbs / peak, 4),
                         "frac_of_nominal_8000": round(ogbs / NOMINAL_HBM_GBS, 4),
                         "elements_per_s": round(other.elements / (oms * 1e-3), 1), "launches": steps,
                         "timing": how,
                         "traffic": profiled_traffic(KERNEL_OF_PATH[other.plan["path"]], name)}
            del other
            torch.cuda.empty_cache()

    # ---- CPU oracle on a bounded sample (rank 0) --------------------------------
    cpu = None
    if rank == 0 and world == 1:
        cpu = cpu_baseline(spec, args.cpu_seconds)

    if rank == 0:
        kernel_name = KERNEL_OF_PATH[wl.plan["path"]]
        line = {
            "metric": METRIC,
            "value": round(value, 2),
            "unit": "GB/s",
            "n_gpus": world,
            "steps": args.steps,
            "warmup": args.warmup,
            "ms_per_step": round(ms, 6),
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": DTYPE_OF[args.workload],
            "data": "synthetic (seeded SplitMix64 inputs; no dataset)",
            "config": {"workload": f"{args.workload}: {spec_summary(spec)}", "elements": wl.elements,
                       "bytes_per_step": wl.bytes, "path": wl.plan["path"],
                       "l2": "inputs larger than L2 (%d MiB moved per step vs 126 MiB L2); no flush" %
                             (wl.bytes >> 20),
                       "parallelism": f"replicas x{world}"},
            "elements_per_s": round(wl.elements * world / (ms * 1e-3), 1),
            "frac_of_nominal_8000": round(gbs / NOMINAL_HBM_GBS, 4),
            "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peak, "unit": "GB/s",
                         "frac": round(gbs / peak, 4), "peak_kind": peak_kind,
                         "kernel": kernel_name,
                         "traffic": profiled_traffic(kernel_name, args.workload),
                         "algorithmic_bytes_per_launch": wl.bytes},
            "per_launch": per_launch,
            "e2e": {"value": round(e2e_gbs, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "ms_per_step": round(e2e_ms, 4),
                    "how": "one cmd_launch on the pinned host input and output buffers: the kernel reads the inputs "
                           "and writes the result across the host link (no separate copies)",
                    "copy_pipeline": {"value": round(pipe_gbs, 2), "ms_per_step": round(pipe_ms, 4),
                                      "how": "copies in from pinned host memory, launch and copies out, 8 chunks "
                                             "pipelined over three streams"}},
            "gpu_launches": args.steps * wl.launches_per_step,
            "clocks": clocks.summary(),
            "cpu_baseline": cpu,
            "workloads": per,
            "impl": "ours",
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


def spec_summary(spec):
    sizes = "x".join(str(s) for s in spec["sizes"])
    return f"{sizes} elements, {len(W.load_names(spec))} loads, {len(W.store_names(spec))} stores"


def host_cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else the machine
    type)."""
    import platform
    import subprocess
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name:"):
                return line.split(":", 1)[1].strip()
    except Exception:  # lscpu missing or failing: fall through
        pass
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return platform.machine()


def cpu_baseline(spec, seconds):
    """The oracle, as it stands, on the host: single-threaded element walk over
    the first M elements of the same workload, M sized to about `seconds`."""
    import oracle
    bufs = {}
    dts = W.tensor_dtypes(spec)
    import inputgen
    n_total = W.numel(spec)
    # a bounded sample: first M logical elements (calibrated)
    probe = min(n_total, 1 << 16)
    for k, name in enumerate(W.load_names(spec)):
        kind, lo, hi = spec["inputs"][name]
        bufs[name] = inputgen.generate(kind, spec["seed"], k, spec["views"][name]["alloc"], lo, hi).view(
            NP_OF[dts[name]] if dts[name] != "bf16" else np.uint16)
    for name in W.store_names(spec):
        bufs[name] = np.zeros(spec["views"][name]["alloc"], dtype=NP_OF[dts[name]])
    oc = oracle.OracleCommand(spec, bufs)
    t = time.perf_counter()
    oc.eval_range(0, probe)
    rate = probe / max(1e-9, time.perf_counter() - t)
    m = int(min(n_total, max(probe, rate * seconds)))
    t = time.perf_counter()
    oc.eval_range(0, m)
    dt = time.perf_counter() - t
    bpe = W.algorithmic_bytes(spec) / n_total
    return {"value": round(m * bpe / dt / 1e9, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"first {m} of {n_total} logical elements of the same workload, single thread, "
                      f"{dt:.1f} s", "elements_per_s": round(m / dt, 1), "cpu_model": host_cpu_model(),
            "multicore": oracle_threads(oc, n_total, bpe, m / dt, seconds)}


def split_ranges(m: int, parts: int, align: int = 32) -> list:
    """[0, m) cut into `parts` contiguous ranges whose inner boundaries are
    multiples of `align` (so no two ranges write the same packed-bit word)."""
    step = -(-max(1, m // max(1, parts)) // align) * align
    cuts = list(range(0, m, step)) + [m]
    return [(a, b) for a, b in zip(cuts, cuts[1:]) if a < b]


def oracle_threads(oc, n_total: int, bpe: float, rate1: float, seconds: float) -> dict:
    """The same oracle split over the host cores by element ranges (one
    thread per core; the C walk runs without the interpreter lock)."""
    from concurrent.futures import ThreadPoolExecutor
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
    m = int(min(n_total, max(1 << 16, rate1 * cores * seconds / 2)))
    ranges = split_ranges(m, cores)
    t = time.perf_counter()
    with ThreadPoolExecutor(cores) as ex:
        list(ex.map(lambda r: oc.eval_range(*r), ranges))
    dt = time.perf_counter() - t
    return {"value": round(m * bpe / dt / 1e9, 4), "unit": "GB/s", "cores": cores,
            "sample": f"first {m} of {n_total} logical elements, {len(ranges)} element ranges on {cores} threads, "
                      f"{dt:.1f} s", "elements_per_s": round(m / dt, 1)}


def run_reference(args):
    """The oracle (the CPU reference of this path) timed on the host cores on
    the same workload, metric and unit; each step a bounded sample."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import inputgen
    import oracle
    spec = make_spec(args.workload, 0)
    dts = W.tensor_dtypes(spec)
    bufs = {}
    for k, name in enumerate(W.load_names(spec)):
        kind, lo, hi = spec["inputs"][name]
        bufs[name] = inputgen.generate(kind, spec["seed"], k, spec["views"][name]["alloc"], lo, hi).view(
            NP_OF[dts[name]] if dts[name] != "bf16" else np.uint16)
    for name in W.store_names(spec):
        bufs[name] = np.zeros(spec["views"][name]["alloc"], dtype=NP_OF[dts[name]])
    oc = oracle.OracleCommand(spec, bufs)
    n_total = W.numel(spec)
    probe = min(n_total, 1 << 16)
    t = time.perf_counter()
    oc.eval_range(0, probe)
    rate = probe / max(1e-9, time.perf_counter() - t)
    # whole run about two minutes by default (12 x --cpu-seconds in all)
    budget = min(120.0, 12.0 * args.cpu_seconds) / max(1, args.steps + args.warmup)
    m = int(min(n_total, max(4096, rate * budget)))
    for s in range(args.warmup):
        oc.eval_range(s * m % n_total, s * m % n_total + m)
    t = time.perf_counter()
    for s in range(args.steps):
        b = (s * m) % max(1, n_total - m)
        oc.eval_range(b, b + m)
    dt = (time.perf_counter() - t) / args.steps
    bpe = W.algorithmic_bytes(spec) / n_total
    val = m * bpe / dt / 1e9
    line = {"metric": METRIC, "value": round(val, 4), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": DTYPE_OF[args.workload], "data": "synthetic",
            "config": {"workload": f"{args.workload}: {spec_summary(spec)}"},
            "impl": "reference",
            "cpu_baseline": {"value": round(val, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                             "sample": f"{m} consecutive logical elements per step of {n_total}",
                             "cpu_model": host_cpu_model()},
            "e2e": {"value": round(val, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
