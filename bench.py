#!/usr/bin/env python3
"""Benchmark of the recurrent-layer forward pass on GB300.

One "step" of this benchmark is one whole layer run through the library
(input projection + the persistent step kernel that runs every recurrent time
step and writes Y, Y_h, Y_c) on seeded synthetic inputs already resident in
device memory.  The default workload is the pages' bidirectional LSTM,
sequence 80, batch 1, input and hidden 256, float32.

Printed: one JSON line (rank 0).  ``value`` is whole-job GFLOP/s of
algorithmic work (projection 2*S*N*I*G*H*D + recurrence 2*sum(len)*G*H*H*D);
``us_per_step`` is the layer time divided by the sequence length.  L2 is
flushed (a 256 MiB write) between timed layer runs; each run is timed with
CUDA events on the launching stream.  ``roofline`` describes the dominant
kernel, timed live with events the library records around its launches.

``--impl reference`` times the CPU oracle instead (the slow, plain double
precision definition) on bounded samples of the same workload.
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "recurrent layer µs/step and GFLOP/s at 1 GB300; achieved fraction of roofline"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "sm_max_mhz": 2070.0}
# the pages' own figure for the default workload (other hardware: context, not the target)
PAGES_LAYER_MS = {"bilstm_s80_b1_i256_h256_f32": (0.7, "RTX 4070, Vulkan, one dispatch per step")}


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--workload", default=None)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=12.0, help="seconds of oracle work for cpu_baseline")
    ap.add_argument("--e2e-steps", type=int, default=None)
    ap.add_argument("--no-sub", action="store_true", help="measure the headline workload only")
    ap.add_argument("--sub-cpu-budget", type=float, default=2.0,
                    help="seconds of oracle work for each other workload's cpu_baseline")
    ap.add_argument("--seq-cut", type=int, default=None,
                    help="profiling aid: the workload with its sequence cut to this many steps (workload name gets "
                         "a _seqN suffix; not the headline configuration)")
    return ap.parse_args()


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ---------------------------------------------------------------- distributed helpers

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def dist_init(world, backend):
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        os.environ.setdefault("MASTER_PORT", "29531")
        dist.init_process_group(backend=backend)
    return dist


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int, device=None) -> float:
    """Maximum of a per-rank float over all ranks (identity for one rank)."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x: float, world: int, device=None) -> float:
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# ---------------------------------------------------------------- clocks

class ClockSampler:
    """SM clock and clock-event reasons sampled every ~2 ms on a thread while
    the benchmark runs, through NVML's read-only queries (libnvidia-ml, loaded
    with ctypes); nvidia-smi polling every 200 ms where NVML cannot be loaded.
    ``mark()`` opens a named window (a timed region) and ``window(name)``
    summarises the samples taken inside it."""
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
               0x80: "hw_power_brake_slowdown"}
    FIELDS = ("index,uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid=None, period_s=0.002):
        self.uuid = str(uuid) if uuid is not None else None
        self.period = period_s
        self.samples = []          # (t, sm_mhz, reasons bitmask)
        self.windows = {}          # name -> [t0, t1]
        self.sm_max = None
        self.source = None
        self._stop = None
        self._thread = None
        self._proc = None

    def _nvml(self):
        import ctypes
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        h = ctypes.c_void_p()
        ok = False
        if self.uuid:
            u = self.uuid if self.uuid.startswith("GPU-") else "GPU-" + self.uuid
            ok = lib.nvmlDeviceGetHandleByUUID(u.encode(), ctypes.byref(h)) == 0
        if not ok:
            idx = int((os.environ.get("CUDA_VISIBLE_DEVICES") or "0").split(",")[0] or 0)
            if lib.nvmlDeviceGetHandleByIndex_v2(idx, ctypes.byref(h)) != 0:
                raise OSError("no NVML device handle")
        mx = ctypes.c_uint()
        if lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:  # 1: SM clock domain
            self.sm_max = float(mx.value)
        reasons_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            lib.nvmlDeviceGetCurrentClocksThrottleReasons
        return lib, h, reasons_fn

    def start(self):
        import threading
        try:
            import ctypes
            lib, h, reasons_fn = self._nvml()
            self.source = "nvml, %.0f ms" % (self.period * 1e3)
            self._stop = threading.Event()

            def run():
                clk, rs = ctypes.c_uint(), ctypes.c_ulonglong()
                while not self._stop.is_set():
                    a = lib.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(clk))
                    b = reasons_fn(h, ctypes.byref(rs))
                    if a == 0:
                        self.samples.append((time.perf_counter(), float(clk.value), int(rs.value) if b == 0 else 0))
                    self._stop.wait(self.period)
            self._thread = threading.Thread(target=run, daemon=True)
            self._thread.start()
        except (OSError, AttributeError):
            self._start_smi()
        time.sleep(0.05)

    def _start_smi(self):
        self.source = "nvidia-smi, 200 ms"
        try:
            self._proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                           "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self._proc = None
        self._t0 = time.perf_counter()
        time.sleep(0.3)

    def mark(self, name):
        self.windows[name] = [time.perf_counter(), None]

    def end(self, name):
        self.windows[name][1] = time.perf_counter()

    def stop(self):
        if self._thread is not None:
            time.sleep(2 * self.period)
            self._stop.set()
            self._thread.join(timeout=2)
        elif self._proc is not None:
            time.sleep(0.25)
            self._proc.terminate()
            try:
                out, _ = self._proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self._proc.kill()
                out, _ = self._proc.communicate()
            rows = [[p.strip() for p in line.split(",")] for line in out.splitlines()]
            rows = [r for r in rows if len(r) >= 10]
            mine = [r for r in rows if self.uuid and self.uuid in r[1]]
            rows = mine or [r for r in rows if rows and r[0] == rows[0][0]]
            bits = {6: 0x8, 7: 0x40, 8: 0x20, 9: 0x4}
            t = self._t0
            for r in rows:
                t += 0.2
                try:
                    sm = float(r[2])
                    self.sm_max = float(r[3])
                except ValueError:
                    continue
                self.samples.append((t, sm, sum(b for i, b in bits.items() if r[i].lower() == "active")))

    def window(self, name=None):
        """Clock record of the samples inside window `name` (all samples when
        None or when the window caught fewer than 3): median SM clock of the
        samples under load (at least half the highest clock seen), max clock,
        the clock-event reasons seen, sample counts."""
        sel = self.samples
        scope = "whole run"
        if name in self.windows and self.windows[name][1] is not None:
            t0, t1 = self.windows[name]
            inside = [x for x in self.samples if t0 <= x[0] <= t1]
            if len(inside) >= 3 or self._thread is None:
                sel, scope = inside, "timed region"
        if not sel:
            return {"sm_mhz": None, "sm_max_mhz": self.sm_max, "reasons": ["no samples"], "samples": 0,
                    "source": self.source}
        sm = [x[1] for x in sel]
        hi = max(sm)
        load = [v for v in sm if v >= 0.5 * hi] or sm
        mask = 0
        for x in sel:
            mask |= x[2]
        reasons = sorted(v for b, v in self.REASONS.items() if mask & b)
        return {"sm_mhz": statistics.median(load), "sm_max_mhz": self.sm_max, "reasons": reasons,
                "samples": len(sel), "samples_under_load": len(load), "scope": scope, "source": self.source}


# ---------------------------------------------------------------- launch latency

def empty_launch_us(dev, stream, n=400):
    """Device time per launch of a 1-element kernel issued back to back on
    the stream: from the host one by one ("stream"), and replayed from a CUDA
    graph ("graph", no host in the way).  A design with one launch per
    recurrent step pays at least this per step."""
    import torch
    x = torch.zeros(1, device=dev)
    out = {"stream": None, "graph": None}
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        for _ in range(20):
            x.add_(1.0)
        torch.cuda.synchronize(dev)
        e0.record(stream)
        for _ in range(n):
            x.add_(1.0)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        out["stream"] = e0.elapsed_time(e1) * 1e3 / n
    try:
        g = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream(dev)
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            x.add_(1.0)  # warm-up on the capture stream
            torch.cuda.synchronize(dev)
            with torch.cuda.graph(g, stream=side):
                for _ in range(n):
                    x.add_(1.0)
        torch.cuda.synchronize(dev)
        g.replay()
        torch.cuda.synchronize(dev)
        e0.record(stream)
        with torch.cuda.stream(stream):
            g.replay()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        out["graph"] = e0.elapsed_time(e1) * 1e3 / n
    except RuntimeError:
        pass
    return out


# ---------------------------------------------------------------- peaks measured in the run

def measure_fp32_peak(dev, stream):
    """float32 FMA throughput of the SMs: a kernel of independent fused
    multiply-adds only (libfmapeak.so, built next to the library), 8 blocks
    of 256 threads per SM, best of 10 launches timed with CUDA events on the
    launching stream.  Returns TFLOP/s."""
    import ctypes
    import torch
    from onnx_lstm_gru_gb300 import _build
    lib = ctypes.CDLL(_build.PROBE_LIB)
    lib.rk_probe_fma_flops.restype = ctypes.c_double
    lib.rk_probe_fma_flops.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int]
    lib.rk_probe_fma_launch.restype = ctypes.c_int
    lib.rk_probe_fma_launch.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_void_p]
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    blocks, threads, iters = sms * 8, 256, 2048
    out = torch.empty(blocks * threads, dtype=torch.float32, device=dev)
    flops = lib.rk_probe_fma_flops(blocks, threads, iters)
    best = None
    for i in range(13):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        rc = lib.rk_probe_fma_launch(out.data_ptr(), blocks, threads, iters, stream.cuda_stream)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        if rc != 0:
            raise RuntimeError(f"FMA peak probe launch failed: cudaError {rc}")
        if i >= 3:
            ms = e0.elapsed_time(e1)
            best = ms if best is None else min(best, ms)
    return flops / (best * 1e-3) / 1e12


def measure_tensor_peak(dev, stream, dtype):
    """Dense tensor-core throughput of torch.matmul at 8192^3 (2 * 8192^3
    FLOPs) in `dtype`, best of 10 after 3 warm-ups, CUDA events on the
    stream: the same recipe as the driver's measured bf16 peak."""
    import torch
    n = 8192
    with torch.cuda.stream(stream):
        a = torch.randn(n, n, device=dev).to(dtype)
        b = torch.randn(n, n, device=dev).to(dtype)
        best = None
        for i in range(13):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            c = a @ b
            e1.record(stream)
            torch.cuda.synchronize(dev)
            if i >= 3:
                ms = e0.elapsed_time(e1)
                best = ms if best is None else min(best, ms)
        del a, b, c
    return 2.0 * n ** 3 / (best * 1e-3) / 1e12


# ---------------------------------------------------------------- profile summaries

# Source files of each kernel, hashed so a committed ncu summary is only used
# while the kernel it measured is unchanged.
KERNEL_SOURCES = {
    "fast": ("step_kernel", ("rk_elem.cuh", "rk_step_common.cuh", "rk_step_fast.cuh")),
    "cluster": ("step_cluster_kernel", ("rk_elem.cuh", "rk_step_common.cuh", "rk_step.cuh", "rk_step_launch.cuh")),
    "grid": ("step_grid_kernel", ("rk_elem.cuh", "rk_step_common.cuh", "rk_step.cuh", "rk_step_launch.cuh")),
    "tensor": ("step_tc_kernel", ("rk_elem.cuh", "rk_step_common.cuh", "rk_proj_tc.cuh", "rk_step_tc.cuh",
                                  "rk_step_tc.cu", "rk_step_tc_pair.cu", "rk_step_tc_cluster.cu")),
    "tensor_small": ("step_tcs_kernel", ("rk_elem.cuh", "rk_step_common.cuh", "rk_step_tc.cuh", "rk_step_tcs.cuh",
                                         "rk_step_tcs.cu")),
    "proj_tc": ("proj_tc_kernel", ("rk_elem.cuh", "rk_proj_tc.cuh", "rk_proj_tc.cu")),
    "proj_simt": ("projection", ("rk_elem.cuh", "rk_proj.cu")),
}


def kernel_source_hash(files):
    h = hashlib.sha256()
    for name in files:
        with open(os.path.join(ROOT, "onnx_lstm_gru_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def step_kernel_source_hash():
    return kernel_source_hash(KERNEL_SOURCES["fast"][1])


def plan_fields(plan: str) -> dict:
    """'proj=tc step=tensor shape=..' -> {'proj': 'tc', 'step': 'tensor', ...}"""
    return dict(kv.split("=", 1) for kv in plan.split() if "=" in kv)


def profiled_traffic(kernel: str, workload: str, source_hash: str):
    """DRAM bytes per launch of `kernel` on `workload` from the committed ncu
    summary, or None if there is none or the kernel source changed since."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.md")
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", text)
    hs = re.search(r"source_hash:\s*([0-9a-f]+)", text)
    if not m or not hs or hs.group(1) != source_hash:
        return None
    return float(m.group(1))


def kernel_roofline(kind: str, flops: float, ms: float, peaks: dict, workload: str, dtype: str) -> dict:
    """Roofline entry of one kernel: tcgen05 kernels against the measured
    dense tensor rate of their operand type (fp16 or bf16), float32 SIMT
    kernels (and 16-bit layers on SIMT kernels, whose arithmetic is float32)
    against the measured float32 FMA rate."""
    achieved = flops / (ms * 1e-3) / 1e12 if ms > 0 else 0.0
    name, files = KERNEL_SOURCES[kind]
    traffic = profiled_traffic(name, workload, kernel_source_hash(files))
    if kind in ("tensor", "tensor_small", "proj_tc"):
        key = "bf16" if dtype == "bf16" else "f16"
        peak, src = peaks[key]
        return {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
                "traffic": traffic, "kernel": name, "peak_source": src}
    peak, src = peaks["f32"]
    return {"bound": "alu", "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
            "traffic": traffic, "kernel": name, "peak_source": src}


# ---------------------------------------------------------------- CPU oracle timing

def make_oracle_sampler(w):
    """Return sample(seq_cut) -> (seconds, algorithmic flops): one single-
    threaded oracle run on the workload with its sequence cut to seq_cut steps
    (and, for batches above 8, batch row 0 only), all directions."""
    import numpy as np
    import oracle
    from onnx_lstm_gru_gb300 import Problem, workloads
    pr = w.problem
    inp = workloads.make_inputs(w)
    rows = list(range(pr.batch)) if pr.batch <= 8 else [0]

    def sample(seq_cut):
        sub = Problem(pr.cell, seq=seq_cut, batch=len(rows), input=pr.input, hidden=pr.hidden,
                      direction=pr.direction, dtype=pr.dtype, layout=pr.layout, clip=pr.clip,
                      input_forget=pr.input_forget, linear_before_reset=pr.linear_before_reset,
                      activations=pr.activations)
        a = {}
        for k, v in inp.items():
            v = v.astype(np.float64) if k != "sequence_lens" else v
            if k == "X":
                v = v[:seq_cut][:, rows] if pr.layout == 0 else v[rows][:, :seq_cut]
            elif k in ("initial_h", "initial_c"):
                v = v[:, rows] if pr.layout == 0 else v[rows]
            elif k == "sequence_lens":
                v = np.minimum(v[rows], seq_cut).astype(np.int32)
            a[k] = np.ascontiguousarray(v)
        spec = dict(cell=sub.cell, direction=sub.direction, layout=sub.layout, seq=sub.seq, batch=sub.batch,
                    input=sub.input, hidden=sub.hidden, clip=sub.clip, input_forget=sub.input_forget,
                    linear_before_reset=sub.linear_before_reset,
                    activations=list(sub.activations) if sub.activations else None)
        t0 = time.perf_counter()
        oracle.layer(spec, **a)
        dt = time.perf_counter() - t0
        return dt, workloads.algorithmic_flops(sub, a.get("sequence_lens"))

    sample.rows = rows
    return sample


def seq_cut_for(sample, w, seconds):
    """Steps of the sequence that one oracle sample may take to last about
    `seconds` (calibrated on a one-step run)."""
    dt1, _ = sample(1)
    return int(max(1, min(w.problem.seq, seconds / max(dt1, 1e-6))))


def oracle_sample_rate(w, budget_s: float):
    """Oracle GFLOP/s on bounded samples of w for about budget_s seconds."""
    sample = make_oracle_sampler(w)
    seq_cut = seq_cut_for(sample, w, budget_s / 4)
    total_t, total_f, n = 0.0, 0.0, 0
    while total_t < budget_s and n < 1000:
        dt, fl = sample(seq_cut)
        total_t += dt
        total_f += fl
        n += 1
    pr = w.problem
    desc = (f"{n} oracle runs of the workload cut to {seq_cut} of {pr.seq} steps, "
            f"{len(sample.rows)} of {pr.batch} batch rows, all directions; {total_t:.1f} s")
    return total_f / total_t / 1e9, desc


# ---------------------------------------------------------------- the GPU arm

# the other layer shapes of the benchmark's configuration list, each measured
# in the same run as a record of its own (the line's config stays the headline)
SUB_WORKLOADS = ["lstm_fwd_s8_b1_i16_h16_f32", "bigru_s128_b8_i512_h512_f16_lbr0",
                 "bigru_s128_b8_i512_h512_f16_lbr1", "revlstm_peep_clip_s200_b4_i128_h1024_f32",
                 "bilstm_s512_b64_i1024_h1024_f16"]
L2_NOTE = "GPU arm: L2 flushed between timed layer runs (256 MiB write, untimed)"


def config_of(name, pr, world):
    """The config object of both arms' JSON lines (same keys and values)."""
    return {"workload": name, "cell": pr.cell, "direction": pr.direction, "seq": pr.seq, "batch": pr.batch,
            "input": pr.input, "hidden": pr.hidden, "layout": pr.layout, "tensor_dtype": pr.dtype,
            "l2": L2_NOTE, "parallelism": f"replicas x{world}"}


class Measured:
    """One workload measured on the GPU: the timed layer runs, the per-kernel
    durations, the algorithmic work and the clocks seen meanwhile (the
    window spans the timed runs and the kernel-timing runs of the same
    layer); rooflines are attached once the peaks are known."""


def measure_workload(rk, workloads, name, w, steps, warmup, n_prof, dev, stream, flush, sampler, world, keep=False):
    import numpy as np
    import torch
    pr = w.problem
    inp = workloads.make_inputs(w)
    tdt = rk.torch_dtype(pr.dtype)

    def host_tensor(k, v):
        # bfloat16 inputs arrive as float32 arrays of bfloat16 numbers: exact cast
        t = torch.from_numpy(v)
        return t if k == "sequence_lens" else t.to(tdt)

    dev_in = {k: host_tensor(k, v).to(dev) for k, v in inp.items()}
    shp = pr.shapes()
    outs = {n: torch.empty(shp[n], dtype=tdt, device=dev) for n in w.outputs if not (n == "Y_c" and pr.cell != "lstm")}
    layer = rk.RecurrentLayer()
    plan = layer.plan(pr)

    def run_once():
        layer.encode(pr, stream=stream, **dev_in, **outs)

    for _ in range(max(3, warmup)):
        flush.zero_()
        run_once()
    torch.cuda.synchronize()
    layer.poll(stream)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    launches0 = layer.launches()
    barrier(world)
    torch.cuda.synchronize()
    sampler.mark(name)
    for i in range(steps):
        flush.zero_()
        starts[i].record(stream)
        run_once()
        ends[i].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    launches = layer.launches() - launches0
    layer.poll(stream)
    times = [s_.elapsed_time(e) for s_, e in zip(starts, ends)]
    ms_local = sum(times) / len(times)
    ms = max_over_ranks(ms_local, world, dev)

    # per-kernel durations (events recorded by the library around its launches)
    rk.rk_set_profiling(layer.handle, True)
    kproj, kstep = [], []
    for _ in range(n_prof):
        flush.zero_()
        run_once()
        a, b = rk.rk_last_timings(layer.handle)
        kproj.append(a)
        kstep.append(b)
    rk.rk_set_profiling(layer.handle, False)
    sampler.end(name)  # the clock window covers the timed runs and these
    m = Measured()
    m.name, m.w, m.pr, m.inp, m.plan = name, w, pr, inp, plan
    m.ms_local, m.ms, m.launches, m.steps = ms_local, ms, launches, steps
    m.proj_ms = statistics.mean(kproj) if kproj and kproj[0] >= 0 else 0.0
    m.step_ms = statistics.mean(kstep)
    m.flops = workloads.algorithmic_flops(pr, inp.get("sequence_lens"))
    D, G, H = pr.num_directions, pr.gates, pr.hidden
    lens = inp.get("sequence_lens")
    tot_len = pr.seq * pr.batch if lens is None else int(np.clip(lens, 0, pr.seq).sum())
    m.step_flops = 2.0 * tot_len * G * H * H * D
    m.proj_flops = 2.0 * pr.seq * pr.batch * pr.input * G * H * D
    if m.proj_ms <= 0.0:  # projection computed inside the step kernel's launch
        m.step_flops += m.proj_flops
    pf = plan_fields(plan)
    m.step_kind = pf.get("step", "fast")
    if m.step_kind == "tensor" and pf.get("variant") == "small":
        m.step_kind = "tensor_small"
    m.proj_kind = "proj_tc" if pf.get("proj") == "tc" else "proj_simt"
    m.cbytes = workloads.compulsory_bytes(pr, {**inp, **{n: None for n in outs}})
    m.clocks = sampler.window(name)
    if keep:
        m.layer, m.dev_in, m.outs, m.host_tensor = layer, dev_in, outs, host_tensor
    else:
        layer.close()
        del dev_in, outs
    return m


def rooflines(m, peaks, hbm_gbs, peak_src):
    """(roofline of the dominant kernel with the other kernel under
    'others', whole-layer roofline) of a measured workload."""
    r_step = kernel_roofline(m.step_kind, m.step_flops, m.step_ms, peaks, m.name, m.pr.dtype)
    r_proj = kernel_roofline(m.proj_kind, m.proj_flops, m.proj_ms, peaks, m.name, m.pr.dtype) \
        if m.proj_ms > 0 else None
    dom = r_step if (r_proj is None or m.step_ms >= m.proj_ms) else r_proj
    dom = dict(dom, others=[r for r in (r_step, r_proj) if r is not None and r is not dom])
    # whole layer: max(FLOPs at the peak of the unit each kernel runs on,
    # compulsory bytes at HBM bandwidth) / measured layer time
    t_flops = m.step_flops / (r_step["peak"] * 1e12) + (m.proj_flops / (r_proj["peak"] * 1e12) if r_proj else 0.0)
    t_bytes = m.cbytes / (hbm_gbs * 1e9)
    layer = {"t_roofline_us": max(t_flops, t_bytes) * 1e6, "t_measured_us": m.ms_local * 1e3,
             "frac": max(t_flops, t_bytes) / (m.ms_local * 1e-3), "flops": m.flops, "compulsory_bytes": m.cbytes,
             "hbm_gbs": hbm_gbs, "hbm_source": peak_src}
    return dom, layer


def sub_record(m, peaks, hbm_gbs, peak_src, world, cpu):
    dom, layer = rooflines(m, peaks, hbm_gbs, peak_src)
    return {"config": config_of(m.name, m.pr, world), "plan": m.plan, "steps": m.steps, "ms_per_layer": m.ms,
            "us_per_step": m.ms * 1e3 / max(m.pr.seq, 1), "steps_per_s": m.pr.seq / (m.ms * 1e-3) * world,
            "gflops": m.flops * world / (m.ms * 1e-3) / 1e9,
            "kernels_ms": {"projection": m.proj_ms, "step": m.step_ms}, "roofline": dom, "layer_roofline": layer,
            "clocks": m.clocks, "gpu_launches": m.launches, "cpu_baseline": cpu}


def run_gb300(args):
    import torch
    import onnx_lstm_gru_gb300 as rk
    from onnx_lstm_gru_gb300 import workloads

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dist_init(world, "nccl")
    dev = torch.device("cuda", local)
    rk.build()
    name = args.workload or workloads.HEADLINE
    w = workloads.WORKLOADS[name]
    if args.seq_cut:
        w = dataclasses.replace(w, problem=dataclasses.replace(w.problem, seq=min(args.seq_cut, w.problem.seq)))
        name = f"{name}_seq{w.problem.seq}"
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    sampler = ClockSampler(getattr(torch.cuda.get_device_properties(dev), "uuid", None))
    sampler.start()

    # the headline workload: the line's value
    # 200 kernel-timing runs: with them the headline's clock window holds
    # enough samples even when the timed runs take a few milliseconds
    main = measure_workload(rk, workloads, name, w, args.steps, args.warmup, 200, dev, stream, flush, sampler,
                            world, keep=True)
    pr, inp, layer = main.pr, main.inp, main.layer
    total_flops = sum_over_ranks(main.flops, world, dev)
    gflops = total_flops / (main.ms * 1e-3) / 1e9

    # e2e through the host-buffer entry point (copies inside the timed region)
    tdt = rk.torch_dtype(pr.dtype)
    shp = pr.shapes()
    n_e2e = args.e2e_steps or max(3, min(args.steps, 300))
    pinned_in = {}
    for k, v in inp.items():
        hv = main.host_tensor(k, v)
        t = torch.empty(hv.shape, dtype=hv.dtype, pin_memory=True)
        t.copy_(hv)
        pinned_in[k] = t
    pinned_out = {n: torch.empty(shp[n], dtype=tdt, pin_memory=True) for n in main.outs}
    h2d = sum(t.numel() * t.element_size() for t in pinned_in.values())
    d2h = sum(t.numel() * t.element_size() for t in pinned_out.values())
    for _ in range(3):
        layer.encode_host(pr, stream=stream, **pinned_in, **pinned_out)
    barrier(world)
    t0 = time.perf_counter()
    for _ in range(n_e2e):
        layer.encode_host(pr, stream=stream, **pinned_in, **pinned_out)
    e2e_s = (time.perf_counter() - t0) / n_e2e
    e2e_s = max_over_ranks(e2e_s, world, dev)
    e2e_gflops = total_flops / e2e_s / 1e9
    layer.close()
    del main.dev_in, main.outs

    # the other configurations, one record each
    subs = []
    if not args.no_sub and not args.seq_cut:
        sub_steps = max(1, min(args.steps, 50))
        for sname in SUB_WORKLOADS:
            if sname == name:
                continue
            subs.append(measure_workload(rk, workloads, sname, workloads.WORKLOADS[sname], sub_steps,
                                         max(3, min(args.warmup, 5)), max(10, min(sub_steps, 20)), dev, stream,
                                         flush, sampler, world))
    launch_us = empty_launch_us(dev, stream)

    # peaks measured in this run: the float32 FMA rate and the dense fp16
    # tensor rate; dense bf16 from the driver's measurement
    file_peaks, file_src = load_peaks()
    sampler.mark("fp32_peak")
    fp32 = measure_fp32_peak(dev, stream)
    sampler.end("fp32_peak")
    sampler.mark("f16_peak")
    f16 = measure_tensor_peak(dev, stream, torch.float16)
    sampler.end("f16_peak")
    sampler.stop()
    peaks = {"f32": (fp32, "measured in this run: float32 FMA kernel, best of 10"),
             "f16": (f16, "measured in this run: torch.matmul fp16 8192^3, best of 10"),
             "bf16": (float(file_peaks["bf16_tflops"]), f"{file_src}: dense bf16 burst (MEASURED_PEAKS.json)")}
    hbm_gbs = float(file_peaks["hbm_gbs"])
    peaks_rec = {"fp32_tflops": fp32, "fp32_clocks": sampler.window("fp32_peak"), "f16_tflops": f16,
                 "f16_clocks": sampler.window("f16_peak"), "bf16_tflops": peaks["bf16"][0],
                 "hbm_gbs": hbm_gbs, "source": {k: v[1] for k, v in peaks.items()}}

    roofline, layer_roofline = rooflines(main, peaks, hbm_gbs, file_src)
    cpu = None
    sub_cpu = {}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        rate, desc = oracle_sample_rate(w, args.cpu_budget)
        cpu = {"value": rate, "unit": "GFLOP/s", "cores": 1, "kind": "oracle", "sample": desc}
        for m in subs:
            r, d = oracle_sample_rate(m.w, args.sub_cpu_budget)
            sub_cpu[m.name] = {"value": r, "unit": "GFLOP/s", "cores": 1, "kind": "oracle", "sample": d}

    vs = None
    if name in PAGES_LAYER_MS:
        pages_ms, _ = PAGES_LAYER_MS[name]
        vs = gflops / (main.flops / (pages_ms * 1e-3) / 1e9)

    line = {
        "metric": METRIC, "value": gflops, "unit": "GFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": main.ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": vs, "dtype": "f32" if pr.dtype == "f32" else f"{pr.dtype} storage, f32 arithmetic",
        "data": "synthetic (seeded numpy PCG64, random weights)",
        "config": config_of(name, pr, world), "plan": main.plan,
        "us_per_step": main.ms * 1e3 / max(pr.seq, 1), "steps_per_s": pr.seq / (main.ms * 1e-3) * world,
        "kernels_ms": {"projection": main.proj_ms, "step": main.step_ms},
        "roofline": roofline, "layer_roofline": layer_roofline, "cpu_baseline": cpu,
        "e2e": {"value": e2e_gflops, "unit": "GFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": e2e_s * 1e3,
                "transfer": "pinned host buffers through rk_encode_host: X and W copied, the other inputs read "
                            "and the outputs written in place by the step kernel over the CPU-GPU link"},
        "clocks": main.clocks, "gpu_launches": main.launches,
        "peaks": peaks_rec,
        # the other configurations of the benchmark list, measured in this run
        "workloads": {m.name: sub_record(m, peaks, hbm_gbs, file_src, world, sub_cpu.get(m.name)) for m in subs},
        # what one dependent launch per step would cost at least on this machine
        # (a 1-element kernel back to back on the stream), next to us_per_step
        "empty_launch_us": launch_us,
    }
    if vs is not None:
        line["vs_baseline_note"] = "value / the pages' %.1f ms layer on %s (other hardware: context)" % PAGES_LAYER_MS[name]
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# ---------------------------------------------------------------- the reference arm (CPU oracle)

def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    from onnx_lstm_gru_gb300 import workloads
    import oracle
    oracle.build()
    name = args.workload or workloads.HEADLINE
    w = workloads.WORKLOADS[name]
    n_total = args.steps + args.warmup
    sample = make_oracle_sampler(w)
    # each step is one oracle sample sized so that W + K of them take ~2.5 min
    seq_cut = seq_cut_for(sample, w, max(0.005, 150.0 / max(n_total, 1)))
    times, flops = [], []
    for i in range(n_total):
        dt, fl = sample(seq_cut)
        if i >= args.warmup:
            times.append(dt)
            flops.append(fl)
    value = sum(flops) / sum(times) / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * sum(times) / len(times),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded numpy PCG64, random weights)", "config": config_of(name, w.problem, world),
            "cpu_baseline": {"value": value, "unit": "GFLOP/s", "cores": 1, "kind": "oracle",
                             "sample": (f"each step: one oracle run of the workload cut to {seq_cut} of "
                                        f"{w.problem.seq} steps, {len(sample.rows)} of {w.problem.batch} rows")},
            "e2e": {"value": value, "unit": "GFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gb300(args)


if __name__ == "__main__":
    main()
