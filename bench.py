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
    """nvidia-smi sampled every 200 ms while the timed region runs."""
    FIELDS = ("index,uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid=None):
        self.uuid = str(uuid) if uuid is not None else None
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = []
        for line in out.splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 10:
                rows.append(parts)
        mine = [r for r in rows if self.uuid and self.uuid in r[1]]
        if mine:
            rows = mine
        elif len({r[0] for r in rows}) > 1:
            rows = [r for r in rows if r[0] == rows[0][0]]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        sm = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        mx = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[6 + i].lower() == "active"})
        # "under load": samples at or above half the highest clock seen
        hi = max(sm) if sm else 0.0
        load = [v for v in sm if v >= 0.5 * hi] or sm
        return {"sm_mhz": statistics.median(load) if load else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


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


# ---------------------------------------------------------------- profile summaries

# Source files of each kernel, hashed so a committed ncu summary is only used
# while the kernel it measured is unchanged.
KERNEL_SOURCES = {
    "fast": ("step_kernel", ("rk_elem.cuh", "rk_step.cuh", "rk_step_fast.cuh", "rk_step_launch.cuh")),
    "cluster": ("step_cluster_kernel", ("rk_elem.cuh", "rk_step.cuh", "rk_step_launch.cuh")),
    "grid": ("step_grid_kernel", ("rk_elem.cuh", "rk_step.cuh", "rk_step_launch.cuh")),
    "tensor": ("step_tc_kernel", ("rk_elem.cuh", "rk_step.cuh", "rk_proj_tc.cuh", "rk_step_tc.cuh", "rk_step_tc.cu",
                                  "rk_step_tc_pair.cu", "rk_step_tc_cluster.cu")),
    "tensor_small": ("step_tcs_kernel", ("rk_elem.cuh", "rk_step.cuh", "rk_step_tc.cuh", "rk_step_tcs.cuh",
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


def kernel_roofline(kind: str, flops: float, ms: float, peaks: dict, alu_peak: float, alu_src: str,
                    workload: str) -> dict:
    """Roofline entry of one kernel: tensor-core kernels against the measured
    dense bf16 rate (fp16 has the same nominal dense rate), FP32 SIMT kernels
    against the FP32 FMA rate derived from the SM count and clock."""
    fp16 = "_f16" in workload
    achieved = flops / (ms * 1e-3) / 1e12 if ms > 0 else 0.0
    name, files = KERNEL_SOURCES[kind]
    traffic = profiled_traffic(name, workload, kernel_source_hash(files))
    if kind in ("tensor", "tensor_small", "proj_tc"):
        peak = float(peaks["bf16_tflops"])
        return {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
                "traffic": traffic, "kernel": name,
                "peak_source": "measured dense bf16 burst" +
                               ("; fp16 runs at the same nominal dense rate" if fp16 else "")}
    return {"bound": "alu", "achieved": achieved, "peak": alu_peak, "unit": "TFLOP/s", "frac": achieved / alu_peak,
            "traffic": traffic, "kernel": name, "peak_source": alu_src}


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

def run_gb300(args):
    import numpy as np
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
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    plan = layer.plan(pr)

    def run_once():
        layer.encode(pr, stream=stream, **dev_in, **outs)

    for _ in range(max(3, args.warmup)):
        flush.zero_()
        run_once()
    torch.cuda.synchronize()
    layer.poll(stream)

    sampler = ClockSampler(getattr(torch.cuda.get_device_properties(dev), "uuid", None))
    if rank == 0:
        sampler.start()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    launches0 = layer.launches()
    barrier(world)
    torch.cuda.synchronize()
    for i in range(args.steps):
        flush.zero_()
        starts[i].record(stream)
        run_once()
        ends[i].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    launches = layer.launches() - launches0
    clocks = sampler.stop() if rank == 0 else None
    layer.poll(stream)
    times = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    ms_local = sum(times) / len(times)
    ms = max_over_ranks(ms_local, world, dev)
    flops = workloads.algorithmic_flops(pr, inp.get("sequence_lens"))
    total_flops = sum_over_ranks(flops, world, dev)
    gflops = total_flops / (ms * 1e-3) / 1e9

    # per-kernel durations (events recorded by the library around its launches)
    rk.rk_set_profiling(layer.handle, True)
    kproj, kstep = [], []
    for _ in range(max(20, min(args.steps, 200))):
        flush.zero_()
        run_once()
        a, b = rk.rk_last_timings(layer.handle)
        kproj.append(a)
        kstep.append(b)
    rk.rk_set_profiling(layer.handle, False)
    proj_ms = statistics.mean(kproj) if kproj and kproj[0] >= 0 else 0.0
    step_ms = statistics.mean(kstep)

    # e2e through the host-buffer entry point (copies inside the timed region)
    n_e2e = args.e2e_steps or max(3, min(args.steps, 300))
    pinned_in = {}
    for k, v in inp.items():
        hv = host_tensor(k, v)
        t = torch.empty(hv.shape, dtype=hv.dtype, pin_memory=True)
        t.copy_(hv)
        pinned_in[k] = t
    pinned_out = {n: torch.empty(shp[n], dtype=tdt, pin_memory=True) for n in outs}
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

    peaks, peak_src = load_peaks()
    sm_count = torch.cuda.get_device_properties(dev).multi_processor_count
    sm_max = float(peaks.get("sm_max_mhz", 2070.0))
    alu_peak_tflops = sm_count * 128 * 2 * sm_max * 1e6 / 1e12  # FP32 FMA lanes x 2 x max clock
    D, G, H = pr.num_directions, pr.gates, pr.hidden
    lens = inp.get("sequence_lens")
    import numpy as _np
    tot_len = pr.seq * pr.batch if lens is None else int(_np.clip(lens, 0, pr.seq).sum())
    step_flops = 2.0 * tot_len * G * H * H * D
    proj_flops = 2.0 * pr.seq * pr.batch * pr.input * G * H * D
    if proj_ms <= 0.0:  # projection fused into the step kernel
        step_flops += proj_flops
    pf = plan_fields(plan)
    alu_src = f"derived: {sm_count} SMs x 128 FP32 lanes x 2 x {sm_max:.0f} MHz"
    step_kind = pf.get("step", "fast")
    if step_kind == "tensor" and pf.get("variant") == "small":
        step_kind = "tensor_small"
    proj_kind = "proj_tc" if pf.get("proj") == "tc" else "proj_simt"
    r_step = kernel_roofline(step_kind, step_flops, step_ms, peaks, alu_peak_tflops, alu_src, name)
    r_proj = kernel_roofline(proj_kind, proj_flops, proj_ms, peaks, alu_peak_tflops, alu_src, name) \
        if proj_ms > 0 else None
    roofline = r_step if (r_proj is None or step_ms >= proj_ms) else r_proj
    roofline = dict(roofline, others=[r for r in (r_step, r_proj) if r is not None and r is not roofline])
    # whole-layer roofline: max(FLOPs at peak, compulsory bytes at HBM) / measured time
    cbytes = workloads.compulsory_bytes(pr, {**inp, **{n: None for n in outs}})
    # FLOPs at the peak of the unit each kernel runs on
    t_flops = step_flops / (r_step["peak"] * 1e12) + (proj_flops / (r_proj["peak"] * 1e12) if r_proj else 0.0)
    t_bytes = cbytes / (float(peaks["hbm_gbs"]) * 1e9)
    layer_roofline = {"t_roofline_us": max(t_flops, t_bytes) * 1e6, "t_measured_us": ms_local * 1e3,
                      "frac": max(t_flops, t_bytes) / (ms_local * 1e-3), "flops": flops, "compulsory_bytes": cbytes,
                      "hbm_gbs": float(peaks["hbm_gbs"]), "peak_source": peak_src}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        rate, desc = oracle_sample_rate(w, args.cpu_budget)
        cpu = {"value": rate, "unit": "GFLOP/s", "cores": 1, "kind": "oracle", "sample": desc}

    vs = None
    if name in PAGES_LAYER_MS:
        pages_ms, _ = PAGES_LAYER_MS[name]
        vs = gflops / (flops / (pages_ms * 1e-3) / 1e9)

    launch_us = empty_launch_us(dev, stream)

    line = {
        "metric": METRIC, "value": gflops, "unit": "GFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": vs, "dtype": "f32" if pr.dtype == "f32" else f"{pr.dtype} storage, f32 arithmetic",
        "data": "synthetic (seeded numpy PCG64, random weights)",
        "config": {"workload": name, "cell": pr.cell, "direction": pr.direction, "seq": pr.seq, "batch": pr.batch,
                   "input": pr.input, "hidden": pr.hidden, "layout": pr.layout, "tensor_dtype": pr.dtype,
                   "l2": "flushed between timed layer runs (256 MiB write, untimed)",
                   "parallelism": f"replicas x{world}", "plan": plan},
        "us_per_step": ms * 1e3 / max(pr.seq, 1), "steps_per_s": pr.seq / (ms * 1e-3) * world,
        "kernels_ms": {"projection": proj_ms, "step": step_ms},
        "roofline": roofline, "layer_roofline": layer_roofline, "cpu_baseline": cpu,
        "e2e": {"value": e2e_gflops, "unit": "GFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": e2e_s * 1e3},
        "clocks": clocks, "gpu_launches": launches,
        # what one dependent launch per step would cost at least on this machine
        # (a 1-element kernel back to back on the stream), next to us_per_step
        "empty_launch_us": launch_us,
    }
    if vs is not None:
        line["vs_baseline_note"] = "value / the pages' %.1f ms layer on %s (other hardware: context)" % PAGES_LAYER_MS[name]
    layer.close()
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
            "data": "synthetic (seeded numpy PCG64, random weights)", "config": {"workload": name},
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
