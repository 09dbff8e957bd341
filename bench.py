#!/usr/bin/env python3
"""Benchmark of the block-scaled small-M GEMV on GB300.

Metric: achieved HBM GB/s on cold weights (algorithmic bytes W + scales + zp + A + y per call,
divided by the device time of the call), with microseconds per call and the fraction of the
measured HBM copy bandwidth, against M.

Default workload (one "step" = one pass of the hot path over the workload): the int4
MatMulNBits small-M sweep -- int4 weights, block size 32, zero point fixed at 8, fp16 and bf16
activations, shapes (K x N) 4096x4096, 4096x12288, 12288x4096, 4096x151936, at M = 1, 2, 4, 8
and 16: forty GEMV calls per step, one plan per shape sized for 16 rows.  Calls run M by M over
all shapes, so two calls on one weight are separated by the other shapes' calls (> 3x L2), and
each shape's two weight copies alternate between steps: the weights are cold.  The timed region
replays CUDA graphs holding exactly --steps steps of back-to-back launches (programmatic
dependent launch overlaps each call's start-up with the previous call's tail); separate replays
of a graph with an event between every launch give per-call durations (per_shape, by_M).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--sweep]
                    [--config C]

--config 2 times the int8-with-zero-points workload (M = 1) instead.  With --gpus N > 1
(launched under torchrun) every rank runs the same workload on its own GPU (independent
replicas: the GEMV has no exchange step), the time is the maximum over ranks and the value is
the bytes of all ranks over that time.  --impl reference times the CPU oracle on the host cores
instead.  --sweep prints one JSON line per (configuration shape, M) with isolated-cold and
streamed-cold timings.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

FALLBACK_HBM_GBS = 6800.0
METRIC = "achieved HBM GB/s (cold weights) and µs/call vs M=1..16, fraction of HBM roofline"
WORKLOAD_CONFIG = 3
GRAPH_STEPS = 24  # steps per captured graph: even, so that weight copies alternate across replays


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=24)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--sweep", action="store_true")
    ap.add_argument("--config", type=int, default=WORKLOAD_CONFIG, help=argparse.SUPPRESS)
    ap.add_argument("--M", type=int, default=None, help=argparse.SUPPRESS)
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help=argparse.SUPPRESS)
    ap.add_argument("--skip-cpu", action="store_true", help=argparse.SUPPRESS)
    # --sweep and --one: run the plans as this variant (cuda_core: calls with M <= 8)
    ap.add_argument("--variant", choices=["auto", "mma", "cuda_core"], default="auto",
                    help=argparse.SUPPRESS)
    # one configuration shape by name (see synth.config_shapes), isolated cold calls: for
    # capturing one launch of one kernel under a profiler
    ap.add_argument("--one", default=None, help=argparse.SUPPRESS)
    # --sweep: let each plan measure its candidate geometries first (bsgemv_plan_autotune)
    ap.add_argument("--autotune", action="store_true", help=argparse.SUPPRESS)
    # --sweep: these M values instead of the configuration's (e.g. 17,24,32)
    ap.add_argument("--Ms", default=None, help=argparse.SUPPRESS)
    # --sweep / --one: plans sized for this many rows (default: the configuration's largest M up
    # to 8 for calls with M <= 8, else its largest M)
    ap.add_argument("--plan-max-M", type=int, default=0, help=argparse.SUPPRESS)
    # --sweep: output columns per CTA tile of every plan (64 or 128; 0 = the plan's choice)
    ap.add_argument("--tile-rows", type=int, default=0, help=argparse.SUPPRESS)
    # the dense small-N split-K GEMV against cuBLAS (torch.mm), streamed cold
    ap.add_argument("--dense", action="store_true", help=argparse.SUPPRESS)
    ap.add_argument("--dense-shape", default=None, help=argparse.SUPPRESS)  # "N,K": one shape
    # the fused GEMV against cuBLAS on the already dequantised fp16 weight, M = 1 .. 32
    ap.add_argument("--crossover", action="store_true", help=argparse.SUPPRESS)
    ap.add_argument("--calls", type=int, default=5, help=argparse.SUPPRESS)
    return ap.parse_args()


# ------------------------------------------------------------------------------ environment
def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def init_dist(world, backend):
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend)
    return dist if world > 1 else None


def max_over_ranks(value: float, world: int, device=None) -> float:
    """Max of a float over the ranks (identity for one rank)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def workload_name(config: int, shapes, Ms) -> str:
    """The workload of a configuration named by what it is, with its sizes (both arms)."""
    Ms = [Ms] if isinstance(Ms, int) else list(Ms)
    s0 = shapes[0]
    kind = {"int4": "int4 MatMulNBits GEMV", "int8": "int8 MatMulNBits GEMV",
            "fp8": "FP8 E4M3 block-scaled GEMV", "nvfp4": "NVFP4 GEMV"}[s0.fmt]
    if s0.has_zp:
        kind += " with zero points"
    elif s0.fmt in ("int4", "int8"):
        kind += f" (zero point fixed at {8 if s0.fmt == 'int4' else 128})"
    dims, acts = [], []
    for s in shapes:
        d = f"{s.K}x{s.N} bs{s.block_size}"
        if d not in dims:
            dims.append(d)
        a = "bf16" if s.act == "bf16" else "fp16"
        if a not in acts:
            acts.append(a)
    return (f"{kind}: " + ", ".join(dims) + f" (K x N), M={','.join(str(m) for m in Ms)}, "
            + " and ".join(acts))


def workload_dtype(shapes) -> str:
    """The arithmetic types of the path: stored weight codes, activation type(s), accumulation."""
    s0 = shapes[0]
    w = {"int4": "u4 weights", "int8": "u8 weights", "fp8": "e4m3 weights",
         "nvfp4": "e2m1 weights + e4m3 block scales"}[s0.fmt]
    acts = sorted({"bf16" if s.act == "bf16" else "f16" for s in shapes})
    return f"{w}, {' and '.join(acts)} activations, f32 accumulate"


def job_throughput_gbps(world: int, steps: int, step_bytes: int, seconds: float) -> float:
    """Whole-job GB/s: every rank moves `step_bytes` per step (replicas, weak scaling) and the
    job takes the slowest rank's time."""
    return world * steps * step_bytes / seconds / 1e9


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source_hash() -> str:
    h = hashlib.sha1()
    csrc = os.path.join(ROOT, "block_scaled_bit_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        if name.endswith((".cu", ".cuh", ".h", ".cpp")):
            with open(os.path.join(csrc, name), "rb") as f:
                h.update(name.encode())
                h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on this kernel."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f).get(workload)
        if rec and rec.get("kernel_hash") == kernel_source_hash():
            return float(rec["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 100 ms while running."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        rows = []
        try:
            with open(self.path) as f:
                for line in f:
                    parts = [p.strip() for p in line.split(",")]
                    if len(parts) >= 9 and parts[1].isdigit():
                        rows.append(parts)
            os.unlink(self.path)
        except Exception:
            pass
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        sm = [int(r[1]) for r in rows]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        power = [float(r[3]) for r in rows if r[3].replace(".", "", 1).isdigit()]
        return {"sm_mhz": int(statistics.median(sm)), "sm_max_mhz": int(rows[0][2]),
                "reasons": reasons, "samples": len(rows),
                "power_w_max": max(power) if power else None}


# ------------------------------------------------------------------------------ our arm
class Workload:
    """Plans, device buffers (weight copies) and the call list of one configuration.

    One plan per shape, sized for the largest M the configuration is quoted at (so that every M
    of a shape sums each row in the same order).  One step calls every shape at every M, M in the
    outer loop: two calls on one weight copy are separated by the calls on every other shape
    (with the lm_head shapes among them, hundreds of MB > 3x L2), and a shape's copies alternate
    from step to step, so the weights come from HBM."""

    def __init__(self, config: int, M: int | None, device, copies: int):
        from block_scaled_bit_gb300 import bsgemv, synth
        self.config = config
        self.shapes = synth.config_shapes(config)
        per_shape = []
        for shape in self.shapes:
            Ms = (M,) if M else tuple(shape.Ms)
            case = shape.case(max(Ms))
            plan = bsgemv.Plan(case.fmt, case.act, case.block_size, case.has_zp, case.N, case.K,
                               max(Ms))
            bufs = [bsgemv.upload(case, device) for _ in range(copies)]
            per_shape.append((shape, case, plan, bufs, Ms))
        self.plans = [ps[2] for ps in per_shape]
        self.Ms = sorted({m for ps in per_shape for m in ps[4]})
        self.items = []
        for m in self.Ms:
            for shape, case, plan, bufs, Ms in per_shape:
                if m in Ms:
                    self.items.append({"shape": shape, "case": case, "M": m, "plan": plan,
                                       "bufs": bufs, "bytes": case.algorithmic_bytes(m)})
        self.copies = copies

    @property
    def bytes_per_step(self) -> int:
        return sum(it["bytes"] for it in self.items)

    def launch(self, it, copy, stream=None):
        b = it["bufs"][copy % self.copies]
        M = it["M"]
        it["plan"].run(b.A[:M], b.W, b.scales, b.zp, b.y[:M], M=M, stream=stream)

    def close(self):
        for p in self.plans:
            p.close()


def capture(wl, stream, steps, with_events):
    """CUDA graph of `steps` workload steps (optionally with timing events between launches);
    step s uses weight copy s."""
    import torch
    L = len(wl.items)
    events = None
    if with_events:
        events = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(steps * L + 1)]
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        i = 0
        for s in range(steps):
            for it in wl.items:
                if events:
                    events[i].record(stream)
                    i += 1
                wl.launch(it, s)
        if events:
            events[i].record(stream)
    return graph, events


def graph_plan(steps: int, chunk: int = GRAPH_STEPS):
    """Graph sizes covering exactly `steps` steps: (steps per graph, full replays, remainder)."""
    S = max(1, min(steps, chunk))
    full, rem = divmod(steps, S)
    return S, full, rem


def time_graph(wl, steps, warmup, stream):
    """Time exactly `steps` steps of back-to-back launches, replayed from CUDA graphs (consecutive
    launches overlap start-up and tail through programmatic dependent launch).  Then, outside the
    timed region, replays of a graph with an event between every launch give per-launch
    durations (events serialise the launches).
    Returns (seconds, {item index: [per-launch seconds]}, launches)."""
    import torch
    L = len(wl.items)
    S, full, rem = graph_plan(steps)
    with torch.cuda.stream(stream):
        for s in range(2):                # warm every plan and weight copy outside capture
            for it in wl.items:
                wl.launch(it, s)
        stream.synchronize()
    g_full, _ = capture(wl, stream, S, False)
    g_rem = capture(wl, stream, rem, False)[0] if rem else None
    isteps = 2
    inst, events = capture(wl, stream, isteps, True)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        for _ in range(max(1, -(-warmup // S))):
            g_full.replay()
        stream.synchronize()
        start.record(stream)
        for _ in range(full):
            g_full.replay()
        if g_rem is not None:
            g_rem.replay()
        end.record(stream)
        end.synchronize()
        total = start.elapsed_time(end) / 1e3
        per = {j: [] for j in range(L)}
        for _ in range(5):                # per-launch durations (not part of the timed region)
            inst.replay()
            stream.synchronize()
            for s in range(isteps):
                for j in range(L):
                    i = s * L + j
                    per[j].append(events[i].elapsed_time(events[i + 1]) / 1e3)
    return total, per, steps * L


def streamed_per_item(wl, stream, peak):
    """Per (shape, M) of the workload, outside the timed region: a CUDA graph of back-to-back
    calls of that one item alone, cycling through enough weight copies to exceed 3x L2 (the
    workload's own copies plus more for small shapes), replayed 5 times; the time per call.  This
    is each call's cost with start-up and tail overlapped by the next call, cold weights."""
    import torch
    from block_scaled_bit_gb300 import bsgemv
    l2 = torch.cuda.get_device_properties(stream.device).L2_cache_size
    extra = {}
    out = []
    for it in wl.items:
        case, M, plan = it["case"], it["M"], it["plan"]
        foot = case.algorithmic_bytes(1)
        need = max(1, min(8, -(-3 * l2 // foot)))
        key = it["shape"].name
        if key not in extra:
            extra[key] = [bsgemv.upload(case, stream.device)
                          for _ in range(max(0, need - len(it["bufs"])))]
        bufs = list(it["bufs"]) + extra[key]
        reps = max(len(bufs), 40 // len(bufs) * len(bufs))
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            for b in bufs:
                plan.run(b.A[:M], b.W, b.scales, b.zp, b.y[:M], M=M, stream=stream)
            stream.synchronize()
            with torch.cuda.graph(g, stream=stream):
                for r in range(reps):
                    b = bufs[r % len(bufs)]
                    plan.run(b.A[:M], b.W, b.scales, b.zp, b.y[:M], M=M, stream=stream)
            g.replay()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(5):
                g.replay()
            e1.record(stream)
            e1.synchronize()
        us = e0.elapsed_time(e1) * 1e3 / (5 * reps)
        gbps = it["bytes"] / (us * 1e-6) / 1e9
        out.append({"shape": key, "M": M, "us_per_call": round(us, 3), "GBps": round(gbps, 1),
                    "frac": round(gbps / peak, 4), "bytes": it["bytes"],
                    "weight_copies": len(bufs)})
        del g
    extra.clear()
    torch.cuda.empty_cache()
    return out


def e2e_run(wl, steps, stream):
    """End to end through the library's host-buffer entry point: every call of a step goes
    through bsgemv_run_host_async (its activations copied from pinned host memory into the plan's
    staging buffer, the GEMV, its output copied back to pinned host memory, all enqueued on the
    stream), and the step waits for the stream once, when all results are on the host.  The step
    is captured once per weight copy into a CUDA graph (the calls only enqueue work) and
    replayed.  Weights stay device-resident, as model weights do."""
    import torch
    dev = stream.device
    A_host, y_host = [], []
    for it in wl.items:
        M, case = it["M"], it["case"]
        a = np.ascontiguousarray(case.A[:M]).view(np.int16)
        A_host.append(torch.from_numpy(a).pin_memory())
        y_host.append(torch.empty((M, case.N), dtype=torch.int16).pin_memory())
    h2d = sum(it["M"] * it["case"].K * 2 for it in wl.items)
    d2h = sum(it["M"] * it["case"].N * 2 for it in wl.items)

    def enqueue(s):
        for it, ah, yh in zip(wl.items, A_host, y_host):
            b = it["bufs"][s % wl.copies]
            it["plan"].run_host_async(ah, b.W, b.scales, b.zp, yh, M=it["M"], stream=stream)

    with torch.cuda.stream(stream):
        for s in range(2):                # staging buffers are allocated outside capture
            enqueue(s)
            stream.synchronize()
    graphs = []
    for c in range(wl.copies):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            enqueue(c)
        graphs.append(g)
    with torch.cuda.stream(stream):
        for g in graphs:
            g.replay()
        stream.synchronize()
    for yh in y_host:                     # every output must come back from the timed steps
        yh.fill_(-1)
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    with torch.cuda.stream(stream):
        for s in range(steps):
            graphs[s % len(graphs)].replay()
            stream.synchronize()
    dt = time.perf_counter() - t0
    # the outputs made the round trip: each equals the device run of its call
    with torch.cuda.stream(stream):
        for it, yh in zip(wl.items, y_host):
            b = it["bufs"][(steps - 1) % wl.copies]
            M = it["M"]
            ref = torch.empty_like(b.y[:M])
            it["plan"].run(b.A[:M], b.W, b.scales, b.zp, ref, M=M, stream=stream)
            stream.synchronize()
            if not torch.equal(ref.cpu(), yh):
                raise RuntimeError(f"e2e: host output of {it['shape'].name} M={M} differs from the device run")
    return dt, h2d, d2h


def oracle_sample(items, cols_per_item: int):
    """One bounded oracle pass: `cols_per_item` output columns (a window moving with `s`) of
    every call; returns (step function, algorithmic bytes per step pro rata)."""
    import oracle
    step_bytes = sum(it["bytes"] * min(cols_per_item, it["case"].N) / it["case"].N for it in items)

    def step(s):
        for it in items:
            c = it["case"]
            n = min(cols_per_item, c.N)
            n0 = (s * n) % max(1, c.N - n + 1)
            oracle.gemv(c, rows=list(range(n0, n0 + n)), M=it["M"])
    return step, step_bytes


def cpu_baseline(wl, seconds: float):
    """The oracle as it stands, on the host cores, over a bounded sample of the same workload:
    64 output columns per host thread of every call, repeated until `seconds` of work are done;
    GB/s counts the sampled columns' share of each call's algorithmic bytes."""
    import oracle
    oracle.build()
    cores = oracle.max_threads()
    cols = 64 * cores
    step, step_bytes = oracle_sample(wl.items, cols)
    done, reps = 0.0, 0
    t0 = time.perf_counter()
    while True:
        step(reps)
        done += step_bytes
        reps += 1
        if time.perf_counter() - t0 >= seconds:
            break
    dt = time.perf_counter() - t0
    return {"value": done / dt / 1e9, "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"{reps} pass(es) of {cols} output columns of each of the {len(wl.items)} calls "
                      f"(M as timed), {dt:.1f} s, OpenMP over output columns"}


def run_ours(args):
    import torch
    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    dist = init_dist(world, "nccl")
    from block_scaled_bit_gb300 import bsgemv
    bsgemv.lib()
    wl = Workload(args.config, args.M, device, copies=2)
    stream = torch.cuda.Stream(device)
    peak, peak_kind = hbm_peak()

    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        barrier(world)
        total, per, launches = time_graph(wl, args.steps, args.warmup, stream)
        torch.cuda.synchronize()
        barrier(world)
    clocks = clk.summary()
    total = max_over_ranks(total, world, device)
    step_bytes = wl.bytes_per_step
    value = job_throughput_gbps(world, args.steps, step_bytes, total)

    per_shape = []
    for j, it in enumerate(wl.items):
        us = statistics.median(per[j]) * 1e6
        per_shape.append({"shape": it["shape"].name, "M": it["M"], "us_per_call": round(us, 3),
                          "GBps": round(it["bytes"] / (us * 1e-6) / 1e9, 1),
                          "frac": round(it["bytes"] / (us * 1e-6) / 1e9 / peak, 4),
                          "bytes": it["bytes"]})
    # the dominant (only) kernel's average launch duration over the timed region: launches run
    # back to back with start-up overlapped, so the region divided by its launches
    L = len(wl.items)
    mean_launch = total / launches
    achieved = (step_bytes / L) / mean_launch / 1e9
    workload = f"config{args.config}"
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4), "traffic": recorded_traffic(workload),
                "peak_kind": f"{peak_kind} copy bandwidth (of {peak_kind})",
                "kernel": "bsgemv_mma_kernel"}

    streamed = streamed_per_item(wl, stream, peak)

    e2e_steps = max(10, min(200, args.steps))
    e2e_dt, h2d, d2h = e2e_run(wl, e2e_steps, stream)
    e2e_dt = max_over_ranks(e2e_dt, world, device)
    e2e = {"value": round(job_throughput_gbps(world, e2e_steps, step_bytes, e2e_dt), 1),
           "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
           "steps": e2e_steps,
           "api": f"bsgemv_run_host_async for each of the {L} calls of a step (pinned host A in, "
                  "pinned host y out: a copy kernel reads A into the plan's staging buffer and "
                  "the GEMV writes y, both through the pinned buffers' device mapping), "
                  "device-resident weights, the step replayed from a CUDA graph, one stream "
                  "synchronisation per step"}

    out = None
    if rank == 0:
        cpu = None
        if world == 1 and not args.skip_cpu:
            cpu = cpu_baseline(wl, args.cpu_seconds)
        S, full, rem = graph_plan(args.steps)
        s0 = wl.shapes[0]
        out = {
            "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(total / args.steps * 1e3, 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": workload_dtype(wl.shapes),
            "data": "synthetic (seeded), no trained weights",
            "config": {"workload": workload_name(args.config, wl.shapes, wl.Ms),
                       "calls_per_step": L, "bytes_per_step": step_bytes,
                       "plan_max_M": {s.name: max((args.M,) if args.M else s.Ms) for s in wl.shapes},
                       "cold": "M in the outer loop: two calls on one weight copy are separated by the "
                               "calls on every other shape of the step (> 3x L2), and each shape's 2 "
                               "weight copies alternate between steps; inputs larger than L2",
                       "timing": f"exactly {args.steps} steps replayed from CUDA graphs ({full} x {S} steps"
                                 + (f" + {rem}" if rem else "") + "), CUDA events on the launch stream "
                                 "around the timed region; per_shape from separate replays of a graph "
                                 "with an event between every launch (serialised); per_shape_streamed "
                                 "from a graph of back-to-back calls of one (shape, M) over weight "
                                 "copies > 3x L2 (overlapped like the step's calls)",
                       "parallelism": f"replicas x{world}" if world > 1 else "1 GPU"},
            "roofline": roofline,
            "fraction_of_nominal_7900_GBps": round(value / world / 7900.0, 4),
            "per_shape": per_shape,
            "per_shape_streamed": streamed,
            "e2e": e2e,
            "gpu_launches": launches,
            "clocks": clocks,
            "cpu_baseline": cpu,
            "impl": "ours",
        }
        if s0.fmt == "int4" and len(wl.Ms) > 1:
            out["by_M"] = by_M_summary(per_shape, peak)
            out["by_M_streamed"] = by_M_summary(streamed, peak)
    if dist is not None:
        dist.barrier()
    wl.close()
    if out is not None:
        print(json.dumps(out), flush=True)


def by_M_summary(per_shape, peak):
    """Per M: total bytes and time of that M's calls (as timed in `per_shape`), and the fraction
    of the peak."""
    out = {}
    for e in per_shape:
        d = out.setdefault(str(e["M"]), {"bytes": 0, "us": 0.0})
        d["bytes"] += e["bytes"]
        d["us"] += e["us_per_call"]
    for d in out.values():
        d["frac"] = round(d["bytes"] / (d["us"] * 1e-6) / 1e9 / peak, 4)
        d["us"] = round(d["us"], 2)
    return out


# ------------------------------------------------------------------------------ sweep
def run_sweep(args):
    """Every configuration shape and M: isolated-cold (L2 flushed before each call, median of
    repeats) and streamed-cold (graph of back-to-back calls over weight copies > 3x L2)."""
    import torch
    from block_scaled_bit_gb300 import bsgemv, synth
    torch.cuda.set_device(0)
    peak, _ = hbm_peak()
    stream = torch.cuda.Stream()
    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    flush = torch.empty(4 * l2 // 4, dtype=torch.int32, device="cuda")
    cfgs = [args.config] if args.config != WORKLOAD_CONFIG or "--config" in sys.argv else [1, 2, 3, 4, 5]
    for c in cfgs:
        for shape in synth.config_shapes(c):
            Ms = tuple(int(x) for x in args.Ms.split(",")) if args.Ms else shape.Ms
            case = shape.case(max(Ms))
            foot = case.algorithmic_bytes(1)
            copies = max(1, min(8, -(-3 * l2 // foot)))
            bufs = [bsgemv.upload(case, "cuda") for _ in range(copies)]
            # one plan per residency class: max_M <= 8 (4 CTAs per SM) and max_M > 8 (3)
            plans = {}

            def plan_for(M):
                pm = min(max(Ms), 8) if M <= 8 else max(Ms)
                if args.plan_max_M:
                    pm = max(args.plan_max_M, M)
                if pm not in plans:
                    plans[pm] = bsgemv.Plan(case.fmt, case.act, case.block_size, case.has_zp,
                                            case.N, case.K, pm)
                    if args.variant != "auto":
                        assert plans[pm].set_override(variant=bsgemv.VARIANTS[args.variant]) == bsgemv.OK
                    if args.tile_rows:
                        rc = plans[pm].set_override(rows_per_tile=args.tile_rows)
                        assert rc == bsgemv.OK, bsgemv.status_string(rc)
                    if args.autotune:
                        b = bufs[0]
                        plans[pm].autotune(b.A[:pm], b.W, b.scales, b.zp, b.y[:pm], M=pm, reps=10)
                return plans[pm]

            try:
                for M in Ms:
                    if args.variant == "cuda_core" and M > 8:
                        continue
                    plan = plan_for(M)
                    # isolated cold
                    t = []
                    with torch.cuda.stream(stream):
                        for r in range(25):
                            flush.add_(1)
                            b = bufs[r % copies]
                            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                            e0.record(stream)
                            plan.run(b.A[:M], b.W, b.scales, b.zp, b.y[:M], M=M, stream=stream)
                            e1.record(stream)
                            e1.synchronize()
                            t.append(e0.elapsed_time(e1) * 1e3)
                    iso = statistics.median(t[5:])
                    # streamed cold: graph of back-to-back calls cycling through the copies
                    reps = max(copies, 40 // copies * copies)
                    g = torch.cuda.CUDAGraph()
                    with torch.cuda.stream(stream):
                        for r in range(copies):
                            b = bufs[r]
                            plan.run(b.A[:M], b.W, b.scales, b.zp, b.y[:M], M=M, stream=stream)
                        stream.synchronize()
                        with torch.cuda.graph(g, stream=stream):
                            for r in range(reps):
                                b = bufs[r % copies]
                                plan.run(b.A[:M], b.W, b.scales, b.zp, b.y[:M], M=M, stream=stream)
                        g.replay()
                        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                        e0.record(stream)
                        for _ in range(5):
                            g.replay()
                        e1.record(stream)
                        e1.synchronize()
                    streamed = e0.elapsed_time(e1) * 1e3 / (5 * reps)
                    nbytes = case.algorithmic_bytes(M)
                    print(json.dumps({
                        "shape": shape.name, "config": c, "M": M, "bytes": nbytes,
                        "us_isolated_cold": round(iso, 3), "us_streamed_cold": round(streamed, 3),
                        "GBps_isolated": round(nbytes / iso / 1e3, 1),
                        "GBps_streamed": round(nbytes / streamed / 1e3, 1),
                        "frac_streamed": round(nbytes / streamed / 1e3 / peak, 4),
                        "frac_isolated": round(nbytes / iso / 1e3 / peak, 4),
                        "weight_copies": copies, "plan_max_M": plan.max_M,
                        "variant": "cuda_core" if plan.describe()["variant"] == 2 else "mma",
                        "autotuned": bool(args.autotune),
                        "geometry": {k: plan.describe()[k] for k in ("rows_per_tile", "ctas", "cluster",
                                                                    "stages", "ctas_per_sm")}}),
                          flush=True)
                    del g
            finally:
                for pl in plans.values():
                    pl.close()
            del bufs
            torch.cuda.empty_cache()


def run_one(args):
    """`--calls` isolated cold calls (L2 flushed before each) of one configuration shape."""
    import torch
    from block_scaled_bit_gb300 import bsgemv, synth
    shapes = {s.name: s for s in synth.all_shapes()}
    if args.one not in shapes:
        raise SystemExit(f"unknown shape {args.one!r}; one of: {', '.join(sorted(shapes))}")
    shape = shapes[args.one]
    torch.cuda.set_device(0)
    M = args.M or shape.Ms[0]
    case = shape.case(M)
    max_M = min(max(shape.Ms), 8) if M <= 8 else max(shape.Ms)   # as the sweep's plans
    if args.plan_max_M:
        max_M = args.plan_max_M
    stream = torch.cuda.Stream()
    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    flush = torch.empty(4 * l2 // 4, dtype=torch.int32, device="cuda")
    b = bsgemv.upload(case, "cuda")
    t = []
    with bsgemv.Plan(case.fmt, case.act, case.block_size, case.has_zp, case.N, case.K,
                     max(max_M, M)) as plan:
        if args.variant != "auto":
            assert plan.set_override(variant=bsgemv.VARIANTS[args.variant]) == bsgemv.OK
        with torch.cuda.stream(stream):
            for _ in range(args.calls):
                flush.add_(1)
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                plan.run(b.A, b.W, b.scales, b.zp, b.y, M=M, stream=stream)
                e1.record(stream)
                e1.synchronize()
                t.append(e0.elapsed_time(e1) * 1e3)
        variant = "cuda_core" if plan.describe()["variant"] == 2 else "mma"
        assert plan.device_status() == bsgemv.OK
    print(json.dumps({"shape": shape.name, "M": M, "variant": variant, "calls": args.calls,
                      "us_isolated_cold_median": round(statistics.median(t), 3),
                      "bytes": case.algorithmic_bytes(M)}), flush=True)


DENSE_SHAPES = [(32, 2048), (256, 2048), (512, 2048), (1024, 2048), (1024, 4096), (4096, 4096)]


def run_dense_sweep(args):
    """Dense y[M, N] = A[M, K] . B[K, N] (fp16, B row-major; the split-K GEMV page's shape corner
    M <= 8, N <= 1024 and one larger N): this library's split-K kernel and cuBLAS (torch.mm), each
    as a CUDA graph of back-to-back calls over copies of B totalling >= 3x L2 (cold weights)."""
    import torch
    from block_scaled_bit_gb300 import bsgemv, synth
    torch.cuda.set_device(0)
    peak, _ = hbm_peak()
    stream = torch.cuda.Stream()
    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    shapes = DENSE_SHAPES
    if args.dense_shape:
        shapes = [tuple(int(x) for x in args.dense_shape.split(","))]
    for N, K in shapes:
        A_bits, B_bits = synth.dense_operands("f16", 8, N, K, seed=N + K)
        copies = max(2, min(256, -(-3 * l2 // (2 * N * K))))
        B0 = torch.from_numpy(B_bits.view(np.int16)).cuda().view(torch.float16)
        Bs = [B0.clone() for _ in range(copies)]
        for M in ((args.M,) if args.M else (1, 4, 8)):
            A = torch.from_numpy(np.ascontiguousarray(A_bits[:M]).view(np.int16)).cuda().view(torch.float16)
            y = torch.empty((M, N), dtype=torch.float16, device="cuda")
            nbytes = 2 * (N * K + M * K + M * N)
            res = {}
            with bsgemv.DensePlan("f16", N, K, 8) as plan:
                geo = plan.describe()
                for impl in ("ours", "cublas"):
                    def call(b):
                        if impl == "ours":
                            plan.run(A, b, y, M=M, stream=stream)
                        else:
                            torch.mm(A, b, out=y)
                    with torch.cuda.stream(stream):
                        for b in Bs[:2]:
                            call(b)
                        stream.synchronize()
                        g = torch.cuda.CUDAGraph()
                        with torch.cuda.graph(g, stream=stream):
                            for b in Bs:
                                call(b)
                        g.replay()
                        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                        e0.record(stream)
                        for _ in range(5):
                            g.replay()
                        e1.record(stream)
                        e1.synchronize()
                    res[impl] = e0.elapsed_time(e1) * 1e3 / (5 * copies)
                    del g
            print(json.dumps({"dense": True, "N": N, "K": K, "M": M, "bytes": nbytes,
                              "us_ours": round(res["ours"], 3), "us_cublas": round(res["cublas"], 3),
                              "frac_ours": round(nbytes / res["ours"] / 1e3 / peak, 4),
                              "frac_cublas": round(nbytes / res["cublas"] / 1e3 / peak, 4),
                              "B_copies": copies, "geometry": {k: geo[k] for k in ("ctas", "cluster", "stages")}}),
                  flush=True)
        del Bs
        torch.cuda.empty_cache()


CROSSOVER_SHAPES = ["c3_int4_f16_bs32_nozp_N151936_K4096", "c3_int4_f16_bs32_nozp_N12288_K4096",
                    "c2_int8_f16_bs128_zp_N12288_K4096", "c4_fp8_f16_bs128_nozp_N5120_K17408",
                    "c5_nvfp4_f16_bs16_nozp_N248320_K2048"]


def run_crossover(args):
    """Where the fused GEMV stops paying: for M = 1 .. 32, the fused dequantise-and-multiply call
    against a tensor-core GEMM (cuBLAS, torch.mm) on the same weight already dequantised to fp16
    [N, K] (its dequantisation not counted, which favours cuBLAS).  Both as CUDA graphs of
    back-to-back calls over weight copies totalling >= 3x L2 (cold weights), same run."""
    import torch
    from block_scaled_bit_gb300 import bsgemv, synth
    torch.cuda.set_device(0)
    stream = torch.cuda.Stream()
    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    shapes = {s.name: s for s in synth.all_shapes()}
    Ms = tuple(int(x) for x in args.Ms.split(",")) if args.Ms else (1, 4, 8, 16, 24, 32)

    def graph_time(call, copies):
        with torch.cuda.stream(stream):
            for c in range(min(2, copies)):
                call(c)
            stream.synchronize()
            g = torch.cuda.CUDAGraph()
            reps = max(copies, 8 // copies * copies)
            with torch.cuda.graph(g, stream=stream):
                for r in range(reps):
                    call(r % copies)
            g.replay()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(3):
                g.replay()
            e1.record(stream)
            e1.synchronize()
        return e0.elapsed_time(e1) * 1e3 / (3 * reps)

    for name in CROSSOVER_SHAPES:
        shape = shapes[name]
        case = shape.case(1)
        fused_copies = max(1, min(8, -(-3 * l2 // case.algorithmic_bytes(1))))
        dense_copies = max(1, min(8, -(-3 * l2 // (2 * case.N * case.K))))
        bufs = [bsgemv.upload(case, "cuda") for _ in range(fused_copies)]
        with bsgemv.Plan(case.fmt, case.act, case.block_size, case.has_zp, case.N, case.K, 1) as p1:
            deq = torch.empty((case.N, case.K), dtype=torch.float32, device="cuda")
            p1.debug_dequant(bufs[0].W, bufs[0].scales, bufs[0].zp, deq)
            torch.cuda.synchronize()
            w16 = deq.to(torch.float16)
            del deq
        Ws = [w16] + [w16.clone() for _ in range(dense_copies - 1)]
        A32 = torch.randn((32, case.K), generator=torch.Generator().manual_seed(7)).to("cuda", torch.float16)
        plans = {}
        for M in Ms:
            pm = 8 if M <= 8 else 16 if M <= 16 else 24 if M <= 24 else 32
            if pm not in plans:
                plans[pm] = bsgemv.Plan(case.fmt, case.act, case.block_size, case.has_zp, case.N,
                                        case.K, pm)
            plan = plans[pm]
            A = A32[:M].contiguous()
            y = torch.empty((M, case.N), dtype=torch.float16, device="cuda")
            yt = torch.empty((M, case.N), dtype=torch.float16, device="cuda")
            t_fused = graph_time(lambda c: plan.run(A, bufs[c].W, bufs[c].scales, bufs[c].zp, y,
                                                    M=M, stream=stream), fused_copies)
            t_cublas = graph_time(lambda c: torch.mm(A, Ws[c].t(), out=yt), dense_copies)
            print(json.dumps({"crossover": True, "shape": name, "M": M,
                              "us_fused": round(t_fused, 2), "us_cublas_fp16": round(t_cublas, 2),
                              "fused_over_cublas": round(t_fused / t_cublas, 3),
                              "plan_max_M": pm}), flush=True)
        for pl in plans.values():
            pl.close()
        del bufs, Ws, w16
        torch.cuda.empty_cache()


# ------------------------------------------------------------------------------ reference arm
def run_reference(args):
    """The oracle (CPU, fp64) timed on the host cores on this workload; rank 0 only.  Each step
    is a bounded sample: 8 output columns per host thread of every call of the workload's step
    (every shape at every M), bytes pro rata."""
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import oracle
    from block_scaled_bit_gb300 import synth
    oracle.build()
    cores = oracle.max_threads()
    shapes = synth.config_shapes(args.config)
    items = []
    Ms = sorted({m for s in shapes for m in ((args.M,) if args.M else s.Ms)})
    cases = {s.name: s.case(max((args.M,) if args.M else s.Ms)) for s in shapes}
    for m in Ms:
        for s in shapes:
            if m in ((args.M,) if args.M else s.Ms):
                c = cases[s.name]
                items.append({"case": c, "M": m, "bytes": c.algorithmic_bytes(m)})
    cols = 8 * cores
    step, step_bytes = oracle_sample(items, cols)
    for s in range(max(3, args.warmup)):
        step(s)
    t0 = time.perf_counter()
    for s in range(args.steps):
        step(s)
    dt = time.perf_counter() - t0
    value = args.steps * step_bytes / dt / 1e9
    out = {"metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": world,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 4),
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
           "dtype": "f64 (oracle)", "data": "synthetic (seeded), no trained weights",
           "config": {"workload": workload_name(args.config, shapes, Ms),
                      "sample_per_step": f"{cols} output columns of each of the {len(items)} calls"},
           "impl": "reference",
           "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                            "sample": f"{cols} output columns per call per step, {args.steps} steps"},
           "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


def main():
    args = parse_args()
    if args.impl == "reference":
        run_reference(args)
    elif args.sweep:
        run_sweep(args)
    elif args.one:
        run_one(args)
    elif args.dense:
        run_dense_sweep(args)
    elif args.crossover:
        run_crossover(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
