#!/usr/bin/env python3
"""Benchmark of the block-scaled small-M GEMV on GB300.

Metric: achieved HBM GB/s on cold weights (algorithmic bytes W + scales + zp + A + y per call,
divided by the device time of the call), with microseconds per call and the fraction of the
measured HBM copy bandwidth.

Default workload (one "step" = one pass of the hot path over the workload): the 8-bit
MatMulNBits configuration -- int8 weights with zero points, fp16 activations, M = 1, block
sizes 128 and 32, shapes (K x N) 2048x5120, 4096x2048, 4096x4096, 4096x12288, 12288x4096:
ten GEMV calls per step.  Every shape has two weight copies used on alternate steps, so each
call reads weights last touched 19 calls (~0.5 GB of other traffic, > 4x L2) earlier: the
weights are cold.  The timed region replays a CUDA graph of 25 steps of back-to-back launches
(programmatic dependent launch overlaps each call's start-up with the previous call's tail);
a separate graph with an event between every launch gives per-call durations.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--sweep]

With --gpus N > 1 (launched under torchrun) every rank runs the same workload on its own GPU
(independent replicas: the GEMV has no exchange step), the time is the maximum over ranks and
the value is the bytes of all ranks over that time.  --impl reference times the CPU oracle on
the host cores instead.  --sweep prints one JSON line per (configuration shape, M) with
isolated-cold and streamed-cold timings.
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
WORKLOAD_CONFIG = 2
GRAPH_STEPS = 25


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=4000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--sweep", action="store_true")
    ap.add_argument("--config", type=int, default=WORKLOAD_CONFIG, help=argparse.SUPPRESS)
    ap.add_argument("--M", type=int, default=None, help=argparse.SUPPRESS)
    ap.add_argument("--no-graph", action="store_true", help=argparse.SUPPRESS)
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


def workload_name(config: int, shapes, M: int) -> str:
    """The workload of a configuration named by what it is, with its sizes (both arms)."""
    s0 = shapes[0]
    fmt = {"int4": "int4", "int8": "int8", "fp8": "FP8 E4M3", "nvfp4": "NVFP4"}[s0.fmt]
    zp = " with zero points" if s0.has_zp else ""
    return (f"{fmt} MatMulNBits GEMV{zp}: "
            + ", ".join(f"{s.K}x{s.N} bs{s.block_size}" for s in shapes)
            + f" (K x N), M={M}, {'bf16' if s0.act == 'bf16' else 'fp16'}")


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
    """Plans, device buffers (several weight copies) and host copies for one configuration."""

    def __init__(self, config: int, M: int | None, device, copies: int):
        from block_scaled_bit_gb300 import bsgemv, synth
        self.items = []
        for shape in synth.config_shapes(config):
            m = M or shape.Ms[0]
            case = shape.case(m)
            # plans are sized for the configuration's largest M (the M values it is quoted at)
            plan = bsgemv.Plan(case.fmt, case.act, case.block_size, case.has_zp, case.N, case.K,
                               max(max(shape.Ms), m))
            bufs = [bsgemv.upload(case, device) for _ in range(copies)]
            self.items.append({"shape": shape, "case": case, "M": m, "plan": plan, "bufs": bufs,
                               "bytes": case.algorithmic_bytes(m)})
        self.copies = copies

    @property
    def bytes_per_step(self) -> int:
        return sum(it["bytes"] for it in self.items)

    def launch(self, it, copy, stream=None):
        b = it["bufs"][copy % self.copies]
        it["plan"].run(b.A, b.W, b.scales, b.zp, b.y, M=it["M"], stream=stream)


def capture(wl, stream, steps, with_events):
    """CUDA graph of `steps` workload steps (optionally with timing events between launches)."""
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


def time_graph(wl, steps, warmup, stream, use_graph=True):
    """Time `steps` steps (rounded up to whole graphs of GRAPH_STEPS steps) of back-to-back
    launches; consecutive launches overlap start-up and tail (programmatic dependent launch).
    Then, outside the timed region, one replay of a graph with an event between every launch
    gives per-launch durations (events serialise the launches).
    Returns (seconds, per-launch seconds of the instrumented replay, steps, launches)."""
    import torch
    L = len(wl.items)
    S = GRAPH_STEPS
    replays = max(1, -(-steps // S))
    with torch.cuda.stream(stream):
        for s in range(S):                # warm every plan and weight copy outside capture
            for it in wl.items:
                wl.launch(it, s)
        stream.synchronize()
    graph = inst = events = None
    if use_graph:
        try:
            graph, _ = capture(wl, stream, S, False)
            inst, events = capture(wl, stream, S, True)
        except Exception as e:  # older torch: no external events in graphs
            sys.stderr.write(f"[bench] graph capture unavailable ({e}); timing eager launches\n")
            graph = inst = None
    if events is None or inst is None:
        events = [torch.cuda.Event(enable_timing=True) for _ in range(S * L + 1)]

    def replay():
        if graph is not None:
            graph.replay()
            return
        for s in range(S):
            for it in wl.items:
                wl.launch(it, s, stream)

    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        for _ in range(max(1, -(-warmup // S))):
            replay()
        stream.synchronize()
        start.record(stream)
        for _ in range(replays):
            replay()
        end.record(stream)
        end.synchronize()
        total = start.elapsed_time(end) / 1e3
        # per-launch durations (not part of the timed region)
        if inst is not None:
            inst.replay()
        else:
            i = 0
            for s in range(S):
                for it in wl.items:
                    events[i].record(stream)
                    i += 1
                    wl.launch(it, s, stream)
            events[i].record(stream)
        stream.synchronize()
    per_launch = [events[i].elapsed_time(events[i + 1]) / 1e3 for i in range(S * L)]
    return total, per_launch, replays * S, replays * S * L


def e2e_run(wl, steps, stream):
    """End to end through the public API: every step copies the activations of its ten GEMVs from
    pinned host memory to the device (one copy), runs the ten bsgemv_run calls on them and copies
    the ten outputs back to pinned host memory (one copy), and waits for the stream once, when
    all results are on the host.  The step is captured once per weight copy into a CUDA graph
    (the library's calls only enqueue work) and replayed; without graph support the step is
    issued directly."""
    import numpy as np
    import torch
    dev = stream.device

    def pad8(n):  # keep every slice 16-byte aligned
        return (n + 7) // 8 * 8
    a_off, y_off, na, ny = [], [], 0, 0
    for it in wl.items:
        a_off.append(na)
        y_off.append(ny)
        na += pad8(it["M"] * it["case"].K)
        ny += pad8(it["M"] * it["case"].N)
    A_host = torch.zeros(na, dtype=torch.int16).pin_memory()
    y_host = torch.empty(ny, dtype=torch.int16).pin_memory()
    for it, o in zip(wl.items, a_off):
        a = np.ascontiguousarray(it["case"].A[: it["M"]]).view(np.int16).reshape(-1)
        A_host[o:o + a.size] = torch.from_numpy(a)
    A_dev = torch.empty(na, dtype=torch.int16, device=dev)
    y_dev = torch.empty(ny, dtype=torch.int16, device=dev)
    h2d = sum(it["M"] * it["case"].K * 2 for it in wl.items)
    d2h = sum(it["M"] * it["case"].N * 2 for it in wl.items)

    def enqueue(s):
        with torch.cuda.stream(stream):
            A_dev.copy_(A_host, non_blocking=True)
            for it, ao, yo in zip(wl.items, a_off, y_off):
                b = it["bufs"][s % wl.copies]
                M, case = it["M"], it["case"]
                it["plan"].run(A_dev[ao:ao + M * case.K], b.W, b.scales, b.zp,
                               y_dev[yo:yo + M * case.N], M=M, stream=stream)
            y_host.copy_(y_dev, non_blocking=True)

    for s in range(3):
        enqueue(s)
        stream.synchronize()
    graphs = []
    try:
        for c in range(wl.copies):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                enqueue(c)
            graphs.append(g)
        with torch.cuda.stream(stream):  # (a graph replays on the current stream)
            for g in graphs:
                g.replay()
        stream.synchronize()
    except Exception as e:  # no graph capture: issue the step directly
        sys.stderr.write(f"[bench] e2e graph capture unavailable ({e}); direct calls\n")
        graphs = []
    y_host.fill_(-1)  # every output must come back from the timed steps
    y_dev.fill_(-1)
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    with torch.cuda.stream(stream):
        for s in range(steps):
            if graphs:
                graphs[s % len(graphs)].replay()
            else:
                enqueue(s)
            stream.synchronize()
    dt = time.perf_counter() - t0
    # the step's outputs made the round trip: check them against the device run of each plan
    ref = torch.empty_like(y_dev)
    with torch.cuda.stream(stream):
        for it, ao, yo in zip(wl.items, a_off, y_off):
            b = it["bufs"][(steps - 1) % wl.copies]
            M, case = it["M"], it["case"]
            it["plan"].run(A_dev[ao:ao + M * case.K], b.W, b.scales, b.zp, ref[yo:yo + M * case.N],
                           M=M, stream=stream)
    stream.synchronize()
    if not torch.equal(ref.cpu(), y_host):
        raise RuntimeError("e2e: host outputs differ from the device run")
    return dt, h2d, d2h, bool(graphs)


def cpu_baseline(wl, seconds: float):
    """The oracle as it stands, on the host cores, over the same workload until `seconds` of
    work are done (whole steps; all shapes, all output columns)."""
    import oracle
    oracle.build()
    cores = oracle.max_threads()
    done_bytes, reps = 0, 0
    t0 = time.perf_counter()
    while True:
        for it in wl.items:
            oracle.gemv(it["case"], M=it["M"])
            done_bytes += it["bytes"]
        reps += 1
        if time.perf_counter() - t0 >= seconds:
            break
    dt = time.perf_counter() - t0
    return {"value": done_bytes / dt / 1e9, "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"{reps} full pass(es) over the {len(wl.items)} GEMVs of the workload "
                      f"(all output columns, M as timed), {dt:.1f} s, OpenMP over output columns"}


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
        total, per_launch, steps_timed, launches = time_graph(wl, args.steps, args.warmup, stream,
                                                              not args.no_graph)
        torch.cuda.synchronize()
        barrier(world)
    clocks = clk.summary()
    total = max_over_ranks(total, world, device)
    step_bytes = wl.bytes_per_step
    value = job_throughput_gbps(world, steps_timed, step_bytes, total)

    # per-launch durations of the last replayed graph: L launches per step, GRAPH_STEPS steps
    L = len(wl.items)
    per_shape = []
    for j, it in enumerate(wl.items):
        d = [per_launch[s * L + j] for s in range(GRAPH_STEPS)]
        us = statistics.median(d) * 1e6
        per_shape.append({"shape": it["shape"].name, "M": it["M"], "us_per_call": round(us, 3),
                          "GBps": round(it["bytes"] / (us * 1e-6) / 1e9, 1),
                          "frac": round(it["bytes"] / (us * 1e-6) / 1e9 / peak, 4),
                          "bytes": it["bytes"]})
    # the dominant (only) kernel's average launch duration over the timed region: launches run
    # back to back with start-up overlapped, so the region divided by its launches
    mean_launch = total / launches
    achieved = (step_bytes / L) / mean_launch / 1e9
    workload = f"config{args.config}"
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4), "traffic": recorded_traffic(workload),
                "peak_kind": f"{peak_kind} copy bandwidth", "kernel": "bsgemv_mma_kernel"}

    e2e_dt, h2d, d2h, e2e_graph = e2e_run(wl, max(20, min(400, args.steps // 10)), stream)
    e2e_steps = max(20, min(400, args.steps // 10))
    e2e_dt = max_over_ranks(e2e_dt, world, device)
    e2e = {"value": round(job_throughput_gbps(world, e2e_steps, step_bytes, e2e_dt), 1), "unit": "GB/s",
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
           "api": "bsgemv_run on the step's activations copied host->device (pinned, one copy per step) "
                  "with the ten outputs copied device->host (one copy per step), device-resident weights, "
                  + ("the step replayed from a CUDA graph, " if e2e_graph else "") + "one stream synchronisation per step"}

    out = None
    if rank == 0:
        cpu = None
        if world == 1 and not args.skip_cpu:
            cpu = cpu_baseline(wl, args.cpu_seconds)
        shapes = [it["shape"] for it in wl.items]
        out = {
            "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world,
            "steps": steps_timed, "warmup": args.warmup,
            "ms_per_step": round(total / steps_timed * 1e3, 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "u8 weights (int8 + zp), f16 activations, f32 accumulate",
            "data": "synthetic (seeded), no trained weights",
            "config": {"workload": workload_name(args.config, shapes, wl.items[0]["M"]),
                       "calls_per_step": L, "bytes_per_step": step_bytes,
                       "cold": "2 weight copies per shape on alternate steps: each call's weights "
                               "were last read 19 calls (>0.5 GB, >4x L2) earlier; inputs larger than L2",
                       "timing": f"CUDA graph of {GRAPH_STEPS} steps replayed, CUDA events on the launch stream "
                                 "around the timed region; per_shape from a separate graph with an "
                                 "event between every launch (serialised)",
                       "parallelism": f"replicas x{world}" if world > 1 else "1 GPU"},
            "roofline": roofline,
            "fraction_of_nominal_7900_GBps": round(value / world / 7900.0, 4),
            "per_shape": per_shape,
            "e2e": e2e,
            "gpu_launches": launches,
            "clocks": clocks,
            "cpu_baseline": cpu,
            "impl": "ours",
        }
    if dist is not None:
        dist.barrier()
    for it in wl.items:
        it["plan"].close()
    if out is not None:
        print(json.dumps(out), flush=True)


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
                if pm not in plans:
                    plans[pm] = bsgemv.Plan(case.fmt, case.act, case.block_size, case.has_zp,
                                            case.N, case.K, pm)
                    if args.variant != "auto":
                        assert plans[pm].set_override(variant=bsgemv.VARIANTS[args.variant]) == bsgemv.OK
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
                        "geometry": {k: plan.describe()[k] for k in ("ctas", "cluster", "stages")}}),
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
    """The oracle (CPU, fp64) timed on the host cores on this workload; rank 0 only."""
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import oracle
    from block_scaled_bit_gb300 import synth
    oracle.build()
    cores = oracle.max_threads()
    items = []
    for shape in synth.config_shapes(args.config):
        m = args.M or shape.Ms[0]
        case = shape.case(m)
        items.append((case, m, case.algorithmic_bytes(m)))
    # each step: a bounded sample of output columns of every shape, 8 per host thread (the
    # oracle hands its OpenMP threads columns in chunks of 8); bytes pro rata
    cols = 8 * cores
    step_bytes = sum(b * min(cols, c.N) / c.N for c, _, b in items)

    def step(s):
        for c, m, _ in items:
            n = min(cols, c.N)
            n0 = (s * n) % max(1, c.N - n + 1)
            oracle.gemv(c, rows=list(range(n0, n0 + n)), M=m)

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
           "config": {"workload": workload_name(args.config, [synth_shape for synth_shape in
                                                             synth.config_shapes(args.config)],
                                                items[0][1]),
                      "sample_per_step": f"{cols} output columns of each of the {len(items)} GEMVs"},
           "impl": "reference",
           "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                            "sample": f"{cols} output columns per GEMV per step, {args.steps} steps"},
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
