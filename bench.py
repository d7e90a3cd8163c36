#!/usr/bin/env python3
"""Benchmark of the Q4_0 weight-only matmul on GB300.

Default workload (``--workload decode``): one decode step = the four 27B-class
layer matrices (QKV 7168x5120, O 5120x5120, gate+up 34816x5120, down
5120x17408) at M = 1, through q4_0_matmul.  Eight distinct layer copies
(1.49 GB of Q4_0 weights, 11.6x the 129 MB L2) stay resident in HBM and step
i uses copy i mod 8, so no step finds its weights in L2.  The metric is
algorithmic GB/s (0.5625 N K + 2 M K + 4 M N bytes per matrix) with the
weights-per-second equivalent in tokens/s of a 64-layer stack.

Other workloads: ``batched`` (M = 16), ``prefill`` (M = 2048, TFLOP/s) and
``sweep`` (64 layers at M = 1).  ``--impl reference`` times the CPU oracle on
the host cores instead (a bounded sample of the same workload).

One JSON line is printed by rank 0.  Under torchrun every rank runs an
independent replica (the matmul has no exchange step); the value is the
bytes of all ranks over the slowest rank's time.
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, HERE)

SHAPE_ORDER = ("qkv", "o", "gate_up", "down")
LAYER_WEIGHTS_64 = 21.139e9  # Q4_0 weights in 64 layers of the four matrices
METRIC = "Q4_0 matmul: decode GB/s (% HBM peak), prefill TFLOP/s, tok/s-equivalent"


def alg_bytes(M, N, K, y_bytes=4):
    return 0.5625 * N * K + 2 * M * K + y_bytes * M * N


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20000)
    p.add_argument("--warmup", type=int, default=200)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", choices=["decode", "batched", "prefill", "sweep", "chunked", "chunked_split"],
                   default="decode")
    p.add_argument("--m", type=int, default=None, help="rows of x (overrides the workload's M)")
    p.add_argument("--layers", type=int, default=8, help="resident layer copies (decode/batched)")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--e2e-steps", type=int, default=2000)
    p.add_argument("--grouped", action="store_true",
                   help="decode (M = 1): each layer's matrices as one q4_0_matmul_grouped call")
    p.add_argument("--y-dtype", choices=["f32", "bf16"], default="f32",
                   help="element type of y (bf16: the rounded-once output of q4_0_matmul_ex)")
    p.add_argument("--no-sub", action="store_true",
                   help="decode: skip the batched / prefill / chunked results beside the headline")
    return p.parse_args()


def peaks():
    path = os.path.join(HERE, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d["hbm_gbs"], d["bf16_tflops"], d.get("bf16_tflops_sustained", d["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


def workload_shapes(name, m=None):
    """M and the four layer shapes of a workload.  chunked: one 256-token
    prefill chunk and a 16-row decode batch as one M = 272 call per matrix."""
    from q4_weight_only_gb300 import synth
    M = {"decode": 1, "batched": 16, "prefill": 2048, "sweep": 1, "chunked": 272, "chunked_split": 272}[name]
    if m is not None:
        M = m
    return M, [(s, synth.SHAPES[s]) for s in SHAPE_ORDER]


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi clock/throttle samples of this process's GPU, 200 ms apart."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        import torch
        self.proc = None
        self.t0 = self.t1 = None
        try:
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            ident = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
        except Exception:
            ident = str(device_index)
        self.out = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={ident}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.out, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

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
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.out.flush()
        rows = []
        with open(self.out.name) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                    rows.append((ts, float(parts[1]), float(parts[2]), parts[4:]))
                except Exception:
                    continue
        os.unlink(self.out.name)
        if not rows:
            return None
        inside = [r for r in rows if self.t0 - 1 <= r[0] <= self.t1 + 1] or rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in inside for i, v in enumerate(r[3][1:5])
                          if v.lower().startswith("active")})
        return {"sm_mhz": statistics.median(r[1] for r in inside),
                "sm_max_mhz": max(r[2] for r in inside), "reasons": reasons,
                "samples": len(inside)}


# ------------------------------------------------------------ distributed

def dist_setup(gpus):
    """One process per GPU (torchrun env).  NCCL when CUDA is present, gloo
    otherwise; the matmul itself exchanges nothing between ranks."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
            dist.init_process_group(backend="nccl", device_id=torch.device("cuda", local))
        else:
            dist.init_process_group(backend="gloo")
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v, world):
    """The slowest rank's value (all ranks get it)."""
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(v)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------- our arm

def build_layers(q4, synth, shapes, layers, device):
    import torch
    wq = []
    for l in range(layers):
        per = []
        for s, (N, K) in shapes:
            w = synth.device_layer_weights(l, s, device=device)
            per.append(q4.quantize(w))
            del w
        wq.append(per)
    torch.cuda.synchronize()
    return wq


# Spin kernel run just before the start event: the device stays busy while
# the host enqueues the start event and the timed graph replays, so the timed
# region holds the K steps back to back and no host submission latency.
BUSY_CYCLES = 2_000_000


def measure(q4, synth, wq, workload, M, args, dev, world, grouped=False, cpu=False):
    """Time `args.steps` steps of one workload on the resident layer copies
    `wq` (a list of per-layer lists of the four Q4_0 matrices) and return the
    workload's result: value, roofline of the dominant kernel, e2e through
    the host-buffer entry point, clocks and launch counts."""
    import torch
    hbm, tf_burst, tf_sust, peak_kind = peaks()
    shapes = [(s, synth.SHAPES[s]) for s in SHAPE_ORDER]
    sweep = workload == "sweep"
    layers = len(wq)
    g = torch.Generator(device=dev)
    g.manual_seed(7)
    xs = [torch.randn((M, K), generator=g, device=dev).to(torch.bfloat16) for _, (N, K) in shapes]
    ydt = torch.bfloat16 if args.y_dtype == "bf16" else torch.float32
    ysz = 2 if args.y_dtype == "bf16" else 4
    ys = [torch.empty((M, N), dtype=ydt, device=dev) for _, (N, K) in shapes]
    # row ranges of x issued as separate calls: chunked_split runs the
    # 256-token chunk and the 16 decode rows of each matrix as two calls
    parts = [(0, 256), (256, M)] if workload == "chunked_split" else [(0, M)]
    wss = [[torch.empty(max(1, q4.lib().q4_0_matmul_workspace_bytes(m1 - m0, N, K)), dtype=torch.uint8,
                        device=dev) for m0, m1 in parts] for _, (N, K) in shapes]
    stream = torch.cuda.Stream(device=dev)

    per_step_layers = layers if sweep else 1  # a sweep step passes through every layer
    step_bytes = per_step_layers * sum(alg_bytes(M, N, K, ysz) for _, (N, K) in shapes)
    step_flops = per_step_layers * sum(2.0 * M * N * K for _, (N, K) in shapes)
    step_weights = per_step_layers * sum(N * K for _, (N, K) in shapes)
    Ns = [N for _, (N, K) in shapes]
    Ks = [K for _, (N, K) in shapes]

    def enqueue_step(i):
        ls = range(layers) if sweep else (i % layers,)
        for l in ls:
            if grouped:
                q4.matmul_grouped(xs, wq[l], Ns, Ks, outs=ys, stream=stream, out_dtype=ydt)
                continue
            for j, (_, (N, K)) in enumerate(shapes):
                for p, (m0, m1) in enumerate(parts):
                    q4.matmul(xs[j][m0:m1], wq[l][j], N, K, out=ys[j][m0:m1], workspace=wss[j][p], stream=stream,
                              out_dtype=ydt)

    calls_per_step = len(shapes) * len(parts) * (layers if sweep else 1)
    if grouped:
        launches_per_step = q4.grouped_launches(M, Ns, Ks) * (layers if sweep else 1)
    else:
        launches_per_step = sum(kernels_per_call(q4, m1 - m0, N, K) for _, (N, K) in shapes
                                for m0, m1 in parts) * (layers if sweep else 1)

    # CUDA graphs (a decode engine captures a whole pass the same way): the
    # timed steps as one graph when they fit about a thousand kernels,
    # otherwise a graph of a whole number of layer cycles replayed, plus one
    # graph for the remainder.  Step i of a graph uses layer copy i mod the
    # copies, and every graph but the last holds whole cycles, so the copies
    # rotate without a break across replays.
    cycle = 1 if sweep else layers
    max_steps_per_graph = max(1, 1024 // max(1, launches_per_step))

    def capture(n):
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=stream):
            for v in range(n):
                enqueue_step(v)
        return gr

    with torch.cuda.stream(stream):
        for i in range(3):  # load/initialise before capture
            enqueue_step(i)
        stream.synchronize()
        if args.steps <= max_steps_per_graph:
            plan = [(capture(args.steps), args.steps, 1)]
        else:
            C = max(cycle, max_steps_per_graph // cycle * cycle)
            reps, rem = divmod(args.steps, C)
            plan = [(capture(C), C, reps)] + ([(capture(rem), rem, 1)] if rem else [])

    def run_timed():
        for gr, _, reps in plan:
            for _ in range(reps):
                gr.replay()

    # warm-up: every graph replays at least once before the timed region
    # (a graph's first replay uploads it), then at least the requested
    # warm-up steps
    warm = 0
    with torch.cuda.stream(stream):
        for gr, n, _ in plan:
            gr.replay()
            warm += n
        while warm < max(3, args.warmup):
            plan[0][0].replay()
            warm += plan[0][1]
    torch.cuda.synchronize()
    clocks = ClockSampler(dev.index if dev.index is not None else 0)
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    clocks.mark_start()
    with torch.cuda.stream(stream):
        torch.cuda._sleep(BUSY_CYCLES)
        ev0.record(stream)
        run_timed()
        ev1.record(stream)
    ev1.synchronize()
    # keep the clock sampler's window on the work for short regions
    elapsed = ev0.elapsed_time(ev1) / 1e3
    if elapsed < 0.5:
        with torch.cuda.stream(stream):
            for _ in range(int(0.5 / max(elapsed, 1e-6)) + 1):
                run_timed()
        stream.synchronize()
    clocks.mark_end()
    torch.cuda.synchronize()
    barrier(world)
    ms_local = ev0.elapsed_time(ev1)
    ms = max_over_ranks(ms_local, world)
    clk = clocks.stop()
    if q4.device_error() != 0:
        raise RuntimeError("a kernel reported a device timeout during the benchmark")

    sec = ms / 1e3
    gbs = step_bytes * args.steps * world / sec / 1e9
    tflops = step_flops * args.steps * world / sec / 1e12
    tok_s = M * step_weights * args.steps * world / sec / LAYER_WEIGHTS_64

    # ---- end to end through the public API with host buffers
    e2e_steps = max(1, min(args.e2e_steps, args.steps))
    x_host = [torch.empty((M, K), dtype=torch.bfloat16).pin_memory() for _, (N, K) in shapes]
    for j, xh in enumerate(x_host):
        xh.copy_(xs[j].cpu())
    y_host = [torch.empty((M, N), dtype=ydt).pin_memory() for _, (N, K) in shapes]
    # q4_0_matmul_host: one library call per matmul with x and y in
    # page-locked host memory (read and written in place by the kernels
    # where the device maps it, else copied); its device scratch holds the
    # rest
    whs = [[torch.empty(q4.host_workspace_bytes(m1 - m0, N, K, ydt), dtype=torch.uint8, device=dev)
            for m0, m1 in parts] for _, (N, K) in shapes]
    # the row ranges of each call as views made once (a user's own buffers)
    x_views = [[x_host[j][m0:m1] for m0, m1 in parts] for j in range(len(shapes))]
    y_views = [[y_host[j][m0:m1] for m0, m1 in parts] for j in range(len(shapes))]
    h2d = sum(x.numel() * 2 for x in x_host) * (layers if sweep else 1)
    d2h = sum(y.numel() * ysz for y in y_host) * (layers if sweep else 1)

    # where an e2e step's time goes: host time inside the library calls,
    # device time of the step (events around it), and the wait for it
    parts_t = {"api": 0.0, "sync": 0.0, "device": 0.0}
    ev_a, ev_b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def issue(i):
        ls = range(layers) if sweep else (i % layers,)
        for l in ls:
            if grouped:
                # the grouped call takes device buffers: x copied in and y
                # copied out around it, on the same stream
                for j in range(len(shapes)):
                    xs[j].copy_(x_host[j], non_blocking=True)
                q4.matmul_grouped(xs, wq[l], Ns, Ks, outs=ys, stream=stream, out_dtype=ydt)
                for j in range(len(shapes)):
                    y_host[j].copy_(ys[j], non_blocking=True)
                continue
            for j, (_, (N, K)) in enumerate(shapes):
                for p in range(len(parts)):
                    q4.matmul_host(x_views[j][p], wq[l][j], N, K, out=y_views[j][p], workspace=whs[j][p],
                                   stream=stream, out_dtype=ydt)

    def e2e_step(i, account=False):
        t_a = time.perf_counter()
        if account:
            ev_a.record(stream)
        issue(i)
        if account:
            ev_b.record(stream)
        t_b = time.perf_counter()
        stream.synchronize()
        if account:
            parts_t["api"] += t_b - t_a
            parts_t["sync"] += time.perf_counter() - t_b
            parts_t["device"] += ev_a.elapsed_time(ev_b) / 1e3

    with torch.cuda.stream(stream):
        for i in range(min(3, e2e_steps)):  # first calls of the host path outside the timing
            e2e_step(i)
    torch.cuda.synchronize()
    barrier(world)
    t0 = time.perf_counter()
    with torch.cuda.stream(stream):
        for i in range(e2e_steps):
            e2e_step(i)
    t_e2e = max_over_ranks(time.perf_counter() - t0, world)
    # the breakdown from a separate, shorter pass (its events and timers stay
    # out of the timed e2e loop)
    acc_steps = max(1, min(200, e2e_steps))
    with torch.cuda.stream(stream):
        for i in range(acc_steps):
            e2e_step(i, account=True)
    # the same calls captured once per layer copy (per step of the sweep) as
    # CUDA graphs, one replay and one wait per step: the step of a server that
    # replays its calls as a graph, host copies still inside every step
    # (the grouped form's e2e copies x and y with torch around its call and
    # is timed with direct calls only)
    t_graph = None
    if not grouped:
        n_gr = 1 if sweep else layers
        graphs = []
        for i in range(n_gr):
            gr = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gr, stream=stream):
                issue(i)
            graphs.append(gr)
        with torch.cuda.stream(stream):
            for i in range(max(3, n_gr)):  # every graph replays once (its upload) before the timing
                graphs[i % n_gr].replay()
                stream.synchronize()
        barrier(world)
        t0 = time.perf_counter()
        with torch.cuda.stream(stream):
            for i in range(e2e_steps):
                graphs[i % n_gr].replay()
                stream.synchronize()
        t_graph = max_over_ranks(time.perf_counter() - t0, world)
        del graphs, gr
    barrier(world)
    tensor_bound = M >= 256
    e2e_val = (step_flops if tensor_bound else step_bytes) * e2e_steps * world / t_e2e / (1e12 if tensor_bound else 1e9)
    graph_val = e2e_val * t_e2e / t_graph if t_graph else None

    unit = "TFLOP/s" if tensor_bound else "GB/s"
    value = tflops if tensor_bound else gbs
    launches = args.steps * launches_per_step
    if grouped:
        calls_per_step = launches_per_step  # one grouped launch covers several matmuls
    calls = args.steps * calls_per_step  # launches of the dominant kernel (one per matmul)
    if not tensor_bound:
        roof = {"bound": "hbm", "achieved": round(gbs / world, 1), "peak": hbm, "unit": "GB/s",
                "frac": round(gbs / world / hbm, 4), "traffic": None,
                "kernel": dominant_kernel(M, grouped), "peak_source": peak_kind + " (copy bandwidth)",
                "bytes_per_launch": round(step_bytes / calls_per_step),
                "avg_launch_us": round(ms_local * 1e3 / calls, 3),
                "timing": "whole step on the launching stream (every kernel of the step), / matmul calls"}
    else:
        # a GEMM timed inside a short region: the burst peak; the sustained
        # fraction beside it
        roof = {"bound": "tensor", "achieved": round(tflops / world, 1), "peak": tf_burst,
                "unit": "TFLOP/s", "frac": round(tflops / world / tf_burst, 4), "traffic": None,
                "kernel": dominant_kernel(M, q4=q4), "peak_source": peak_kind + " bf16 burst (kind::f16 runs at the bf16 rate)",
                "frac_of_sustained": round(tflops / world / tf_sust, 4), "peak_sustained": tf_sust,
                "flops_per_launch": round(step_flops / calls_per_step),
                "avg_launch_us": round(ms_local * 1e3 / calls, 3),
                "timing": "whole step on the launching stream (x pre-pass and split-K sum included), / matmul calls"}
    # the sweep runs the decode (M = 1) or batched (M = 16) step's four
    # shapes through the same kernels, every layer's weights cold in L2 as
    # in those steps: the same bytes per launch
    traffic = load_traffic("grouped" if grouped else ("decode" if M == 1 else "batched") if sweep else workload, M)
    if traffic is not None:
        roof["traffic"] = traffic
    res = {"workload": workload_name(workload, M, layers, grouped), "M": M,
           "value": round(value, 2), "unit": unit, "steps": args.steps, "warmup": warm,
           "ms_per_step": round(ms / args.steps, 5),
           "tok_s_eq": round(tok_s, 1), "tflops": round(tflops, 2), "gbs": round(gbs, 1),
           "gpu_launches": launches, "roofline": roof, "clocks": clk,
           "e2e": {"value": round(e2e_val, 2), "unit": unit, "h2d_bytes_per_step": h2d,
                   "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                   "us_per_step": round(t_e2e / e2e_steps * 1e6, 2),
                   "breakdown_us_per_step": {
                       "steps": acc_steps,
                       "host_in_library_calls": round(parts_t["api"] / acc_steps * 1e6, 2),
                       "waiting_for_the_step": round(parts_t["sync"] / acc_steps * 1e6, 2),
                       "device_time_of_the_step": round(parts_t["device"] / acc_steps * 1e6, 2)},
                   "graph_replay": None if t_graph is None else {
                       "value": round(graph_val, 2), "us_per_step": round(t_graph / e2e_steps * 1e6, 2),
                       "steps": e2e_steps,
                       "how": "the step's library calls captured once per layer copy as CUDA graphs; "
                              "one replay and one stream wait per step"}},
           "layer_copies": layers,
           "graphs": " + ".join(f"{reps} x {n} steps" for _, n, reps in plan)}
    if cpu:
        res["cpu_baseline"] = cpu_baseline(wq[0], xs, shapes, M, budget_s=10.0)
    del xs, ys, wss, whs, plan
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return res


# The default run reports these beside the decode headline: the other parts
# of the metric (batched decode, prefill TFLOP/s, chunked prefill) on the
# same resident layer copies.
SUB_WORKLOADS = (("batched_m16", "batched", 16), ("prefill_m2048", "prefill", 2048),
                 ("chunked_m272", "chunked", 272))


def run_ours(args, rank, world, local):
    import torch
    from q4_weight_only_gb300 import build as lib_build
    lib_build.build()
    import q4_weight_only_gb300 as q4
    from q4_weight_only_gb300 import synth

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    M, shapes = workload_shapes(args.workload, args.m)
    layers = 64 if args.workload == "sweep" else (1 if args.workload == "prefill" else args.layers)
    wq = build_layers(q4, synth, shapes, layers, dev)
    Ns = [N for _, (N, K) in shapes]
    Ks = [K for _, (N, K) in shapes]
    grouped = args.grouped and q4.grouped_launches(M, Ns, Ks) > 0
    if args.grouped and not grouped:
        raise SystemExit("--grouped: the grouped decode does not take these shapes at this M")
    cpu = rank == 0 and world == 1 and not args.no_cpu_baseline
    head = measure(q4, synth, wq, args.workload, M, args, dev, world, grouped=grouped, cpu=cpu)

    subs = {}
    if args.workload == "decode" and args.m is None and not grouped and not args.no_sub:
        for key, wl, m in SUB_WORKLOADS:
            subs[key] = measure(q4, synth, wq[:1] if wl == "prefill" else wq, wl, m, args, dev, world)

    dt = ("q4_0 codes x 15-bit fixed-point x: int dp4a in-block, f32 across blocks" if M <= 2 else
          "q4_0 weights -> f16 tiles; f16 MMA, f32 accumulate")
    line = {
        "metric": METRIC, "value": head["value"], "unit": head["unit"], "n_gpus": world,
        "steps": args.steps, "warmup": head["warmup"], "ms_per_step": head["ms_per_step"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": dt,
        "data": "synthetic: W ~ N(0, 0.02) quantized on device, x ~ N(0, 1) bf16",
        "config": {"workload": head["workload"], "M": M,
                   "shapes": {s: list(nk) for s, nk in shapes}, "layer_copies": layers,
                   "l2": "inputs larger than L2: %d resident layer copies, %.2f GB cycled"
                         % (layers, layers * sum(0.5625 * N * K for _, (N, K) in shapes) / 1e9),
                   "y": args.y_dtype, "parallelism": f"replicas x{world}",
                   "graph": f"timed steps as CUDA graph replays ({head['graphs']}); PDL between kernels; "
                            "a spin kernel keeps the device busy across the start event"},
        "tok_s_eq": head["tok_s_eq"],
        "tflops": head["tflops"],
        "gpu_launches": head["gpu_launches"],
        "roofline": head["roofline"],
        "clocks": head["clocks"],
        "e2e": head["e2e"],
    }
    if "cpu_baseline" in head:
        line["cpu_baseline"] = head["cpu_baseline"]
    if subs:
        line["sub"] = subs
    return line if rank == 0 else None


def workload_name(w, M, layers, grouped=False):
    if grouped:
        return (f"decode M={M}, four 27B-class layer matrices per step as one grouped call, "
                f"{layers} layer copies" if w != "sweep" else
                f"64-layer decode sweep at M={M}, each layer's four matrices as one grouped call")
    return {"decode": f"decode M={M}, four 27B-class layer matrices per step, {layers} layer copies",
            "batched": f"batched decode M={M}, four 27B-class layer matrices per step, {layers} layer copies",
            "prefill": f"prefill M={M}, four 27B-class layer matrices per step",
            "sweep": f"64-layer decode sweep at M={M} (256 matrices per step)",
            "chunked_split": f"chunked prefill: 256-token chunk + 16 decode rows as two calls per matrix "
                             f"(M=256 and M={M - 256}), four matrices per step, {layers} layer copies",
            "chunked": f"chunked prefill: 256-token chunk + 16 decode rows as one M={M} call per matrix, "
                       f"four matrices per step, {layers} layer copies"}[w]


# q4_0_matmul sends M up to this to the decode kernels, larger M to the GEMM
DECODE_MAX_M = 64
# gate+up, the largest matrix of a layer (N, K): its GEMM plan names the prefill kernel
SHAPES_FOR_PLAN = (34816, 5120)


def kernels_per_call(q4, M, N, K):
    """Kernels one q4_0_matmul call launches: the integer-dot decode
    (M <= 2); x tiles + tensor-core decode (3 <= M <= DECODE_MAX_M); x ->
    binary16 + GEMM, plus the split-K sum when the workspace holds partial
    tiles."""
    if M <= 2:
        return 1
    if M <= DECODE_MAX_M:
        return 2
    x16 = (M * K * 2 + 255) // 256 * 256 + (M * 4 + 255) // 256 * 256  # x as binary16 and its row scales
    return 3 if q4.lib().q4_0_gemm_workspace_bytes(M, N, K) > x16 else 2


def dominant_kernel(M, grouped=False, q4=None):
    if grouped:
        return f"gemv_dp4a_grouped_kernel<{M}>"
    if M <= 2:
        return f"gemv_dp4a_kernel<{M}>"
    if M <= DECODE_MAX_M:
        return f"gemv_tc_kernel<{16 if M <= 16 else (32 if M <= 32 else 64)}>"
    # the largest matrix of the step (gate+up) decides: one CTA per tile, or
    # the persistent form (the library's launch plan)
    if q4 is not None:
        N, K = SHAPES_FOR_PLAN
        try:
            if q4.gemm_plan(M, N, K)["persistent"]:
                return "gemm_persistent_kernel"
        except Exception:
            pass
    return "gemm_kernel"


def load_traffic(workload, M):
    """DRAM bytes per launch of the dominant kernel, from the committed ncu
    summary (profiles/traffic.json); None when there is none for this
    workload and M or the kernel source has changed since it was captured."""
    import hashlib
    path = os.path.join(HERE, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    try:
        with open(path) as f:
            d = json.load(f).get(workload)
        if not d or d.get("M") != M:
            return None
        with open(os.path.join(HERE, d["kernel_source"]), "rb") as f:
            if hashlib.sha256(f.read()).hexdigest()[:16] != d["sha256_16"]:
                return None
        return d["bytes_per_launch"]
    except Exception:
        return None


# ------------------------------------------------------------ CPU oracle

def cpu_baseline(wq_layer, xs, shapes, M, budget_s=10.0):
    """The oracle on the host cores over a bounded sample of the workload."""
    import oracle
    o = oracle.get()
    host_w = [w.cpu().numpy() for w in wq_layer]
    host_x = [x.view(__import__("torch").int16).cpu().numpy().view(np.uint16) for x in xs]
    done_bytes, done_flops, t_used, reps = 0.0, 0.0, 0.0, 0
    while t_used < budget_s:
        for j, (_, (N, K)) in enumerate(shapes):
            rows = N if M < 256 else max(1, N // 64)
            t0 = time.perf_counter()
            o.matmul(host_x[j][:M], host_w[j][:rows], rows, K)
            t_used += time.perf_counter() - t0
            done_bytes += alg_bytes(M, rows, K)
            done_flops += 2.0 * M * rows * K
        reps += 1
    unit = "GB/s" if M < 256 else "TFLOP/s"
    val = done_bytes / t_used / 1e9 if M < 256 else done_flops / t_used / 1e12
    return {"value": round(val, 4), "unit": unit, "cores": o.threads(), "kind": "oracle",
            "sample": f"{reps} pass(es) of the four matrices at M={M}"
                      + ("" if M < 256 else " on 1/64 of the rows") + f", {t_used:.1f} s"}


def run_reference(args, rank, world, local):
    """The oracle as the reference arm: each step is a bounded sample of the
    workload (a slice of rows of each matrix) on the host cores."""
    ref_layers = 64 if args.workload == "sweep" else (1 if args.workload == "prefill" else args.layers)
    if rank != 0:
        return None
    import oracle
    from q4_weight_only_gb300 import synth
    o = oracle.get()
    M, shapes = workload_shapes(args.workload, args.m)
    warm = max(3, args.warmup)
    total_steps = args.steps + warm
    per_step_budget = min(0.5, 150.0 / total_steps)
    # probe the oracle's speed on a small slice to size the per-step sample
    rng = np.random.default_rng(0)
    host = []
    for s, (N, K) in shapes:
        rows = min(N, 1024)
        wq = o.quantize(synth.weights(synth.generator(100 + SHAPE_ORDER.index(s)), rows, K))
        x = synth.to_bf16_bits(rng.standard_normal((M, K), dtype=np.float32))
        host.append((N, K, wq, x))
    t0 = time.perf_counter()
    for N, K, wq, x in host:
        o.matmul(x, wq[:64], 64, K)
    per_row = (time.perf_counter() - t0) / (64 * len(host))
    rows = int(max(1, min(1024, per_step_budget / max(per_row * len(host), 1e-9))))
    for _ in range(warm):
        for N, K, wq, x in host:
            o.matmul(x, wq[:rows], rows, K)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        for N, K, wq, x in host:
            o.matmul(x, wq[:rows], rows, K)
    t = time.perf_counter() - t0
    byts = sum(alg_bytes(M, rows, K, 2 if args.y_dtype == "bf16" else 4) for N, K, _, _ in host) * args.steps
    flops = sum(2.0 * M * rows * K for N, K, _, _ in host) * args.steps
    unit = "GB/s" if M < 256 else "TFLOP/s"
    val = byts / t / 1e9 if M < 256 else flops / t / 1e12
    sample = f"{rows} rows of each of the four matrices per step at M={M}"
    return {"impl": "reference", "metric": METRIC, "value": round(val, 4), "unit": unit,
            "n_gpus": world, "steps": args.steps, "warmup": warm,
            "ms_per_step": round(t / args.steps * 1e3, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": workload_name(args.workload, M, ref_layers), "M": M,
                       "shapes": {s: list(nk) for s, nk in shapes}, "y": args.y_dtype},
            "cpu_baseline": {"value": round(val, 4), "unit": unit, "cores": o.threads(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(val, 4), "unit": unit, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main():
    args = parse()
    rank, world, local = dist_setup(args.gpus)
    if args.impl == "reference":
        line = run_reference(args, rank, world, local)
    else:
        line = run_ours(args, rank, world, local)
    if line is not None:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
