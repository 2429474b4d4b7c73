#!/usr/bin/env python
"""Throughput of one Mixtral-8x7B-shaped MoE FFN layer at decode on GB300.

One step is one pass of the whole path (router GEMM + softmax + top-k,
permute, expert up-projection, down-projection, combine) over each of the
decode batches T = 1, 4, 16, 64 of that layer (m=4096, p=14336, E=8, top-2,
SwiGLU experts, bf16 weights and activations; --weights i8 for the int8
repeat).  Inputs are seeded synthetic data resident in HBM; two copies of the
layer's weights alternate between calls, so no call finds the weights the
previous call read in L2 (every call streams >= 0.7 GB, L2 is 126 MB).

Prints one JSON line: whole-job tokens/s (all ranks), the roofline of the
dominant kernel (the expert up-projection GEMV) from CUDA events recorded on
its launch stream during the timed region, an end-to-end figure with host
buffers, sampled clocks, and the fp64 CPU oracle timed on a bounded sample.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--weights bf16|i8]
  python bench.py --impl reference ...   # the fp64 CPU oracle on host cores
"""
import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
T_START = time.perf_counter()
sys.path.insert(0, ROOT)

TOKENS = (1, 4, 16, 64)
METRIC = "MoE-layer tokens/s; HBM GB/s (decode) & tensor TFLOPS (batch) vs GB300 peak"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1,
                    help="GPUs (one process each under torchrun; each runs the whole step)")
    ap.add_argument("--steps", type=int, default=600, help="timed steps")
    ap.add_argument("--warmup", type=int, default=10, help="untimed warm-up steps (at least 3)")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"],
                    help="ours: the CUDA library; reference: the fp64 oracle on the host cores")
    ap.add_argument("--weights", default="bf16", choices=["bf16", "i8"],
                    help="expert weight type (i8: per-channel symmetric int8)")
    ap.add_argument("--seed", type=int, default=0, help="seed of the synthetic weights and tokens")
    ap.add_argument("--no-cpu-baseline", action="store_true", help="skip the oracle's timed sample")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end leg")
    ap.add_argument("--no-sub", action="store_true",
                    help="skip the int8-decode and batch sub-records of the default run")
    ap.add_argument("--tokens", default="1,4,16,64",
                    help="batch sizes of one step, comma-separated (each runs route + forward)")
    ap.add_argument("--copies", type=int, default=2, help="weight copies that alternate")
    ap.add_argument("--pair-tiles", type=int, default=1, choices=[0, 1],
                    help="up-projection 256-token tiles on CTA pairs (1, default) or one CTA each (0)")
    ap.add_argument("--graph", action="store_true",
                    help="capture one step (all route + forward calls) in a CUDA graph and "
                         "time its replays")
    ap.add_argument("--paged", action="store_true",
                    help="paged-weights run: many Mixtral-shaped layers in pinned host memory, "
                         "a capped GPU slot pool, a seeded decode routing trace")
    ap.add_argument("--paged-layers", type=int, default=32)
    ap.add_argument("--paged-steps", type=int, default=32)
    ap.add_argument("--paged-tokens", type=int, default=16, help="decode batch per layer")
    ap.add_argument("--paged-budget-gib", type=float, default=16.0)
    ap.add_argument("--paged-ways", type=int, default=4)
    ap.add_argument("--paged-page-mib", type=int, default=16,
                    help="granularity of the host-to-device page copies, MiB")
    ap.add_argument("--paged-prefetch", type=int, default=0,
                    help="experts each paged layer prefetches for the next layer (0: off)")
    ap.add_argument("--paged-route-inline", action="store_true",
                    help="route each paged layer on the compute stream right before its forward "
                         "(default: a step's routing is issued ahead on a side stream)")
    ap.add_argument("--zipf", type=float, default=None,
                    help="router bias making expert popularity Zipf(s) (batch workloads)")
    ap.add_argument("--shape", default="mixtral", choices=["mixtral", "phi", "small"],
                    help="mixtral (the benchmark), phi (Phi-3.5-MoE), small (profiling: "
                         "m=4096, p=3584, E=8, 0.7 GB of weights)")
    args = ap.parse_args()
    global TOKENS
    TOKENS = tuple(int(t) for t in args.tokens.split(","))
    return args


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return d["hbm_gbs"], d["bf16_tflops"], d.get("bf16_tflops_sustained"), "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


# ---- clocks --------------------------------------------------------------------------
class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.file = None

    def start(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.file, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.file.flush()
        self.file.seek(0)
        rows = [l.strip().split(", ") for l in self.file.read().splitlines() if l.strip()]
        os.unlink(self.file.name)
        sm = [float(r[1]) for r in rows if len(r) >= 9 and r[1].replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if len(r) >= 9 and r[2].replace(".", "").isdigit()]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            if len(r) < 9:
                continue
            for n, v in zip(names, r[5:9]):
                if v.strip().lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---- distributed plumbing (replicas only: no collective on the data path) ----------
def dist_setup(args):
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    gpu = args.impl == "ours" and torch.cuda.is_available()
    if world > 1:
        import torch.distributed as dist
        if gpu:
            torch.cuda.set_device(local)
        dist.init_process_group(backend="nccl" if gpu else "gloo")
    elif gpu:
        torch.cuda.set_device(0)
    return world, rank, local


def job_value(world, tokens_per_step, steps, ms_max):
    """Whole-job tokens/s of `world` replicas that each ran `steps` steps of
    `tokens_per_step` tokens, timed by the slowest rank (ms_max)."""
    return world * tokens_per_step * steps / (ms_max * 1e-3)


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(world, value):
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64,
                     device="cuda" if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---- CPU oracle (baseline leg and the reference arm) ---------------------------------
def oracle_sample(layer, xs, sample_tokens):
    """Route every token of each batch and evaluate the experts of the first
    `sample_tokens[T]` tokens, exactly as the oracle stands."""
    import oracle
    n = 0
    for T, x in xs.items():
        logits = oracle.router_logits(x, layer.w_router, layer.b_router)
        ids, w = oracle.topk(logits, layer.shape.k)
        s = sample_tokens[T]
        if s:
            oracle.layer(x, layer.w1, layer.w2, layer.w3, ids, w, oracle.SWIGLU,
                         tokens=list(range(s)))
            n += s
    return n


def cpu_threads():
    try:
        return int(os.environ.get("OMP_NUM_THREADS") or len(os.sched_getaffinity(0)))
    except AttributeError:
        return os.cpu_count() or 1


def make_tokens_for(shape, tokens, seed, device):
    import workloads as wl
    return {T: wl.make_tokens(shape, T, seed=seed + 1, device=device) for T in tokens}


def make_inputs(shape, seed, device, tokens):
    import workloads as wl
    layer = wl.make_layer(shape, seed=seed, device=device)
    return layer, make_tokens_for(shape, tokens, seed, device)


def shape_of(args):
    import dataclasses

    import workloads as wl
    base = {"mixtral": wl.MIXTRAL, "phi": wl.PHI35,
            "small": dataclasses.replace(wl.MIXTRAL, name="profile-small", p=3584)}[args.shape]
    if args.zipf is not None:
        base = base.with_zipf(args.zipf)
    return base if args.weights == "bf16" else base.with_weight("i8")


def workload_config(shape, weights, tokens):
    """The workload both arms time: layer shape, batches of one step, and how
    the inputs relate to L2 (identical for the GPU and the CPU arm)."""
    ts = ",".join(str(t) for t in tokens)
    regime = "decode" if max(tokens) <= 64 else "batch"
    b = 1 if weights == "i8" else 2
    min_gb = shape.k * (3 if shape.has_w3 else 2) * shape.m * shape.p * b / 1e9
    return {"workload": f"{shape.name}-shaped MoE FFN layer, {regime}, T in {{{ts}}}, {weights} weights",
            "m": shape.m, "p": shape.p, "E": shape.E, "k": shape.k, "expert": "swiglu",
            "tokens_per_step": sum(tokens), "parallelism": "replicas",
            "l2": f"inputs larger than L2: every call streams >= {min_gb:.2f} GB of expert weights"}


def run_reference(args, world, rank):
    if rank != 0:
        return
    shape = shape_of(args)
    import torch
    device = "cuda" if torch.cuda.is_available() else "cpu"
    layer, xs = make_inputs(shape, args.seed, device, TOKENS)
    # Every token is routed each step; the expert MLPs run for one token per
    # host thread, taken from the batch that has that many (the oracle runs its
    # tokens in parallel, so a step costs about one token's MLPs).
    threads = cpu_threads()
    t_big = max(TOKENS, key=lambda T: min(T, threads))
    n_exp = min(t_big, threads)
    sample = {T: (n_exp if T == t_big else 0) for T in TOKENS}
    for _ in range(args.warmup):
        oracle_sample(layer, xs, sample)
    t0 = time.perf_counter()
    n = 0
    for _ in range(args.steps):
        n += oracle_sample(layer, xs, sample)
    dt = time.perf_counter() - t0
    value = n / dt
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": dt * 1e3 / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(shape, args.weights, TOKENS),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cpu_threads(),
                             "kind": "oracle",
                             "sample": f"per step: router + top-k for all {sum(TOKENS)} tokens of the "
                                       f"batches, expert MLPs for {n_exp} tokens of the T={t_big} batch "
                                       "(one per host thread), fp64"},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---- our arm ----------------------------------------------------------------------------
def traffic_record():
    """DRAM bytes of the up-projection per step from the committed ncu summary,
    if every kernel source it was taken on is unchanged; else None."""
    path = os.path.join(ROOT, "profiles", "decode_up_traffic.json")
    if not os.path.exists(path):
        return None
    rec = json.load(open(path))
    for rel, sha in rec.get("source_sha256", {}).items():
        src = os.path.join(ROOT, rel)
        if not os.path.exists(src) or hashlib.sha256(open(src, "rb").read()).hexdigest() != sha:
            return None
    return rec


def capture(torch, fn, layers):
    """A CUDA graph of fn() (route + forward calls on the current stream) and
    the number of library kernel launches it holds."""
    n0 = sum(c.stats().kernel_launches for c in layers)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    torch.cuda.synchronize()
    return g, sum(c.stats().kernel_launches for c in layers) - n0


def measure(args, world, local, shape, layer, tokens, xs_np, steps, warmup, weights,
            graph=False, e2e=False, traffic=None):
    """Time `steps` steps, each route + forward for every batch size of
    `tokens` on its own seeded tokens, over two (--copies) alternating copies
    of `layer`'s weights.  Returns the measured record: whole-step time (CUDA
    events on the launch stream, no per-launch events), the dominant kernel's
    roofline and the per-batch breakdown from an event-timed second pass,
    sampled clocks, launches, and optionally the end-to-end leg with host
    buffers."""
    import numpy as np
    import torch

    import mixture_experts_layer_gemm_gb300 as moe

    max_t = max(tokens)
    copies = [moe.MoELayer(layer, max_t) for _ in range(max(args.copies, 1))]
    for c in copies:
        c.set_pair_tiles(bool(args.pair_tiles))
    dev = torch.device("cuda", local)
    xs = {T: torch.from_numpy(xs_np[T].view(np.int16).copy()).view(torch.bfloat16).to(dev)
          for T in tokens}
    ys = {T: torch.empty((T, shape.m), dtype=torch.bfloat16, device=dev) for T in tokens}
    stream = torch.cuda.current_stream()

    def step():  # on the current stream (the capture stream while a graph is captured)
        for i, T in enumerate(tokens):
            c = copies[i % len(copies)]
            c.route(xs[T])
            c.forward(xs[T], ys[T])

    for _ in range(max(warmup, 3)):
        step()
    torch.cuda.synchronize()
    launches_per_step = None
    run_step = step
    if graph:
        g, launches_per_step = capture(torch, step, copies)
        run_step = g.replay
        for _ in range(max(warmup, 3)):
            run_step()
        torch.cuda.synchronize()
    for c in copies:
        st, flags = c.sync_check()
        if st != moe.MOE_OK:
            raise RuntimeError(f"device flagged routing error bits {flags:#x}")
    launches0 = sum(c.stats().kernel_launches for c in copies)

    clocks = ClockSampler(local)
    barrier(world)
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for _ in range(steps):
        run_step()
    ev1.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    barrier(world)
    ms = ev0.elapsed_time(ev1)
    ms_max = max_over_ranks(world, ms)
    launches = (launches_per_step * steps if graph
                else sum(c.stats().kernel_launches for c in copies) - launches0)

    # Per-launch kernel durations.  Kernels of one call are launched with
    # programmatic dependent launch, so each may start while its predecessor
    # drains; an event recorded between two launches breaks that overlap.  The
    # timed region above therefore runs without per-launch events, and the
    # same steps run again here with them, for the roofline and the breakdown.
    for c in copies:
        c.set_timing(True)
        c.timings(reset=True)
    ev2, ev3 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev2.record(stream)
    for _ in range(steps):
        step()
    ev3.record(stream)
    torch.cuda.synchronize()
    ms_events = ev2.elapsed_time(ev3)
    tim = [c.timings(reset=True) for c in copies]
    for c in copies:
        c.set_timing(False)

    # ---- algorithmic work per call (per-unit bytes and flops of each kernel) -----------
    # up: active experts' W1 and W3 (+ int8 scales), token rows read, hidden rows written;
    #     flops 2 * (2 m p) per routed (token, slot) for SwiGLU (2 m p for ReLU)
    # down: active experts' W2 (+ scales), hidden rows read; flops 2 m p per (token, slot)
    # layer (the per-batch roof): active experts' weights plus x in and y out at
    #     decode; weights plus T k (m + p + m) bf16 activations on the tensor-core
    #     path (permuted rows, hidden rows, expert outputs)
    wbytes = 1 if weights == "i8" else 2
    n_up = 2 if shape.has_w3 else 1
    work, active = {}, {}
    for i, T in enumerate(tokens):
        c = copies[i % len(copies)]
        c.route(xs[T], stream=stream)
        tc0 = c.stats().tc_runs
        c.forward(xs[T], ys[T], stream=stream)  # which regime the library chose for T
        torch.cuda.synchronize()
        path = "tensor-core" if c.stats().tc_runs > tc0 else "gemv"
        n_act = int((c.counts.cpu() > 0).sum())
        active[T] = n_act
        scale_up = n_up * shape.p * 4 if weights == "i8" else 0
        scale_dn = shape.m * 4 if weights == "i8" else 0
        rows = T * shape.k
        w_all = n_act * ((n_up + 1) * shape.m * shape.p * wbytes + scale_up + scale_dn)
        work[T] = {
            "up_bytes": n_act * (n_up * shape.m * shape.p * wbytes + scale_up) + T * shape.m * 2
            + rows * shape.p * 2,
            "down_bytes": n_act * (shape.m * shape.p * wbytes + scale_dn) + rows * shape.p * 2,
            "up_flops": 2.0 * n_up * shape.m * shape.p * rows,
            "down_flops": 2.0 * shape.m * shape.p * rows,
            "layer_bytes": w_all + (T * shape.m * 2 * 2 if path == "gemv"
                                    else rows * (2 * shape.m + shape.p) * 2),
            "path": path}
        work[T]["layer_flops"] = work[T]["up_flops"] + work[T]["down_flops"]
    bytes_up = sum(w["up_bytes"] for w in work.values())
    bytes_down = sum(w["down_bytes"] for w in work.values())
    flops_up = sum(w["up_flops"] for w in work.values())
    up_ms = sum(t["up"][0] for t in tim)
    up_n = sum(t["up"][1] for t in tim)
    phase_ms = {k: sum(t[k][0] for t in tim) / steps for k in tim[0]}
    hbm, tf, tf_sus, src = peaks()
    layer_bytes = bytes_up + bytes_down
    layer_gbs = layer_bytes * steps / (ms * 1e-3) / 1e9
    layer_flops = flops_up + sum(w["down_flops"] for w in work.values())
    layer_tf = layer_flops * steps / (ms * 1e-3) / 1e12

    # per-T breakdown: each batch alone; first its wall time per layer call
    # (route + forward, no per-launch events, so programmatic launch overlaps
    # the kernels as in the timed region), then every launch event-timed
    per_t = {}
    for i, T in enumerate(tokens):
        w0, w1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        w0.record(stream)
        for it in range(20):
            c = copies[it % len(copies)]
            c.route(xs[T], stream=stream)
            c.forward(xs[T], ys[T], stream=stream)
        w1.record(stream)
        torch.cuda.synchronize()
        wall_us = w0.elapsed_time(w1) / 20 * 1e3
        for c in copies:
            c.timings(reset=True)
            c.set_timing(True)
        for it in range(20):
            c = copies[it % len(copies)]
            c.route(xs[T], stream=stream)
            c.forward(xs[T], ys[T], stream=stream)
        torch.cuda.synchronize()
        tt = [c.timings(reset=True) for c in copies]
        for c in copies:
            c.set_timing(False)
        u_ms = sum(t["up"][0] for t in tt) / 20
        d_ms = sum(t["down"][0] for t in tt) / 20
        tot = sum(sum(v[0] for v in t.values()) for t in tt) / 20
        w = work[T]
        pl = copies[0].plan(T)  # the launch plan the forward took (moe_plan_forward)
        plan = {f: int(getattr(pl, f)) for f in ("tile_up", "tile_down", "splits_up", "splits_down", "pair_up")}
        if moe.PATHS[pl.path] != w["path"]:
            raise RuntimeError(f"T = {T}: plan says {moe.PATHS[pl.path]}, the forward ran {w['path']}")
        # the batch's own roof: min(tensor peak, HBM peak x intensity), as a time
        t_hbm = w["layer_bytes"] / (hbm * 1e9) * 1e6
        t_tc = w["layer_flops"] / (tf * 1e12) * 1e6
        roof_us = max(t_hbm, t_tc)
        per_t[str(T)] = {"path": w["path"], "plan": plan, "active_experts": active[T],
                         "layer_us_wall": wall_us, "layer_us": tot * 1e3,
                         "up_us": u_ms * 1e3, "down_us": d_ms * 1e3,
                         "up_gbs": w["up_bytes"] / (u_ms * 1e-3) / 1e9,
                         "down_gbs": w["down_bytes"] / (d_ms * 1e-3) / 1e9,
                         "up_tflops": w["up_flops"] / (u_ms * 1e-3) / 1e12,
                         "down_tflops": w["down_flops"] / (d_ms * 1e-3) / 1e12,
                         "layer_gbs": w["layer_bytes"] / (tot * 1e-3) / 1e9,
                         "layer_tflops": w["layer_flops"] / (tot * 1e-3) / 1e12,
                         "roof": {"bound": "tensor" if t_tc > t_hbm else "hbm", "us": roof_us,
                                  "frac": roof_us / (tot * 1e3), "frac_wall": roof_us / wall_us}}

    # the dominant kernel: the expert up-projection; HBM-bound while the batch is
    # weight-streaming, tensor-bound once most of the work runs on the tensor-core path
    tensor_bound = sum(w["up_flops"] for w in work.values() if w["path"] == "tensor-core") > \
        0.5 * flops_up and max(tokens) >= 256
    if tensor_bound:
        # each up-projection launch runs for milliseconds inside a multi-ms step:
        # the sustained (power-capped) peak is the denominator, the burst one beside it
        achieved = flops_up * steps / (up_ms * 1e-3) / 1e12
        peak = tf_sus or tf
        roofline = {"kernel": "expert up-projection (W1 and W3 + SiLU*gate), tcgen05 grouped GEMM",
                    "bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                    "frac": achieved / peak,
                    "peak_source": f"{src} (bf16_tflops_sustained)" if tf_sus else f"{src} (bf16_tflops)",
                    "frac_of_burst": achieved / tf, "peak_burst": tf,
                    "algorithmic_flops_per_step": flops_up,
                    "avg_launch_us": up_ms * 1e3 / max(up_n, 1), "traffic": None}
    else:
        achieved = bytes_up * steps / (up_ms * 1e-3) / 1e9
        gemv_t = [T for T in tokens if work[T]["path"] == "gemv"]
        tc_t = [T for T in tokens if work[T]["path"] != "gemv"]
        paths = ", ".join(p for p in (f"decode GEMV for T in {gemv_t}" if gemv_t else "",
                                      f"tcgen05 for T in {tc_t}" if tc_t else "") if p)
        roofline = {"kernel": f"expert up-projection (W1 and W3 + SiLU*gate): {paths}",
                    "bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                    "frac": achieved / hbm, "peak_source": f"{src} (hbm_gbs)",
                    "algorithmic_bytes_per_step": bytes_up,
                    "avg_launch_us": up_ms * 1e3 / max(up_n, 1),
                    "traffic": None if traffic is None else traffic.get("bytes_per_step")}

    tokens_step = sum(tokens)
    rec = {"value": job_value(world, tokens_step, steps, ms_max), "unit": "tokens/s",
           "steps": steps, "warmup": warmup, "ms_per_step": ms_max / steps,
           "config": workload_config(shape, weights, tokens),
           "roofline": roofline,
           "layer_hbm": {"achieved": layer_gbs, "unit": "GB/s", "frac": layer_gbs / hbm,
                         "algorithmic_bytes_per_step": layer_bytes,
                         "note": "whole step: expert weights + activations / step time"},
           "layer_tflops": layer_tf,
           "phase_ms_per_step": phase_ms,
           "ms_per_step_with_launch_events": ms_events / steps,
           "active_experts": active, "per_T": per_t,
           "per_T_note": "layer_us_wall: route + forward of one batch timed as a whole (launches overlap "
                         "as in the timed region); layer_us, up_us, down_us: sums of per-launch events, "
                         "each of which ends the programmatic overlap of the launches around it",
           "gpu_launches": launches, "clocks": clk}
    if tensor_bound:
        rec["layer_tensor"] = {"achieved": layer_tf, "unit": "TFLOP/s",
                               "frac": layer_tf / (tf_sus or tf), "frac_of_burst": layer_tf / tf,
                               "note": "whole step: all expert flops / step time"}

    if e2e and not args.no_e2e:
        rec["e2e"] = measure_e2e(args, world, copies, shape, tokens, xs, ys, stream, steps, graph)
    for c in copies:
        c.close()
    return rec


def measure_e2e(args, world, copies, shape, tokens, xs, ys, stream, steps, graph):
    """The same step through the public API with pinned host buffers: every
    step copies its inputs in and reads its result back inside the timed
    region, which ends once the last result is on the host."""
    import torch

    xh = {T: xs[T].cpu().pin_memory() for T in tokens}
    yh = {T: torch.empty((T, shape.m), dtype=torch.bfloat16).pin_memory() for T in tokens}
    xd = {T: torch.empty_like(xs[T]) for T in tokens}

    def step_e2e():  # one stream: copy in, compute, copy out (the form a graph captures)
        for i, T in enumerate(tokens):
            c = copies[i % len(copies)]
            xd[T].copy_(xh[T], non_blocking=True)
            c.route(xd[T])
            c.forward(xd[T], ys[T])
            yh[T].copy_(ys[T], non_blocking=True)

    # As a server would, the eager form runs the copies on two side streams
    # and overlaps them with the neighbouring steps' compute: step i's inputs
    # go into one of two device buffers while step i - 1 computes, and its
    # outputs come back while step i + 1 computes.  Every step still copies its
    # inputs in and reads its result back inside the timed region, which ends
    # when the last result is on the host.
    h2d_stream, d2h_stream = torch.cuda.Stream(), torch.cuda.Stream()
    xd2 = [{T: torch.empty_like(xs[T]) for T in tokens} for _ in range(2)]
    yd2 = [{T: torch.empty_like(ys[T]) for T in tokens} for _ in range(2)]
    ev_in = [torch.cuda.Event() for _ in range(2)]    # inputs of buffer b on the device
    ev_done = [torch.cuda.Event() for _ in range(2)]  # compute on buffer b finished
    ev_back = [torch.cuda.Event() for _ in range(2)]  # outputs of buffer b on the host
    pipe = {"it": 0}

    def step_e2e_pipelined():
        b = pipe["it"] % 2
        pipe["it"] += 1
        with torch.cuda.stream(h2d_stream):
            h2d_stream.wait_event(ev_done[b])  # the step two back finished reading buffer b
            for T in tokens:
                xd2[b][T].copy_(xh[T], non_blocking=True)
            ev_in[b].record(h2d_stream)
        stream.wait_event(ev_in[b])
        stream.wait_event(ev_back[b])  # buffer b's previous outputs have been read back
        for i, T in enumerate(tokens):
            c = copies[i % len(copies)]
            c.route(xd2[b][T])
            c.forward(xd2[b][T], yd2[b][T])
        ev_done[b].record(stream)
        with torch.cuda.stream(d2h_stream):
            d2h_stream.wait_event(ev_done[b])
            for T in tokens:
                yh[T].copy_(yd2[b][T], non_blocking=True)
            ev_back[b].record(d2h_stream)

    def e2e_drain():  # the timed region closes once the last result is on the host
        stream.wait_event(ev_back[(pipe["it"] - 1) % 2])

    k_e2e = max(steps // 2, 1)
    run_step, drain = step_e2e_pipelined, e2e_drain
    if graph:
        for _ in range(3):
            step_e2e()
        torch.cuda.synchronize()
        run_step, drain = capture(torch, step_e2e, copies)[0].replay, (lambda: None)
    for _ in range(3):
        run_step()
    drain()
    torch.cuda.synchronize()
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(k_e2e):
        run_step()
    drain()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(world, e0.elapsed_time(e1))
    io_bytes = sum(T * shape.m * 2 for T in tokens)
    return {"value": job_value(world, sum(tokens), k_e2e, e2e_ms), "unit": "tokens/s",
            "h2d_bytes_per_step": io_bytes, "d2h_bytes_per_step": io_bytes,
            "copies": ("on the compute stream, inside the captured step" if graph else
                       "pinned host buffers, on two side streams overlapped with the "
                       "neighbouring steps' compute (double-buffered device inputs and outputs)")}


def run_ours(args, world, rank, local):
    import dataclasses

    import workloads as wl
    from mixture_experts_layer_gemm_gb300 import build as lib_build

    lib_build.build()
    shape = shape_of(args)
    device = f"cuda:{local}"
    layer, xs_np = make_inputs(shape, args.seed + rank, device, TOKENS)
    headline_default = (args.shape == "mixtral" and args.weights == "bf16" and args.zipf is None
                        and TOKENS == wl.DECODE_TOKENS)
    trec = traffic_record() if headline_default else None
    rec = measure(args, world, local, shape, layer, TOKENS, xs_np, args.steps, args.warmup,
                  args.weights, graph=args.graph, e2e=True, traffic=trec)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        # every token is routed; the expert MLPs run for at most 256 tokens,
        # shared over the batches in proportion to their size (the whole step
        # at decode sizes: ~3 s on 16 Grace cores)
        total = sum(TOKENS)
        sample = {T: (T if total <= 256 else max(1, 256 * T // total)) for T in TOKENS}
        t0 = time.perf_counter()
        n = oracle_sample(layer, xs_np, sample)
        dt = time.perf_counter() - t0
        what = (f"the whole step ({n} tokens: router, top-k and the expert MLP of every routed "
                "(token, slot))" if n == total else
                f"router and top-k for all {total} tokens, expert MLPs for {n} of them (the first "
                f"{', '.join(str(sample[T]) for T in TOKENS)} of the batches); tokens/s of that sample")
        cpu = {"value": n / dt, "unit": "tokens/s", "cores": cpu_threads(), "kind": "oracle",
               "sample": f"{what}, fp64, one pass"}

    # The metric's other halves, measured in the same run on the same layer
    # weights: the int8 repeat of the decode step, and the batch regime
    # (T = 512, 2048, 8192 with a Zipf(1.2) router bias), whose expert GEMMs
    # are tensor-bound; then the Phi-3.5-MoE-shaped layer.  Each is its own
    # timed region with its own clocks.
    subs = {}
    if headline_default and not args.no_sub:
        lay_i8 = dataclasses.replace(layer, shape=shape.with_weight("i8"))
        subs["int8_decode"] = measure(args, world, local, lay_i8.shape, lay_i8, TOKENS, xs_np,
                                      max(args.steps, 200), args.warmup, "i8")
        zshape = shape.with_zipf(1.2)
        lay_b = dataclasses.replace(layer, shape=zshape, b_router=wl.zipf_bias(zshape.E, 1.2))
        bt = wl.BATCH_TOKENS
        xb = make_tokens_for(zshape, bt, args.seed + rank, device)
        subs["batch"] = measure(args, world, local, zshape, lay_b, bt, xb, max(args.steps, 40),
                                args.warmup, "bf16")
        # the Phi-3.5-MoE-shaped layer (16 smaller experts), uniform routing,
        # over the batch sizes of its configuration, decode to batch
        pshape = wl.PHI35
        lay_p = wl.make_layer(pshape, seed=args.seed + rank, device=device)
        pt = wl.PHI_TOKENS
        xp = make_tokens_for(pshape, pt, args.seed + rank, device)
        subs["phi"] = measure(args, world, local, pshape, lay_p, pt, xp, max(args.steps, 40),
                              args.warmup, "bf16")

    if rank == 0:
        line = {"metric": METRIC, "value": rec["value"], "unit": "tokens/s", "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": rec["ms_per_step"],
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                # MMA input type (fp32 accumulation): int8 weights are widened
                # exactly to fp16 in the GEMV and to bf16 on the tensor cores
                "dtype": "bf16" if args.weights == "bf16" else "i8->f16/bf16", "data": "synthetic",
                "config": rec["config"],
                "timing": {"weight_copies": max(args.copies, 1),
                           "launch": "one CUDA graph per step, replayed" if args.graph
                           else "stream launches with programmatic dependent launch"}}
        for key in ("roofline", "layer_hbm", "layer_tensor", "layer_tflops", "phase_ms_per_step",
                    "ms_per_step_with_launch_events", "active_experts", "per_T", "per_T_note"):
            if key in rec:
                line[key] = rec[key]
        line["cpu_baseline"] = cpu
        line["e2e"] = rec.get("e2e")
        line["gpu_launches"] = rec["gpu_launches"]
        line["clocks"] = rec["clocks"]
        for name, sub in subs.items():
            sub["dtype"] = "i8->f16/bf16" if name == "int8_decode" else "bf16"
            line[name] = sub
        line["wall_s"] = time.perf_counter() - T_START
        print(json.dumps(line), flush=True)



# ---- paged weights (expert-cache configuration) -----------------------------------------
def host_mem_available():
    for line in open("/proc/meminfo"):
        if line.startswith("MemAvailable:"):
            return int(line.split()[1]) * 1024
    return 0


def link_h2d_gbs(torch, nbytes=1 << 30):
    """Pinned host-to-device copy bandwidth of this machine (cudaMemcpyAsync)."""
    h = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    d = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        for _ in range(2):
            d.copy_(h, non_blocking=True)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s)
        for _ in range(5):
            d.copy_(h, non_blocking=True)
        e1.record(s)
    torch.cuda.synchronize()
    gbs = 5 * nbytes / (e0.elapsed_time(e1) * 1e-3) / 1e9
    del h, d
    return gbs


def run_paged(args, world, rank, local):
    """Decode T=16 through many paged Mixtral-shaped layers sharing a slot pool
    (N-index x M-way, set = layer mod N), fed a seeded routing trace in which a
    layer repeats the previous layer's experts with p = 0.44 and the previous
    token's with p = 0.5 (expert-cache article, section 2.1)."""
    import numpy as np
    import torch

    import mixture_experts_layer_gemm_gb300 as moe
    import workloads as wl
    from mixture_experts_layer_gemm_gb300 import build as lib_build

    lib_build.build()
    shape = wl.MIXTRAL if args.weights == "bf16" else wl.MIXTRAL.with_weight("i8")
    T, L, S = args.paged_tokens, args.paged_layers, args.paged_steps
    layer = wl.make_layer(shape, seed=args.seed + rank, device=f"cuda:{local}")
    probe = moe.MoELayer(layer, T)
    eb = probe.info().expert_bytes
    probe.close()
    need = int(1.15 * L * shape.E * (eb + 1024)) + (8 << 30)
    avail = host_mem_available()
    if avail < need:
        raise SystemExit(f"paged run needs ~{need / 1e9:.0f} GB of host memory, "
                         f"{avail / 1e9:.0f} GB available")
    link = link_h2d_gbs(torch)
    budget = int(args.paged_budget_gib * (1 << 30))
    n_index, n_slots = moe.moe_pool_geometry(budget, eb, args.paged_ways)
    pool = moe.moe_pool_create(budget, eb, args.paged_ways, args.paged_page_mib << 20)
    moe.moe_pool_set_prefetch(pool, args.paged_prefetch)
    layers = [moe.MoELayer(layer, T, pool=pool, layer_id=l) for l in range(L)]
    ids, w = wl.make_topk_trace(shape.E, shape.k, S + 1, L, T, seed=args.seed)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream()
    gen = torch.Generator(device=dev)
    gen.manual_seed(args.seed + 17)
    ids_d = torch.from_numpy(ids.reshape(S + 1, L, T * shape.k)).to(dev)
    w_d = torch.from_numpy(w.reshape(S + 1, L, T * shape.k)).to(dev)
    y = torch.empty((T, shape.m), dtype=torch.bfloat16, device=dev)
    # fresh N(0,1) token rows per (step, layer), drawn before the timed region
    xs = torch.randn((S + 1, L, T, shape.m), generator=gen, device=dev).to(torch.bfloat16)

    # The trace's routing does not depend on the previous layer's output, so
    # by default a step routes all its layers first on a side stream, each
    # layer's routing after that layer's previous forward (which read the
    # tables it overwrites); each paged forward then reads its counts there and
    # issues its page copies while the earlier layers still compute.
    # --paged-route-inline routes each layer on the compute stream just before
    # its forward, as a model whose next routing waits for this layer's output
    # would.
    route_stream = torch.cuda.Stream(device=dev)
    layer_done = [torch.cuda.Event() for _ in layers]

    def step(s):
        if args.paged_route_inline:
            for l, ml in enumerate(layers):
                ml.route_from_topk(ids_d[s, l], w_d[s, l], T=T, stream=stream)
                ml.forward(xs[s, l], y, stream=stream)
            return
        for l, ml in enumerate(layers):
            route_stream.wait_event(layer_done[l])
            ml.route_from_topk(ids_d[s, l], w_d[s, l], T=T, stream=route_stream)
        for l, ml in enumerate(layers):
            ml.forward(xs[s, l], y, stream=stream)
            layer_done[l].record(stream)

    step(0)  # warm-up: kernels, tensor maps, first slot fills
    torch.cuda.synchronize()
    for ml in layers:
        ml.set_timing(True)
        ml.timings(reset=True)
    st0 = [ml.stats() for ml in layers]
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for s_ in range(1, S + 1):
        step(s_)
    e1.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    wall_ms = e0.elapsed_time(e1)
    st1 = [ml.stats() for ml in layers]
    tim = [ml.timings(reset=True) for ml in layers]
    hits = sum(b.slot_hits - a.slot_hits for a, b in zip(st0, st1))
    misses = sum(b.slot_misses - a.slot_misses for a, b in zip(st0, st1))
    h2d = sum(b.h2d_bytes - a.h2d_bytes for a, b in zip(st0, st1))
    pf_copies = sum(b.prefetch_copies - a.prefetch_copies for a, b in zip(st0, st1))
    pf_hits = sum(b.prefetch_hits - a.prefetch_hits for a, b in zip(st0, st1))
    copy_ms = sum(t["copy"][0] for t in tim)
    compute_ms = sum(sum(v[0] for k, v in t.items() if k != "copy") for t in tim)
    overlap = (copy_ms + compute_ms - wall_ms) / max(min(copy_ms, compute_ms), 1e-9)
    for ml in layers:
        ml.close()
    moe.moe_pool_destroy(pool)
    value = S * T / (wall_ms * 1e-3)
    line = {"metric": f"MoE-layer tokens/s, paged expert weights (decode, T={T} per layer)",
            "value": value, "unit": "tokens/s", "n_gpus": 1, "steps": S, "warmup": 1,
            "ms_per_step": wall_ms / S, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": args.weights, "data": "synthetic",
            "config": {"workload": f"{L} paged mixtral-8x7b moe layers, decode T={T}, "
                                   f"{args.paged_budget_gib:g} GiB slot pool, "
                                   f"{n_index} sets x {args.paged_ways} ways, "
                                   f"prefetch {args.paged_prefetch}",
                       "layers": L, "T": T, "trace": "p_layer=0.44, p_token=0.5, seeded",
                       "routing": ("each layer on the compute stream before its forward" if args.paged_route_inline
                                   else "a step's layers routed ahead on a side stream"),
                       "tokens_per_step": T},
            "paged": {"sets": n_index, "ways": args.paged_ways, "slots": n_slots,
                      "expert_bytes": eb, "hit_rate": hits / max(hits + misses, 1),
                      "hits": hits, "misses": misses, "h2d_bytes": h2d,
                      "page_mib": args.paged_page_mib,
                      "prefetch": args.paged_prefetch, "prefetch_copies": pf_copies,
                      "prefetch_hits": pf_hits,
                      "prefetch_used_frac": pf_hits / max(pf_copies, 1),
                      "h2d_gbs_copy_stream": h2d / max(copy_ms * 1e-3, 1e-12) / 1e9,
                      "h2d_gbs_wall": h2d / (wall_ms * 1e-3) / 1e9,
                      "link_gbs_measured": link,
                      "link_frac": (h2d / max(copy_ms * 1e-3, 1e-12) / 1e9) / link,
                      "copy_ms": copy_ms, "compute_ms": compute_ms, "wall_ms": wall_ms,
                      "overlap_frac": max(0.0, min(1.0, overlap)),
                      "bounds_ms": [max(copy_ms, compute_ms), copy_ms + compute_ms]},
            "clocks": clk}
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    world, rank, local = dist_setup(args)
    if args.impl == "reference":
        run_reference(args, world, rank)
    elif args.paged:
        run_paged(args, world, rank, local)
    else:
        run_ours(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
