#!/usr/bin/env python
"""Benchmark of the submanifold convolution hot path on one B300 (or N replicas).

One step = the whole path over one synthetic voxel set: subm3d_build_kmap
(validate/pack, Morton radix sort, hash insert, 27-offset probe) followed by
subm3d_forward (tcgen05 gather-GEMM with fused bias). Default workload: the
1024^3 grid with 16 ellipsoid/torus shells (~2.9 M voxels), I = O = 64, bf16.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload 1..5]
    python bench.py --impl reference ...      # the CPU oracle, as the reference arm
    python bench.py --residual --act relu     # forward with the fused block epilogue
    python bench.py --op downsample|upsample  # SparseDownsample(2) / SparseUpsample(2)
    python bench.py --op spatial2channel|channel2spatial   # sparse pixel-(un)shuffle

Prints one JSON line (rank 0). `value` = effective TFLOP/s of the whole step,
2 * pairs * I * O / step time, summed over ranks (replicas: every rank runs the
full workload). Inputs are resident in HBM before timing; they are larger than L2,
so L2 is not flushed between steps. `e2e` repeats the measurement through the
Python API with pinned-host inputs copied in and the output copied back every step.
"""
from __future__ import annotations

import argparse
import gc
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

METRIC = "SubMConv3d bf16 TFLOP/s & Mvoxels/s (fraction of roofline); kmap build ms"
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}
CPU_SAMPLE_VOXELS = 4_000_000      # oracle CPU baseline: up to the first 4 M voxels (raster order)
REF_STEP_FLOPS = 2e9               # reference arm: ~2 GFLOP of oracle work per step
CSRC = os.path.join(ROOT, "submanifold_sparse_convolution_04_b300", "csrc")


def forward_kernel(I, O):
    """(kernel name, source file) of the bf16 forward the library picks for I x O: the
    narrow kernel (gathered rows in tensor memory) for I, O in {16, 32, 48, 64}, else
    the shared-memory-staged one, its rows gathered by TMA when I is a multiple of 64,
    by cp.async otherwise."""
    if I in (16, 32, 48, 64) and O in (16, 32, 48, 64):
        return "fwd_tm", os.path.join(CSRC, "forward_tm.cu")
    if I % 64 == 0:
        return "fwd_tc_tg", os.path.join(CSRC, "forward_tc.cu")
    return "fwd_tc", os.path.join(CSRC, "forward_tc.cu")


def parse_args():
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--workload", type=int, default=5, choices=[1, 2, 3, 4, 5])
    p.add_argument("--order", default="raster", choices=["raster", "shuffled"])
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--e2e-steps", type=int, default=20)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--op", default="conv",
                   choices=["conv", "downsample", "upsample", "spatial2channel", "channel2spatial"],
                   help="conv: kmap + forward (the default step); the others: SparseDownsample(2), "
                        "its paired SparseUpsample(2), SparseSpatial2Channel(2) and its inverse on "
                        "the workload's voxels and features")
    p.add_argument("--ds-sort", action="store_true",
                   help="--op downsample: sort the voxels itself (subm3d_downsample) instead of "
                        "taking the Morton order of the kernel map on the same voxels "
                        "(subm3d_downsample_sorted)")
    p.add_argument("--ds-wait", action="store_true",
                   help="--op downsample: the call that reads M back to the host every time "
                        "(one stream wait per call) instead of subm3d_downsample_async")
    p.add_argument("--pool", default="mean", choices=["mean", "max"],
                   help="pooling of --op downsample (and of the coarse rows --op upsample uses)")
    p.add_argument("--residual", action="store_true",
                   help="fused block epilogue: add a residual [N, O] input (subm3d_forward_ex)")
    p.add_argument("--act", default="none", choices=["none", "relu", "silu"],
                   help="fused block epilogue: activation after bias (+ residual)")
    p.add_argument("--max-voxels", type=int, default=0,
                   help="keep only the first M voxels (raster order): a slab of the workload")
    p.add_argument("--path", default="morton", choices=["morton", "grouped", "plain"],
                   help="morton: the kernel map as a tile plan of the Morton order (window 1) "
                        "and the forward on its tiles; grouped: a tile plan of mask-grouped "
                        "windows (--window); plain: the input-order nbr and its tiles")
    p.add_argument("--window", type=int, default=0,
                   help="grouping window of the tile plan (0: the library default)")
    p.add_argument("--graph", action="store_true",
                   help="replay each step's kernel map and forward from two CUDA graphs captured "
                        "once (launch-bound small workloads); implies the asynchronous kernel map")
    p.add_argument("--sync-kmap", action="store_true",
                   help="use the kernel-map call that waits for its stream (default: the "
                        "asynchronous one, device status checked after the timed steps)")
    return p.parse_args()


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def workload_desc(case, P):
    cfg = case
    return {"workload": f"{cfg['name']}: res {cfg['res']}^3, N={cfg['coords'].shape[0]}, "
                        f"I={cfg['I']}, O={cfg['O']}, {cfg['dtype']}",
            "name": cfg["name"], "res": cfg["res"], "N": int(cfg["coords"].shape[0]),
            "pairs": None if P is None else int(P), "I": cfg["I"], "O": cfg["O"],
            "order": cfg["info"]["order"]}


def load_case(args):
    from synth import make_case
    case = make_case(args.workload, args.order)
    M = args.max_voxels
    if M and M < case["coords"].shape[0]:
        for k in ("coords", "feats", "feats_bits"):
            if k in case:
                case[k] = case[k][:M]
        case["name"] += f"_first{M}"
        case["info"] = dict(case["info"], N=M)
    return case


# ------------------------------------------------------------------------- distributed

def dist_setup(n_gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    """Largest value of x over all ranks (x itself for one rank)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples (200 ms) of SM clock and throttle reasons during a region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200", "-i", str(self.gpu)], stdout=subprocess.PIPE,
                stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, ValueError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, smax, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm),
                "power_w_max": max(power) if power else None}


# ------------------------------------------------------------------------- roofline

def recorded_traffic(kernel, src, workload):
    """dram bytes per forward launch from the committed ncu summary of this kernel on
    this workload, if it was taken on the current kernel source (sha256 recorded beside
    the number)."""
    prof = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.md")
    if not os.path.exists(prof):
        return None, "no ncu summary"
    text = open(prof).read()
    m = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", text)
    h = re.search(r"source_sha256:\s*([0-9a-f]{64})", text)
    if not m or not h:
        return None, "ncu summary has no traffic line"
    cur = hashlib.sha256(open(src, "rb").read()).hexdigest()
    if h.group(1) != cur:
        return None, "kernel changed since the ncu capture"
    return float(m.group(1)), f"ncu dram__bytes_read.sum + dram__bytes_write.sum ({os.path.relpath(prof, ROOT)})"


def roofline(N, P, I, O, fwd_s, peaks, peak_kind, workload, e=2, residual=False):
    """e: bytes per element of feats, weight and out (2 for bf16, 4 for fp32); residual:
    the fused epilogue reads an [N, O] residual as well."""
    gathered = P * I * e + N * O * e + 108 * N + 27 * I * O * e + (N * O * e if residual else 0)
    compulsory = N * I * e + N * O * e + 108 * N + 27 * I * O * e + (N * O * e if residual else 0)
    flops = 2.0 * P * I * O
    hbm = float(peaks["hbm_gbs"])
    tc = float(peaks["bf16_tflops"])
    achieved = gathered / fwd_s / 1e9
    t_roof = max(flops / (tc * 1e12), gathered / (hbm * 1e9))
    kernel, src = forward_kernel(I, O) if e == 2 else ("fwd_simt", os.path.join(CSRC, "forward_simt.cu"))
    traffic, traffic_src = recorded_traffic(kernel, src, workload)
    return {
        "bound": "hbm", "kernel": kernel, "achieved": achieved, "peak": hbm, "unit": "GB/s",
        "frac": achieved / hbm, "traffic": traffic, "peak_source": f"hbm_gbs, {peak_kind}",
        "algorithmic_bytes": gathered, "traffic_source": traffic_src,
        "compulsory_bytes": compulsory, "compulsory_frac": compulsory / fwd_s / 1e9 / hbm,
        "tensor_tflops": flops / fwd_s / 1e12, "tensor_frac": flops / fwd_s / 1e12 / tc,
        "roofline_time_us": t_roof * 1e6, "roofline_frac": t_roof / fwd_s,
    }


# ------------------------------------------------------------------------- CPU oracle

def oracle_sample(case, start, count):
    """A bounded sample: the voxels [start, start+count) in raster order (a slab of the
    grid) as a problem of its own, and its pair count from the oracle's kernel map."""
    from oracle import cpu
    N = case["coords"].shape[0]
    a, b = start % N, min(start % N + count, N)
    sub = case["coords"][a:b]
    P = int((cpu.kernel_map(sub, case["res"]) >= 0).sum())
    return sub, case["feats"][a:b], P


def time_oracle(case, sub, feats, P):
    from oracle import cpu
    t0 = time.perf_counter()
    cpu.forward_rows(sub, feats, case["weight"], case["bias"], case["res"])
    dt = time.perf_counter() - t0
    return dt, 2.0 * P * case["I"] * case["O"]


def cpu_baseline(case):
    from oracle import cpu
    sub, feats, P = oracle_sample(case, 0, CPU_SAMPLE_VOXELS)
    dt, flops = time_oracle(case, sub, feats, P)
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": cpu.threads(),
            "kind": "oracle", "seconds": dt,
            "sample": f"C++ oracle (std::unordered_map + fp64 triple loop, OpenMP) on the first "
                      f"{sub.shape[0]} voxels in raster order as a voxel set of their own "
                      f"({P} pairs): map build + every output row"}


# ------------------------------------------------------------------------- arms

def run_reference(args, world, rank):
    if rank != 0:
        return
    from oracle import cpu
    case = load_case(args)
    per_step = max(256, int(REF_STEP_FLOPS / (2.0 * 11 * case["I"] * case["O"])))
    steps = []
    for s in range(args.warmup + args.steps):
        steps.append(oracle_sample(case, s * per_step, per_step))
    times, flops = [], []
    for s, (sub, feats, P) in enumerate(steps):
        dt, fl = time_oracle(case, sub, feats, P)
        if s >= args.warmup:
            times.append(dt)
            flops.append(fl)
    total = sum(times)
    value = sum(flops) / total / 1e12
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": total / len(times) * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "impl": "reference",
        "config": dict(workload_desc(case, None), parallelism="1 process, host cores"),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cpu.threads(),
                         "kind": "oracle",
                         "sample": f"each step: the C++ oracle (map build + all rows, fp64) on "
                                   f"{per_step} consecutive voxels (raster order) as a voxel "
                                   "set of their own"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def kmap_algorithmic_bytes(N, grouped, window):
    """Algorithmic bytes of one kernel-map build: every kernel reads its inputs and writes
    its outputs once (the L2-resident block table is not counted). Insert: coords 16 N in,
    a slot index 4 N out; scatter: coords and slot 20 N in, block-grouped keys and rows
    12 N out; probe: keys and rows 12 N in, the table 108 N out (the radix sort of the
    occupied blocks moves 12 bytes per block per pass, about a twelfth of N blocks, and
    is left out). Window 1 (the Morton order): the probe's rows are the plan's, and the
    probe also writes perm (4 N). Larger windows: the probe writes grouping keys and
    values (12 N); then the grouping sort (24 N per pass) and the plan index (keys,
    values, rows 16 N in; perm 4 N out; the table's 108 N read and written again in plan
    order)."""
    base = 16 * N + 4 * N + 20 * N + 12 * N + 12 * N + 108 * N
    if not grouped:
        return base
    if window == 1:
        return base + 4 * N
    last_window = (N - 1) // window
    passes2 = (27 + last_window.bit_length() + 7) // 8
    return base + 12 * N + 24 * N * passes2 + 16 * N + 4 * N + 2 * 108 * N


def warm_steps(step, seconds=0.3, at_least=3):
    """Untimed steps for at least `seconds` of wall time (and `at_least` steps), with a
    device sync every eight so that the host does not run far ahead of the GPU."""
    import torch
    t_end = time.perf_counter() + seconds
    n = 0
    while n < at_least or time.perf_counter() < t_end:
        step()
        n += 1
        if n % 8 == 0:
            torch.cuda.synchronize()
    torch.cuda.synchronize()


def spread(xs):
    s = sorted(xs)
    return {"min": s[0], "median": statistics.median(s), "max": s[-1], "mean": statistics.mean(s),
            "max_at_step": max(range(len(xs)), key=xs.__getitem__)}


def run_ours(args, world, rank, local):
    import numpy as np
    import torch
    from submanifold_sparse_convolution_04_b300 import (GROUP_WINDOW, subm3d_build_kmap,
                                                        subm3d_build_kmap_async,
                                                        subm3d_build_kmap_grouped,
                                                        subm3d_forward_ex, subm3d_forward_grouped,
                                                        subm3d_forward_status,
                                                        subm3d_kernel_launches,
                                                        subm3d_kmap_grouped_workspace_bytes,
                                                        subm3d_kmap_stage_timing,
                                                        subm3d_kmap_stage_times,
                                                        subm3d_kmap_workspace_bytes,
                                                        subm3d_plan_bytes)
    if not torch.cuda.is_available():
        raise SystemExit("bench.py: no CUDA device (the library has no CPU path)")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    case = load_case(args)
    N, I, O, res = case["coords"].shape[0], case["I"], case["O"], case["res"]
    bf16 = case["dtype"] == "bf16"
    grouped = args.path in ("grouped", "morton")
    window = 1 if args.path == "morton" else (args.window or GROUP_WINDOW)
    if args.graph:
        args.sync_kmap = False

    def host(name):
        if bf16:
            return torch.from_numpy(case[name + "_bits"].view(np.int16)).view(torch.bfloat16)
        return torch.from_numpy(case[name])

    coords_h = torch.from_numpy(case["coords"]).pin_memory()
    feats_h, weight_h, bias_h = (host(k).pin_memory() for k in ("feats", "weight", "bias"))
    c = coords_h.to(dev)
    f = feats_h.to(dev)
    w = weight_h.to(dev)
    b = bias_h.to(dev)
    ws_bytes = subm3d_kmap_grouped_workspace_bytes(N) if grouped else subm3d_kmap_workspace_bytes(N)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    res_h = r = None
    if args.residual:
        from synth import make_residual
        rv, rbits = make_residual(N, O, case["dtype"], case["cfg_id"])
        res_h = (torch.from_numpy(rbits.view(np.int16)).view(torch.bfloat16) if bf16
                 else torch.from_numpy(rv)).pin_memory()
        r = res_h.to(dev)
    fused = args.residual or args.act != "none"

    def new_map():
        """The kernel map's output buffer: a tile plan or nbr [N, 27]."""
        if grouped:
            return torch.empty(max(subm3d_plan_bytes(N), 256), dtype=torch.uint8, device=dev)
        return torch.empty((N, 27), dtype=torch.int32, device=dev)

    def build(coords, kmap):
        if grouped:
            subm3d_build_kmap_grouped(coords, res, window=window, plan=kmap, workspace=ws,
                                      async_=not args.sync_kmap)
        elif args.sync_kmap:
            subm3d_build_kmap(coords, res, nbr=kmap, workspace=ws)
        else:
            subm3d_build_kmap_async(coords, res, nbr=kmap, workspace=ws)

    def forward(feats, kmap, wt, bs, resid, o):
        if grouped:
            subm3d_forward_grouped(feats, kmap, wt, bs, residual=resid, act=args.act, out=o)
        else:
            subm3d_forward_ex(feats, kmap, wt, bs, residual=resid, act=args.act, out=o)

    kmap = new_map()
    out = torch.empty((N, O), dtype=f.dtype, device=dev)

    def step():
        build(c, kmap)
        forward(f, kmap, w, b, r, out)

    for _ in range(max(args.warmup - 3, 1)):   # + 3 more just before the timed region
        step()
    subm3d_forward_status()
    run_build = lambda: build(c, kmap)
    run_forward = lambda: forward(f, kmap, w, b, r, out)
    graph_launches = None
    if args.graph:
        # the same two library calls, captured once into CUDA graphs and replayed per step
        n0 = subm3d_kernel_launches()
        g_build, g_fwd = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_build):
            build(c, kmap)
        with torch.cuda.graph(g_fwd):
            forward(f, kmap, w, b, r, out)
        graph_launches = subm3d_kernel_launches() - n0
        run_build, run_forward = g_build.replay, g_fwd.replay
        for _ in range(3):
            run_build()
            run_forward()
        torch.cuda.synchronize()
        subm3d_forward_status()
    nbr_check = subm3d_build_kmap(c, res)           # pair count from the plain map
    P = int((nbr_check >= 0).sum().item())
    del nbr_check
    flops = 2.0 * P * I * O

    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    cvd = [x.strip() for x in os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",") if x.strip()]
    clocks = ClockSampler(int(cvd[local]) if len(cvd) > local and cvd[local].isdigit() else local)
    clocks.start()
    # the sampler needs ~0.3 s to start: the GPU runs warm-up steps meanwhile (an idle GPU
    # drops to a low-power state, and light steps take tens of ms to bring it back)
    warm_steps(lambda: (run_build(), run_forward()))
    barrier(world)
    torch.cuda.synchronize()
    gc.disable()         # no collector pause of the launching thread inside the region
    launches0 = subm3d_kernel_launches()
    e0.record(stream)
    for s in range(K):
        ev[s][0].record(stream)
        run_build()
        ev[s][1].record(stream)
        run_forward()
        ev[s][2].record(stream)
    e1.record(stream)
    torch.cuda.synchronize()
    gc.enable()
    launches = subm3d_kernel_launches() - launches0
    if graph_launches is not None:      # replays launch the captured kernels, not the host
        launches = graph_launches * K
    clk = clocks.stop()
    barrier(world)
    subm3d_forward_status()          # every step's kernel map and forward: no device error
    total_ms = max_over_ranks(e0.elapsed_time(e1), world)
    kmap_each = [ev[s][0].elapsed_time(ev[s][1]) for s in range(K)]
    fwd_each = [ev[s][1].elapsed_time(ev[s][2]) for s in range(K)]
    kmap_ms = statistics.mean(kmap_each)
    fwd_ms = statistics.mean(fwd_each)
    ms_per_step = total_ms / K
    value = world * flops / (ms_per_step / 1e3) / 1e12

    # per-stage GPU times of one more kernel-map build (outside the timed region)
    subm3d_kmap_stage_timing(True)
    for _ in range(3):
        build(c, kmap)
        stages = subm3d_kmap_stage_times()
    subm3d_kmap_stage_timing(False)
    torch.cuda.synchronize()
    subm3d_forward_status()

    unfused_us = None
    if fused:
        # the same epilogue as separate passes (plain forward, then torch's add and
        # activation over [N, O]): what the fusion saves
        def unfused():
            forward_plain_conv()
            if r is not None:
                out.add_(r)
            if args.act == "relu":
                out.relu_()
            elif args.act == "silu":
                torch.nn.functional.silu(out, inplace=True)

        def forward_plain_conv():
            if grouped:
                subm3d_forward_grouped(f, kmap, w, b, out=out)
            else:
                subm3d_forward_ex(f, kmap, w, b, out=out)
        for _ in range(3):
            unfused()
        u0, u1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        u0.record(stream)
        for _ in range(min(K, 50)):
            unfused()
        u1.record(stream)
        torch.cuda.synchronize()
        unfused_us = u0.elapsed_time(u1) / min(K, 50) * 1e3
        forward(f, kmap, w, b, r, out)      # leave the fused result in out
        torch.cuda.synchronize()

    # end to end through the Python API: every step copies its inputs from pinned host
    # memory to the device, builds the map, runs the forward and copies the output back
    # to pinned host memory. Steps are pipelined over three streams with two buffer sets:
    # step i+1's inputs travel host -> device while step i computes and its output
    # travels device -> host (the copy engines run both directions at once).
    ins = [("c", coords_h), ("f", feats_h), ("w", weight_h), ("b", bias_h)]
    if res_h is not None:
        ins.append(("r", res_h))
    h2d = sum(t.numel() * t.element_size() for _, t in ins)
    d2h = N * O * f.element_size()
    s_cmp = torch.cuda.current_stream()
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    bufs = [dict({"r": None}, **{key: torch.empty_like(src, device=dev) for key, src in ins},
                 kmap=new_map(),
                 out=torch.empty((N, O), dtype=f.dtype, device=dev),
                 out_h=torch.empty((N, O), dtype=f.dtype).pin_memory(),
                 ev_in=torch.cuda.Event(), ev_cmp=torch.cuda.Event(), ev_out=torch.cuda.Event())
            for _ in range(2)]

    def copy_in(i):
        B = bufs[i % 2]
        with torch.cuda.stream(s_in):
            if i >= 2:
                s_in.wait_event(B["ev_cmp"])        # step i-2 has finished with these inputs
            for key, src in ins:
                B[key].copy_(src, non_blocking=True)
            B["ev_in"].record(s_in)

    def compute_and_copy_out(i):
        B = bufs[i % 2]
        s_cmp.wait_event(B["ev_in"])
        if i >= 2:
            s_cmp.wait_event(B["ev_out"])           # step i-2's output has left the device
        build(B["c"], B["kmap"])
        forward(B["f"], B["kmap"], B["w"], B["b"], B["r"], B["out"])
        B["ev_cmp"].record(s_cmp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(B["ev_cmp"])
            B["out_h"].copy_(B["out"], non_blocking=True)
            B["ev_out"].record(s_out)

    def e2e_run(k):
        copy_in(0)
        for i in range(k):
            if i + 1 < k:
                copy_in(i + 1)
            compute_and_copy_out(i)
        torch.cuda.synchronize()

    e2e_run(2)
    barrier(world)
    t0 = time.perf_counter()
    e2e_run(args.e2e_steps)
    e2e_s = max_over_ranks((time.perf_counter() - t0) / args.e2e_steps, world)
    subm3d_forward_status()
    ok_e2e = bool(torch.equal(bufs[(args.e2e_steps - 1) % 2]["out_h"], out.cpu()))

    if rank != 0:
        return
    peaks, peak_kind = load_peaks()
    epi = "none" if not fused else ("residual+" if args.residual else "") + args.act
    roof = roofline(N, P, I, O, fwd_ms / 1e3, peaks, peak_kind,
                    case["name"] + ("_" + args.path if grouped else "") +
                    ("" if not fused else "_" + epi.replace("+", "_")),
                    e=2 if bf16 else 4, residual=args.residual)
    kbytes = kmap_algorithmic_bytes(N, grouped, window)
    hbm = float(peaks["hbm_gbs"])
    kmap_roof = {"bound": "hbm", "achieved": kbytes / (kmap_ms / 1e3) / 1e9, "peak": hbm,
                 "unit": "GB/s", "frac": kbytes / (kmap_ms / 1e3) / 1e9 / hbm,
                 "algorithmic_bytes": kbytes,
                 "front_end": "hashed blocks, radix sort of the block keys",
                 "peak_source": f"hbm_gbs, {peak_kind}",
                 "stages_ms": [[n, round(t, 4)] for n, t in stages]}
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if bf16 else "f32",
        "data": "synthetic",
        "config": dict(workload_desc(case, P),
                       l2="inputs larger than L2 (feats, nbr, hash table each > 126 MB); "
                          "no flush between steps",
                       parallelism=f"replicas x{world}" if world > 1 else "1 GPU",
                       epilogue=epi,
                       path=("tile plan (subm3d_build_kmap_grouped + subm3d_forward_grouped, "
                             f"window {window})" if grouped else
                             "input-order nbr (subm3d_build_kmap + subm3d_forward)"),
                       kmap_wait="synchronous" if args.sync_kmap else
                                 "asynchronous (device status checked after the timed steps)",
                       launch="CUDA graph replay" if args.graph else "library calls"),
        "mvoxels_per_s": world * N / (ms_per_step / 1e3) / 1e6,
        "kmap_ms": kmap_ms, "forward_us": fwd_ms * 1e3,
        "kmap_ms_spread": spread(kmap_each),
        "forward_us_spread": {k: (v if k == "max_at_step" else v * 1e3)
                              for k, v in spread(fwd_each).items()},
        "forward_tflops": flops / (fwd_ms / 1e3) / 1e12,
        "roofline": roof,
        "kmap_roofline": kmap_roof,
        **({"unfused_epilogue_forward_us": unfused_us} if fused else {}),
        "e2e": {"value": world * flops / e2e_s / 1e12, "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": e2e_s * 1e3, "steps": args.e2e_steps,
                "pipelining": "2 buffer sets, copy-in / compute / copy-out streams",
                "output_matches_device_run": ok_e2e},
        "gpu_launches": launches,
        "clocks": clk,
    }
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(case)
    print(json.dumps(line), flush=True)


def run_resample(args, world, rank, local):
    """SparseDownsample(2) (`--op downsample`: the Morton sort, the parent scan and the
    pooling, with its one host sync), the cache-paired SparseUpsample(2) (`--op
    upsample`: one gather kernel), SparseSpatial2Channel(2) (`--op spatial2channel`: zero
    fill of absent blocks + scatter) or its inverse (`--op channel2spatial`: one gather)
    on the workload's voxels and features. Metric: fine voxels per second. Roofline
    bytes: downsample 16 N (coords) + N C e (feats) + 4 N (parent) + M (16 + 1 + C e)
    (coarse coords, masks, pooled rows); upsample 4 N + M C e + N C e; spatial2channel
    N C e + 20 N + M + 8 M C e; channel2spatial 2 N C e + 20 N."""
    import numpy as np
    import torch
    from submanifold_sparse_convolution_04_b300 import (lib, subm3d_build_kmap_ex,
                                                        subm3d_channel2spatial,
                                                        subm3d_downsample,
                                                        subm3d_forward_status,
                                                        subm3d_kernel_launches,
                                                        subm3d_spatial2channel, subm3d_upsample)
    if not torch.cuda.is_available():
        raise SystemExit("bench.py: no CUDA device (the library has no CPU path)")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    case = load_case(args)
    N, C, res = case["coords"].shape[0], case["I"], case["res"]
    bf16 = case["dtype"] == "bf16"
    e = 2 if bf16 else 4
    c = torch.from_numpy(case["coords"]).to(dev)
    f = (torch.from_numpy(case["feats_bits"].view(np.int16)).view(torch.bfloat16) if bf16
         else torch.from_numpy(case["feats"])).to(dev)
    ws = torch.empty(max(256, lib().subm3d_downsample_workspace_bytes(N)), dtype=torch.uint8,
                     device=dev)
    cc, cf, parent, mask = subm3d_downsample(c, res, f, args.pool, workspace=ws)
    M = cc.shape[0]
    up = torch.empty((N, C), dtype=f.dtype, device=dev)
    if args.op == "downsample":
        # the kernel map at this resolution (built anyway by the convolutions that run on
        # these voxels) already holds their Morton order
        order = None if args.ds_sort else subm3d_build_kmap_ex(c, res, order=True)[1]

        if args.ds_wait:    # the call that returns M to the host (one wait per call)
            def step():
                subm3d_downsample(c, res, f, args.pool, workspace=ws, order=order)
        else:               # M stays on the device: no wait inside the timed steps
            outs = subm3d_downsample(c, res, f, args.pool, workspace=ws, order=order,
                                     async_=True)

            def step():
                subm3d_downsample(c, res, f, args.pool, workspace=ws, order=order,
                                  async_=True, out=outs)
        nbytes = 16 * N + N * C * e + 4 * N + M * (16 + 1 + C * e)
        kernel = ("downsample: sort + ds_count/ds_scan/ds_emit + ds_pool" if args.ds_sort else
                  "downsample on the kernel map's Morton order: ds_keys_in_order + "
                  "ds_count/ds_scan/ds_emit + ds_pool") + (
                  ", M read by the host every call" if args.ds_wait else
                  ", M on the device (subm3d_downsample_async)")
    elif args.op == "upsample":
        def step():
            subm3d_upsample(cf, parent, out=up)
        nbytes = 4 * N + M * C * e + N * C * e
        kernel = "us_gather"
    else:
        s2c = torch.empty((M, 8 * C), dtype=f.dtype, device=dev)
        subm3d_spatial2channel(f, c, parent, mask, out=s2c)
        if args.op == "spatial2channel":
            def step():
                subm3d_spatial2channel(f, c, parent, mask, out=s2c)
            nbytes = N * C * e + 20 * N + M + 8 * M * C * e
            kernel = "s2c_zero + s2c_scatter"
        else:
            def step():
                subm3d_channel2spatial(s2c, c, parent, out=up)
            nbytes = 2 * N * C * e + 20 * N
            kernel = "c2s_gather"
    stream = torch.cuda.current_stream()
    for _ in range(max(args.warmup - 3, 1)):   # + 3 more just before the timed region
        step()
    subm3d_forward_status()
    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
    cvd = [x.strip() for x in os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",") if x.strip()]
    clocks = ClockSampler(int(cvd[local]) if len(cvd) > local and cvd[local].isdigit() else local)
    clocks.start()
    warm_steps(step)   # (as in the main bench: the GPU busy while the sampler starts)
    barrier(world)
    torch.cuda.synchronize()
    gc.disable()         # no collector pause of the launching thread inside the region
    launches0 = subm3d_kernel_launches()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for k in range(K):
        ev[k][0].record(stream)
        step()
        ev[k][1].record(stream)
    e1.record(stream)
    torch.cuda.synchronize()
    gc.enable()
    launches = subm3d_kernel_launches() - launches0
    clk = clocks.stop()
    barrier(world)
    subm3d_forward_status()
    total_ms = max_over_ranks(e0.elapsed_time(e1), world)
    op_ms = statistics.mean(ev[k][0].elapsed_time(ev[k][1]) for k in range(K))
    ms_per_step = total_ms / K
    if rank != 0:
        return
    peaks, peak_kind = load_peaks()
    hbm = float(peaks["hbm_gbs"])
    achieved = nbytes / (op_ms / 1e3) / 1e9
    line = {
        "metric": f"Sparse{args.op.capitalize()}(2) Mvoxels/s (fine voxels; fraction of roofline)",
        "value": world * N / (ms_per_step / 1e3) / 1e6, "unit": "Mvoxels/s", "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if bf16 else "f32",
        "data": "synthetic",
        "config": dict(workload_desc(case, None), op=args.op, pool=args.pool, coarse_M=int(M),
                       l2="inputs larger than L2; no flush between steps",
                       parallelism=f"replicas x{world}" if world > 1 else "1 GPU"),
        "op_us": op_ms * 1e3,
        "roofline": {"bound": "hbm", "kernel": kernel, "achieved": achieved, "peak": hbm,
                     "unit": "GB/s", "frac": achieved / hbm, "traffic": None,
                     "traffic_source": "no ncu summary", "peak_source": f"hbm_gbs, {peak_kind}",
                     "algorithmic_bytes": nbytes},
        "gpu_launches": launches,
        "clocks": clk,
    }
    if world == 1 and not args.no_cpu_baseline:
        from oracle import ref
        S = min(N, 1_000_000)
        sub, fs = case["coords"][:S], case["feats"][:S]
        t0 = time.perf_counter()
        _, cfs, par, _ = ref.downsample(sub, fs, res, args.pool)
        t1 = time.perf_counter()
        if args.op == "upsample":
            ref.upsample(cfs, par)
        elif args.op in ("spatial2channel", "channel2spatial"):
            _, s2cs, par, _ = ref.spatial2channel(sub, fs, res)
            t2 = time.perf_counter()
            if args.op == "channel2spatial":
                ref.channel2spatial(s2cs, sub, par)
                t1 = t2
        dt = (t1 - t0) if args.op == "downsample" else (time.perf_counter() - t1)
        line["cpu_baseline"] = {"value": S / dt / 1e6, "unit": "Mvoxels/s", "cores": 1,
                                "kind": "oracle", "seconds": dt,
                                "sample": f"Python oracle ({args.op}) on the first {S} voxels in "
                                          f"raster order, single thread"
                                          + ("; includes the oracle's own subdivision"
                                             if args.op == "spatial2channel" else "")}
    print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    world, rank, local = dist_setup(args.gpus)
    if args.impl == "reference":
        run_reference(args, world, rank)
    elif args.op != "conv":
        run_resample(args, world, rank, local)
    else:
        run_ours(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
