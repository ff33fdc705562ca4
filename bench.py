"""Benchmark: one Barnes-Hut force evaluation per step on synthetic Plummer spheres.

A step is one whole evaluation through the C ABI (bounding cube, Morton keys,
radix sort, gather, octree build, moments, coherent walk, scatter) with the
inputs already resident in device memory. Prints one JSON line.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--theta T]
                    [--traversal coherent64|coherent|independent|...] [--term fast|newton]
                    [--impl ours|reference] [--scaling | --crossover | --accuracy]

--scaling runs the evaluation from 1 024 to 16 777 216 particles (one JSON
line per size); --crossover times the tree against direct summation from
1 024 to 262 144 particles; --accuracy prints the accuracy table (worst and
RMS relative error against an fp64 direct sum) at the pages' sizes and on
4096-target samples of the full-size workloads.

--impl reference times the CPU oracle (the plain C restatement of the
method) on this host's cores instead, on a bounded sample of the same
workload. Under torchrun (N > 1) every rank evaluates its own full problem on
its own GPU (independent replicas, weak scaling); there is no collective on
the data path.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "BH force-evaluation ms and interactions/s at N=1M on 1 GB300; % of FP32/HBM roofline"
UNIT = "interactions/s"
FLOPS_PER_INTERACTION = 18  # 3 FADD, 3 FFMA (x2), 1 FADD, 2+1 FMUL, 3 FFMA (x2) per term
FLOPS_PER_VISIT = 9         # acceptance test: 3 FADD, 1 FMUL + 2 FFMA (x2), 1 FMUL
FP32_LANES_PER_SM = 128
L2_FLUSH_BYTES = 256 << 20  # twice the 129 MB L2


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=11)
    p.add_argument("--warmup", type=int, default=3)
    p.add_argument("--workload", default="plummer_1048576")
    p.add_argument("--theta", type=float, default=None,
                   help="opening angle instead of the workload's (the two-sphere set is swept "
                        "over 0.3, 0.5 and 0.7)")
    p.add_argument("--traversal", default="coherent64",
                   choices=["coherent", "coherent16", "coherent64", "ballot", "together",
                            "independent"])
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--cpu-seconds", type=float, default=8.0,
                   help="target wall time of the CPU-oracle sample")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--term", default="fast", choices=["fast", "newton"],
                   help="fast: the hardware approximate inverse square root (ORRERY_FAST_TERM); "
                        "newton: a fixed seed and three Newton steps, reproducible bit for bit "
                        "on an IEEE CPU. Both are within 1e-5 of the oracle's plain law with "
                        "identical counts; the other one is timed too and reported beside the "
                        "headline")
    p.add_argument("--scaling", action="store_true",
                   help="instead of the benchmark line, the pages' scaling study: one JSON "
                        "line per N from 1024 to 16M particles")
    p.add_argument("--crossover", action="store_true",
                   help="instead of the benchmark line, time the tree against direct "
                        "summation over a range of N (one JSON line per N)")
    p.add_argument("--accuracy", action="store_true",
                   help="instead of the benchmark line, the accuracy table: every target at "
                        "4096, 16384 and 65536 particles, 4096 sampled targets at 1M and on the "
                        "two-sphere set at theta 0.3, 0.5 and 0.7 (one JSON line per row)")
    return p.parse_args()


def replica_throughput(local_ms: float, local_units: float, steps: int, dist=None, device=None):
    """Whole-job throughput of independent replicas: the slowest rank's time
    (max over ranks) over the units every rank processed. Returns
    (ms per step, units per second)."""
    total_ms, units = float(local_ms), float(local_units)
    if dist is not None and dist.is_initialized():
        import torch

        t = torch.tensor([total_ms, units], dtype=torch.float64, device=device)
        mx = t.clone()
        dist.all_reduce(mx, op=dist.ReduceOp.MAX)
        dist.all_reduce(t, op=dist.ReduceOp.SUM)
        total_ms, units = float(mx[0].item()), float(t[1].item())
    ms_per_step = total_ms / steps
    return ms_per_step, units / (ms_per_step / 1000.0)


def run_scaling(args) -> None:
    """The pages' "Scaling, and where it stops" table on this GPU: whole
    evaluation and walk per N, ms / (N log2 N), the local exponent, and the
    interaction and visit counts per particle (median of --steps calls)."""
    import math

    import torch

    import tree_traversal_gb300 as tt
    from inputs import plummer
    from tree_traversal_gb300.build import build

    build()
    tt.load()
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream(dev)
    prev = None
    sizes = [1024 << k for k in range(12)] + [4194304, 8388608, 16777216]
    for n in sizes:
        pos_np, mass_np = plummer(n)
        pos = torch.from_numpy(pos_np).to(dev)
        mass = torch.from_numpy(mass_np).to(dev)
        acc = torch.empty((n, 3), device=dev)
        inter = torch.empty((n, 2), dtype=torch.int32, device=dev)
        vis = torch.empty(n, dtype=torch.int32, device=dev)
        total, walk = [], []
        for it in range(args.warmup + args.steps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            tt.bh_forces(pos, mass, 0.5, 0.05, 32, args.traversal, out=(acc, inter, vis),
                         fast_term=args.term == "fast")
            b.record(stream)
            torch.cuda.synchronize(dev)
            if it >= args.warmup:
                total.append(a.elapsed_time(b))
                walk.append(tt.last_timings()["walk_ms"])
        t = statistics.median(total)
        tm = tt.last_timings()
        row = {"n": n, "total_ms": t, "walk_ms": statistics.median(walk),
               "spread": (max(total) - min(total)) / t,
               "ms_per_nlogn": t / (n * math.log2(n)),
               "exponent": (math.log(t / prev[1]) / math.log(n / prev[0])) if prev else None,
               "cells_per_particle": float(inter[:, 0].double().mean()),
               "interactions_per_particle": float(inter.double().sum(1).mean()),
               "visits_per_particle": float(vis.double().mean()),
               "nodes": tm["num_nodes"], "depth": tm["depth"], "traversal": args.traversal,
               "term": args.term}
        prev = (n, t)
        print(json.dumps(row), flush=True)
        del pos, mass, acc, inter, vis
        torch.cuda.empty_cache()


def run_crossover(args) -> None:
    """Tree (whole evaluation) against direct summation, Plummer spheres of
    1024 .. 262144 particles: the pages' "Against the two solvers it has to
    beat" table, on this GPU. Median of --steps timed calls after --warmup."""
    import torch

    import tree_traversal_gb300 as tt
    from inputs import plummer
    from tree_traversal_gb300.build import build

    build()
    tt.load()
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream(dev)

    def timed(fn):
        ms = []
        for it in range(args.warmup + args.steps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            torch.cuda.synchronize(dev)
            if it >= args.warmup:
                ms.append(a.elapsed_time(b))
        return statistics.median(ms)

    for n in (1024, 2048, 4096, 8192, 16384, 32768, 65536, 131072, 262144):
        pos_np, mass_np = plummer(n)
        pos = torch.from_numpy(pos_np).to(dev)
        mass = torch.from_numpy(mass_np).to(dev)
        # the Newton term on both sides: the direct kernel sums the same
        # particle term, so the comparison is of the algorithms alone
        t_tree = timed(lambda: tt.bh_forces(pos, mass, 0.5, 0.05, 32, args.traversal))
        walk = tt.last_timings()["walk_ms"]
        t_direct = timed(lambda: tt.direct_forces(pos, mass, 0.05))
        print(json.dumps({"n": n, "tree_ms": t_tree, "tree_walk_ms": walk, "direct_ms": t_direct,
                          "tree_speedup_vs_direct": t_direct / t_tree,
                          "direct_pairs_per_s": n * (n - 1) / (t_direct / 1000.0),
                          "traversal": args.traversal, "term": "newton (both solvers)"}), flush=True)


def measured_peaks() -> dict:
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f)
    except OSError:
        return {}


# the walk kernel each traversal launches, and the ncu summary holding its
# full-size DRAM traffic
WALK_KERNELS = {"coherent": "k_walk_coherent", "coherent16": "k_walk_coherent",
                "ballot": "k_walk_coherent", "coherent64": "k_walk_paired",
                "together": "k_walk_together", "independent": "k_walk_independent"}
TRAFFIC_PROFILES = {("k_walk_paired", True): "walk_paired_fast_plummer_1m.md",
                    ("k_walk_coherent", True): "walk_coherent_plummer_1m.md",
                    ("k_walk_independent", True): "walk_independent_plummer_1m.md"}


def code_sha256(path: str) -> str:
    """SHA-256 of a CUDA source with its // comments, trailing blanks and
    empty lines removed: changes to comments leave it (and the compiled
    kernel) unchanged, any change to the code changes it."""
    import re

    lines = []
    for line in open(path, encoding="utf-8"):
        line = re.sub(r"//.*$", "", line.rstrip("\n")).rstrip()
        if line.strip():
            lines.append(line)
    return hashlib.sha256("\n".join(lines).encode()).hexdigest()


def profile_traffic(kernel_src: str, kernel: str, fast: bool) -> float | None:
    """Per-launch DRAM bytes of the walk kernel from the committed ncu summary,
    only while the kernel's code is the code that was profiled."""
    name = TRAFFIC_PROFILES.get((kernel, fast))
    path = os.path.join(ROOT, "profiles", name) if name else ""
    if not name or not os.path.exists(path):
        return None
    sha = code_sha256(kernel_src)
    found_sha, traffic = None, None
    for line in open(path):
        if line.startswith("kernel_code_sha256:"):
            found_sha = line.split(":", 1)[1].strip()
        if line.startswith("dram_bytes_per_launch_full_size:"):
            traffic = float(line.split(":", 1)[1].strip())
    return traffic if found_sha == sha else None


class ClockSampler:
    """Samples SM clocks and throttle reasons with nvidia-smi during a region."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.QUERY,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]
        return False

    def summary(self) -> dict:
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in getattr(self, "lines", []):
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax = float(f[2])
            except ValueError:
                continue
            for name, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


def direct_f64_device(pos, mass, eps, targets, device, chunk_bytes=1 << 30):
    """fp64 direct sum of the softened law over every j != i for the given
    caller indices, evaluated with torch in double precision on the device
    (the reference the accuracy figures are measured against; torch's
    reductions sum in a tree, so the rounding of 2M terms stays near 1e-15
    relative to their magnitude). Returns [t, 3] float64 on the host."""
    import torch

    x = torch.from_numpy(np.ascontiguousarray(pos, np.float64)).to(device)
    m = torch.from_numpy(np.ascontiguousarray(mass, np.float64)).to(device)
    tg = torch.from_numpy(np.asarray(targets, np.int64)).to(device)
    n = x.shape[0]
    per = max(1, int(chunk_bytes // (8 * 8 * max(n, 1))))
    out = []
    for b in range(0, tg.shape[0], per):
        t = tg[b:b + per]
        d = x[None, :, :] - x[t][:, None, :]
        r2 = (d * d).sum(-1) + float(eps) * float(eps)
        w = m[None, :] / (r2 * torch.sqrt(r2))
        w[torch.arange(t.shape[0], device=device), t] = 0.0
        out.append((w[:, :, None] * d).sum(1))
    return torch.cat(out).cpu().numpy()


def accuracy_vs_direct(pos, mass, acc, eps, device, count=4096, seed=20260811) -> dict:
    """Worst and RMS relative error of the accelerations (caller order)
    against the fp64 direct sum, on every target when there are at most
    `count`, else on a seeded sample of `count` (after the timed region; the
    pages' accuracy table measures the same two numbers)."""
    n = pos.shape[0]
    if n <= count:
        tgt = np.arange(n)
    else:
        tgt = np.sort(np.random.default_rng(seed).choice(n, count, replace=False))
    ref = direct_f64_device(pos, mass, eps, tgt, device)
    got = np.asarray(acc, np.float64)[tgt]
    errs = np.linalg.norm(got - ref, axis=1) / np.linalg.norm(ref, axis=1)
    return {"vs": "fp64 direct sum", "targets": int(len(tgt)), "worst": float(errs.max()),
            "rms": float(np.sqrt(np.mean(errs * errs)))}


# the pages' accuracy table (docs/performance/sycl_tree.md, "Accuracy"):
# theta 0.5 against a compensated fp64 direct sum, their Plummer generator
PAGES_ACCURACY = {4096: (2.03e-2, 2.03e-3), 16384: (1.34e-2, 1.76e-3), 65536: (7.12e-3, 1.48e-3)}


def run_accuracy(args) -> None:
    """One JSON line per row: the tree's accelerations (width-64 walk, both
    force terms, and the pages' width-32 walk) against the fp64 direct sum,
    every target at the pages' sizes and 4096 sampled targets at full size;
    and the direct kernel at 65536 (the pages quote its RMS error too)."""
    import torch

    import tree_traversal_gb300 as tt
    from inputs import plummer, two_spheres
    from tree_traversal_gb300.build import build

    build()
    tt.load()
    dev = torch.device("cuda", 0)
    rows = [("plummer_%d" % n, plummer(n), 0.5, n) for n in (4096, 16384, 65536)]
    rows.append(("plummer_1048576", plummer(1048576), 0.5, None))
    two = two_spheres(1048576)
    rows += [("two_spheres_2x1048576", two, th, None) for th in (0.3, 0.5, 0.7)]
    for name, (pos_np, mass_np), theta, n_pages in rows:
        pos = torch.from_numpy(pos_np).to(dev)
        mass = torch.from_numpy(mass_np).to(dev)
        for trav, fast in (("coherent64", True), ("coherent64", False), ("coherent", True)):
            acc, inter, _ = tt.bh_forces(pos, mass, theta, 0.05, 32, trav, fast_term=fast)
            # every target at the pages' sizes, 4096 sampled ones at full size
            a = accuracy_vs_direct(pos_np, mass_np, acc.cpu().numpy(), 0.05, dev,
                                   count=n_pages or 4096)
            line = {"workload": name, "n": int(pos_np.shape[0]), "theta": theta, "eps": 0.05,
                    "leaf_cap": 32, "traversal": trav, "term": "fast" if fast else "newton",
                    **a, "interactions_per_particle": float(inter.double().sum().item()) / pos_np.shape[0]}
            if n_pages in PAGES_ACCURACY:
                line["pages_worst"], line["pages_rms"] = PAGES_ACCURACY[n_pages]
            print(json.dumps(line), flush=True)
    pos_np, mass_np = plummer(65536)
    acc = tt.direct_forces(torch.from_numpy(pos_np).to(dev), torch.from_numpy(mass_np).to(dev), 0.05)
    a = accuracy_vs_direct(pos_np, mass_np, acc.cpu().numpy(), 0.05, dev, count=65536)
    print(json.dumps({"workload": "plummer_65536", "n": 65536, "solver": "direct (GPU kernel)",
                      "eps": 0.05, **a, "pages_rms": 3.7e-6}), flush=True)


def cpu_baseline(pos, mass, params, seconds: float) -> dict:
    """The oracle as it stands on this host's cores: full tree build plus the
    walk of a sample of whole 32-target groups; scaled to interactions/s of a
    whole evaluation (build + all targets)."""
    import oracle

    threads = oracle.default_threads()
    n = pos.shape[0]
    t0 = time.perf_counter()
    T = oracle.Tree(pos, mass, params["leaf_cap"])
    t_build = time.perf_counter() - t0
    nw = (n + 31) // 32

    def walk_every(stride):
        warps = np.arange(0, nw, stride)
        tgt = np.concatenate([np.arange(32 * w, min(n, 32 * w + 32)) for w in warps])
        t0 = time.perf_counter()
        _, pc, pp, _ = T.walk(params["theta"], params["eps"], tgt, threads=threads)
        return tgt, pc, pp, time.perf_counter() - t0

    # calibrate on every 512th group, then size the sample to the time budget
    tgt, pc, pp, t_walk = walk_every(min(512, nw))
    per_target = t_walk / len(tgt)
    stride = int(max(1, min(nw, round(n * per_target / max(seconds, 1e-3)))))
    if stride < min(512, nw):
        tgt, pc, pp, t_walk = walk_every(stride)
    inter_sample = float(pc.sum() + pp.sum())
    t_full = t_build + t_walk * n / len(tgt)
    inter_full = inter_sample * n / len(tgt)
    # one thread, on every 64th target of that sample (the pages' protocol
    # times the CPU both ways)
    t0 = time.perf_counter()
    sub = tgt[:: 64] if len(tgt) >= 64 else tgt
    _, pc1, pp1, _ = T.walk(params["theta"], params["eps"], sub, threads=1)
    t_walk1 = time.perf_counter() - t0
    walk1_per_s = float(pc1.sum() + pp1.sum()) / t_walk1
    import platform
    return {"value": inter_full / t_full, "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": "full tree build (%.2f s, 1 thread) + walks of %d of %d targets in whole "
                      "32-target groups (%.2f s, %d threads), scaled to all targets"
                      % (t_build, len(tgt), n, t_walk, threads),
            "ms_per_evaluation_est": 1000.0 * t_full, "cpu": platform.machine(),
            "walk_interactions_per_s_1_thread": walk1_per_s,
            "walk_interactions_per_s_all_threads": inter_sample / t_walk}


def run_reference(args, rank: int, world: int) -> None:
    from inputs import workload

    if rank != 0:
        return
    pos, mass, params = workload(args.workload)
    if args.theta is not None:
        params["theta"] = args.theta
    times, vals, walk1, walk_all = [], [], [], []
    cb = None
    for step in range(args.warmup + args.steps):
        cb = cpu_baseline(pos, mass, params, min(args.cpu_seconds, 4.0))
        if step >= args.warmup:
            times.append(cb["ms_per_evaluation_est"])
            vals.append(cb["value"])
            walk1.append(cb["walk_interactions_per_s_1_thread"])
            walk_all.append(cb["walk_interactions_per_s_all_threads"])
    v = statistics.median(vals)
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": statistics.median(times), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": args.workload, "n": int(pos.shape[0]), **params,
                       "traversal": "independent (CPU oracle)"},
            "cpu_baseline": {"value": v, "unit": UNIT, "cores": cb["cores"], "kind": "oracle",
                             "sample": cb["sample"],
                             "walk_interactions_per_s_1_thread": statistics.median(walk1),
                             "walk_interactions_per_s_all_threads": statistics.median(walk_all)},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if args.crossover:
        run_crossover(args)
        return
    if args.scaling:
        run_scaling(args)
        return
    if args.accuracy:
        run_accuracy(args)
        return
    if args.warmup < 3:
        raise SystemExit("--warmup must be at least 3")

    import torch

    import tree_traversal_gb300 as tt
    from inputs import workload
    from tree_traversal_gb300.build import build

    dist = None
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    device = torch.device("cuda", local_rank)
    torch.cuda.set_device(device)
    if rank == 0:
        build()
    if dist is not None:
        dist.barrier()
    tt.load()

    pos_np, mass_np, params = workload(args.workload)
    if args.theta is not None:
        params["theta"] = args.theta
    n = pos_np.shape[0]
    pos = torch.from_numpy(pos_np).to(device)
    mass = torch.from_numpy(mass_np).to(device)
    acc = torch.empty((n, 3), dtype=torch.float32, device=device)
    inter = torch.empty((n, 2), dtype=torch.int32, device=device)
    visits = torch.empty(n, dtype=torch.int32, device=device)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=device)
    stream = torch.cuda.current_stream(device)
    fast = args.term == "fast"
    call = lambda trav, fast_term=fast: tt.bh_forces(
        pos, mass, params["theta"], params["eps"], params["leaf_cap"], trav,
        out=(acc, inter, visits), fast_term=fast_term)

    # untimed: the comparison traversals (the independent walk's visits give
    # the redundancy ratio; width 32 is the pages' coherent group)
    comparison = {}
    for trav in ("independent", "coherent", "coherent64"):
        if trav == args.traversal:
            continue
        for _ in range(2):
            call(trav)
        comparison[trav] = {"walk_ms": tt.last_timings()["walk_ms"],
                            "visits_per_particle": visits.double().mean().item()}
    other = "independent" if args.traversal != "independent" else "coherent"
    vis_other = comparison[other]["visits_per_particle"]
    for _ in range(args.warmup):
        call(args.traversal)
    torch.cuda.synchronize(device)
    interactions = float(inter.double().sum().item())
    vis_mean = visits.double().mean().item()
    pc_mean = inter[:, 0].double().mean().item()
    pp_mean = inter[:, 1].double().mean().item()

    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    phases, step_ms = [], []
    launches0 = tt.kernel_launches()
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize(device)
    with ClockSampler(device.index) as clocks:
        t0 = time.perf_counter()
        for s in range(args.steps):
            flush.zero_()  # evict L2 between steps (outside the step's events)
            ev[s][0].record(stream)
            call(args.traversal)
            ev[s][1].record(stream)
            phases.append(tt.last_timings())
        torch.cuda.synchronize(device)
        if dist is not None:
            dist.barrier()
        wall = time.perf_counter() - t0
    launches = tt.kernel_launches() - launches0
    step_ms = [a.elapsed_time(b) for a, b in ev]
    ms_per_step, value = replica_throughput(sum(step_ms), interactions, args.steps, dist, device)

    # the other term, timed the same way (reported beside the headline)
    for _ in range(3):
        call(args.traversal, not fast)
    other_ms, other_walk = [], []
    for s in range(args.steps):
        flush.zero_()
        ev[s][0].record(stream)
        call(args.traversal, not fast)
        ev[s][1].record(stream)
        other_walk.append(tt.last_timings()["walk_ms"])
    torch.cuda.synchronize(device)
    other_ms = [a.elapsed_time(b) for a, b in ev]

    def mean(key):
        return statistics.fmean(p[key] for p in phases)

    walk_ms = mean("walk_ms")
    # the pages' independent walk gives the algorithmic count; the coherent
    # walk's extra (union) visits are overhead, not work
    vis_ind = vis_mean if args.traversal == "independent" else vis_other
    flops_inter = FLOPS_PER_INTERACTION * interactions
    sms = torch.cuda.get_device_properties(device).multi_processor_count
    peaks = measured_peaks()
    clk = peaks.get("sm_max_mhz", 2070.0)
    peak_tflops = sms * FP32_LANES_PER_SM * 2 * clk * 1e6 / 1e12
    achieved = flops_inter / (walk_ms / 1000.0) / 1e12
    csum = clocks.summary()

    # e2e: the host entry point with page-locked buffers, inside the timed
    # call: the inputs are copied in, and the walk stores the outputs straight
    # into the page-locked output buffers over the host link
    h_pos = torch.from_numpy(pos_np).pin_memory()
    h_mass = torch.from_numpy(mass_np).pin_memory()
    h_out = (torch.empty((n, 3)).pin_memory(), torch.empty((n, 2), dtype=torch.int32).pin_memory(),
             torch.empty(n, dtype=torch.int32).pin_memory())
    for _ in range(2):
        tt.bh_forces_host(h_pos, h_mass, params["theta"], params["eps"], params["leaf_cap"],
                          args.traversal, out=h_out, device=device, fast_term=fast)
    e2e_ms = []
    for _ in range(args.steps):
        flush.zero_()
        torch.cuda.synchronize(device)
        t1 = time.perf_counter()
        tt.bh_forces_host(h_pos, h_mass, params["theta"], params["eps"], params["leaf_cap"],
                          args.traversal, out=h_out, device=device, fast_term=fast)
        e2e_ms.append(1000.0 * (time.perf_counter() - t1))
    e2e_host = tt.last_timings()
    # measured FP32 FMA rate (long independent chains on every SM), beside
    # the nominal peak: untimed, after everything above
    fma = tt.fp32_fma_rate(device)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()
    if rank != 0:
        return
    cb = None
    if not args.no_cpu_baseline and world == 1:
        cb = cpu_baseline(pos_np, mass_np, params, args.cpu_seconds)
    walk_src = os.path.join(ROOT, "tree_traversal_gb300", "csrc", "bh_walk.cu")
    kernel = WALK_KERNELS[args.traversal]
    traffic = profile_traffic(walk_src, kernel, fast)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": args.workload, "n": n, "theta": params["theta"],
                   "eps": params["eps"], "leaf_cap": params["leaf_cap"],
                   "traversal": args.traversal, "parallelism": "replicas" if world > 1 else "1gpu",
                   "term": "fast: hardware approximate inverse root" if fast
                   else "newton: fixed seed and three Newton steps (bit-reproducible on an IEEE CPU)",
                   "l2": "flushed between steps (256 MiB write outside the step events)"},
        "gpu_launches": int(launches),
        "clocks": {"sm_mhz": csum["sm_mhz"], "sm_max_mhz": csum["sm_max_mhz"],
                   "reasons": csum["reasons"]},
        "roofline": {"bound": "alu", "kernel": kernel,
                     "achieved": achieved, "peak": peak_tflops, "unit": "TFLOP/s",
                     "frac": achieved / peak_tflops, "traffic": traffic,
                     "peak_basis": "%d SMs x %d FP32 lanes x 2 flop x %.0f MHz (max SM clock of "
                                   "measured peaks)" % (sms, FP32_LANES_PER_SM, clk),
                     "flops_per_launch": flops_inter,
                     "flops_per_interaction": FLOPS_PER_INTERACTION,
                     "walk_ms": walk_ms,
                     "frac_at_sampled_clock": (achieved / (peak_tflops * csum["sm_mhz"] / clk))
                     if csum["sm_mhz"] else None,
                     "frac_incl_acceptance": (flops_inter + FLOPS_PER_VISIT * vis_ind * n)
                     / (walk_ms / 1000.0) / 1e12 / peak_tflops,
                     "peak_measured_fma": {"scalar": fma["scalar"], "packed": fma["packed"],
                                           "unit": "TFLOP/s", "sm_mhz": fma["sm_mhz"],
                                           "lanes_per_sm_clock": fma["scalar"] * 1e12 / 2
                                           / (sms * fma["sm_mhz"] * 1e6) if fma["sm_mhz"] else None},
                     "frac_of_measured_fma": achieved / max(fma["scalar"], fma["packed"])},
        "cpu_baseline": None if cb is None else
        {k: cb[k] for k in ("value", "unit", "cores", "kind", "sample", "walk_interactions_per_s_1_thread",
                             "walk_interactions_per_s_all_threads")},
        "e2e": {"value": interactions / (statistics.median(e2e_ms) / 1000.0), "unit": UNIT,
                "h2d_bytes_per_step": 16 * n, "d2h_bytes_per_step": 24 * n,
                "ms_median": statistics.median(e2e_ms), "h2d_ms": e2e_host["h2d_ms"],
                "d2h_ms": e2e_host["d2h_ms"],
                "d2h_by": "the walk's stores into page-locked host buffers (no separate copy)"},
        "phases_ms": {k: mean(k) for k in ("bbox_ms", "morton_ms", "sort_ms", "gather_ms",
                                           "build_ms", "moments_ms", "walk_ms", "scatter_ms",
                                           "total_ms")},
        "step_ms": {"median": statistics.median(step_ms), "min": min(step_ms), "max": max(step_ms),
                    "iqr": (statistics.quantiles(step_ms, n=4)[2] - statistics.quantiles(step_ms, n=4)[0])
                    if len(step_ms) >= 2 else 0.0,
                    "wall_s_incl_flush": wall},
        "tree": {"num_nodes": phases[-1]["num_nodes"], "depth": phases[-1]["depth"]},
        "interactions_per_s_walk": interactions / (walk_ms / 1000.0),
        "per_particle": {"interactions": interactions / n, "cells": pc_mean, "particles": pp_mean,
                         "visits": vis_mean, "visits_" + other: vis_other,
                         "redundancy": (vis_mean / vis_other) if args.traversal != "independent"
                         else (vis_other / vis_mean)},
        ("newton_term" if fast else "fast_term"): {
            "ms_per_step": statistics.fmean(other_ms), "walk_ms": statistics.fmean(other_walk),
            "value": interactions / (statistics.fmean(other_ms) / 1000.0)},
        "comparison_traversals": comparison,
        "accuracy": accuracy_vs_direct(pos_np, mass_np, h_out[0].numpy(), params["eps"], device),
        "redundancy_width32": (comparison["coherent"]["visits_per_particle"] / vis_other)
        if "coherent" in comparison and args.traversal != "independent" else None,
    }
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
