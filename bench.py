#!/usr/bin/env python3
"""Benchmark: left-balanced k-d tree build throughput on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload uniform_100m] [--no-e2e] [--no-cpu-baseline]

One step = one complete build (every level of the method) of the workload's
points, resident in HBM, through the C ABI with a caller-provided workspace.
Prints ONE JSON line on rank 0.

Multi-GPU (torchrun, one rank per GPU): the build does not shard, so every
rank builds its own replica of the workload ("replicas only"); value = total
points built by all ranks / max over ranks of the timed region.

--impl reference times the CPU oracle (the plain single-threaded recursive
builder) on the host cores, on a bounded sample of the same workload per step.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "points/sec for balanced k-d tree build (1×GB300) and % of HBM roofline"
UNIT = "points/s"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0


# ---------------------------------------------------------------------------
# distributed plumbing (replicas only)

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world: int, backend: str):
    if world <= 1:
        return False
    import torch.distributed as dist
    os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
    dist.init_process_group(backend=backend)
    return True


def barrier(active: bool):
    if active:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(value: float, active: bool, device=None) -> float:
    """Max of a per-rank float over all ranks (the slowest rank's time)."""
    if not active:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------
# clocks during the timed region

class ClockSampler:
    """nvidia-smi sampling every 20 ms.  It is started before the warm-up
    (nvidia-smi takes a while to print its first sample) and each sample
    carries nvidia-smi's own timestamp, so stop() keeps the samples taken
    inside the timed region (host wall-clock window) and summarises those."""
    FIELDS = ["timestamp", "clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active",
              "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]
    REASONS = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, gpu_id: str | None, interval_ms: int = 20):
        self.gpu_id = gpu_id
        self.interval_ms = interval_ms
        self.proc = None
        self.lines: list[str] = []
        self.thread = None

    def start(self):
        cmd = ["nvidia-smi", "--query-gpu=" + ",".join(self.FIELDS), "--format=csv,noheader,nounits",
               "-lms", str(self.interval_ms)]
        if self.gpu_id:
            cmd += ["-i", self.gpu_id]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    @staticmethod
    def _stamp(text: str) -> float | None:
        import datetime
        for fmt in ("%Y/%m/%d %H:%M:%S.%f", "%Y/%m/%d %H:%M:%S"):
            try:
                return datetime.datetime.strptime(text, fmt).timestamp()
            except ValueError:
                pass
        return None

    @classmethod
    def summarise(cls, lines: list[str], window: tuple[float, float] | None) -> dict | None:
        """Median SM clock, max clock and active throttle reasons of the
        samples inside `window` (host seconds, with one sampling interval of
        slack); if none falls inside, of the two samples nearest to it."""
        recs = []
        for ln in lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < len(cls.FIELDS):
                continue
            try:
                sm, smax = float(parts[1]), float(parts[2])
            except ValueError:
                continue
            reasons = {nm for nm, v in zip(cls.REASONS, parts[5:9]) if v.lower() == "active"}
            recs.append((cls._stamp(parts[0]), sm, smax, reasons))
        if not recs:
            return None
        where = "all samples"
        sel = recs
        if window is not None:
            t0, t1 = window[0] - 0.02, window[1] + 0.02
            stamped = [r for r in recs if r[0] is not None]
            inside = [r for r in stamped if t0 <= r[0] <= t1]
            if inside:
                sel, where = inside, "timed region"
            elif stamped:
                mid = 0.5 * (t0 + t1)
                sel, where = sorted(stamped, key=lambda r: abs(r[0] - mid))[:2], "nearest to the timed region"
        reasons = set()
        for r in sel:
            reasons |= r[3]
        return {"sm_mhz": statistics.median(r[1] for r in sel), "sm_max_mhz": max(r[2] for r in sel),
                "samples": len(sel), "window": where, "reasons": sorted(reasons)}

    def stop(self, window: tuple[float, float] | None = None) -> dict | None:
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        try:
            return self.summarise(list(self.lines), window)
        except Exception:  # a clock record must never cost the bench line
            return None


def gpu_identifier(dev_index: int) -> str | None:
    try:
        import torch
        props = torch.cuda.get_device_properties(dev_index)
        uuid = getattr(props, "uuid", None)
        if uuid is not None:
            s = str(uuid)
            return s if s.startswith("GPU-") else "GPU-" + s
    except Exception:
        pass
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis:
        return vis.split(",")[dev_index]
    return str(dev_index)


def measured_peaks() -> tuple[float, str]:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def recorded_traffic(kernel: str):
    """DRAM bytes per launch of `kernel` from profiles/traffic_uniform_100m.txt,
    or None if not recorded or if the kernel's source changed since."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "traffic_uniform_100m.txt")
    try:
        with open(path) as f:
            lines = [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]
    except OSError:
        return None
    for t in lines:
        if len(t) >= 8 and t[0] == "kernel" and t[1] == kernel:
            src, sha, nbytes = t[3], t[5], float(t[7])
            try:
                with open(os.path.join(ROOT, src), "rb") as f:
                    if hashlib.sha256(f.read()).hexdigest()[:len(sha)] != sha:
                        return None
            except OSError:
                return None
            return nbytes
    return None


def b_alg(n: int) -> float:
    """Algorithmic bytes of the level-by-level method: per point and sort
    level 20 B (read tag, index and split coordinate; write tag and index),
    plus 12 B per point for the final level-order gather."""
    L = n.bit_length()  # numLevels(n) = floor(log2 n) + 1
    return float(n) * (20.0 * (L - 1) + 12.0)


# ---------------------------------------------------------------------------
# CPU baseline: the oracle on a bounded sample

def cpu_baseline(workload, budget_s: float = 12.0) -> dict:
    import oracle
    o = oracle.get()
    sample_n = 1 << 18
    pts = workload.points(sample_n)
    t0 = time.perf_counter()
    o.build_tree(pts, workload.mode)
    dt = time.perf_counter() - t0
    reps = 1
    # grow the sample towards the time budget (roughly 10-30 s of CPU work)
    while dt * 4 < budget_s and sample_n < (1 << 22) and sample_n < workload.n:
        sample_n *= 4
        pts = workload.points(sample_n)
        t0 = time.perf_counter()
        o.build_tree(pts, workload.mode)
        dt = time.perf_counter() - t0
    return {"value": sample_n / dt, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample_points": sample_n, "workload_points": workload.n,
            "sample": f"a SAMPLE of {sample_n} points (not the workload's {workload.n}) drawn from the "
                      f"{workload.name} distribution (k={workload.k}, mode={workload.mode}), one full build, "
                      f"{reps} run, single-threaded C oracle; the oracle sorts each subtree "
                      f"(O(N log^2 N)), so its rate at the full size is lower"}


def run_reference(args, workload):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    o = oracle.get()
    sample_n = args.ref_sample
    pts = workload.points(sample_n)
    for _ in range(args.warmup):
        o.build_tree(pts, workload.mode)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        o.build_tree(pts, workload.mode)
    dt = time.perf_counter() - t0
    value = sample_n * args.steps / dt
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3 / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": workload_config(workload, extra={"reference_sample_points": sample_n}),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": f"{sample_n} points of the {workload.name} distribution per step"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def workload_config(w, extra=None) -> dict:
    cfg = {"workload": w.name, "N": w.n, "k": w.k,
           "split_mode": "round_robin" if w.mode == 0 else "widest",
           "distribution": w.dist, "seed": w.seed, "layout": "AoS float32 in, int32 level-order perm out",
           "l2": "no flush: inputs and workspace exceed the 129 MB L2"}
    if extra:
        cfg.update(extra)
    return cfg


# ---------------------------------------------------------------------------
# our build

def level_order_extra(kdt, pts, perm, ws, workload, stream, peak) -> dict:
    """Times the points-in-level-order gather (kdt_gather_points) on the bench
    workload's tree, and the in-place build (kdt_build_inplace) on a copy of
    the points; checks a sample of the gathered rows bit for bit."""
    import torch
    n, k = pts.shape
    out = torch.empty_like(pts)
    for _ in range(2):
        kdt.gather_points(pts, perm, out=out, stream=stream)
    reps = 5
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(reps):
        kdt.gather_points(pts, perm, out=out, stream=stream)
    e1.record(stream)
    torch.cuda.synchronize()
    gather_ms = e0.elapsed_time(e1) / reps
    if kdt.status(stream) != 0:
        raise SystemExit("device status after the gather")
    idx = torch.randint(0, n, (min(n, 1 << 20),), device=pts.device)
    if not torch.equal(out[idx].view(torch.int32), pts[perm[idx].long()].view(torch.int32)):
        raise SystemExit("gathered rows differ from pts[perm]")
    alg = float(n) * (4 + 8 * k)  # perm read, row read, row write
    scratch = torch.empty_like(pts)
    times = []
    for i in range(3):
        scratch.copy_(pts)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        kdt.build_inplace(scratch, workload.mode, perm=perm, workspace=ws, stream=stream)
        b.record(stream)
        torch.cuda.synchronize()
        if i > 0:
            times.append(a.elapsed_time(b))
    if kdt.status(stream) != 0:
        raise SystemExit("device status after the in-place build")
    res = {"gather_ms": gather_ms, "gather_alg_bytes": alg, "gather_GBps": alg / (gather_ms / 1e3) / 1e9,
           "gather_frac_of_measured": alg / (gather_ms / 1e3) / 1e9 / peak,
           "inplace_build_ms": sum(times) / len(times), "api": "kdt_gather_points, kdt_build_inplace"}
    return res, out


def knn_extra(kdt, tree_pts, workload, stream, n_queries: int = 1 << 20, K: int = 8) -> dict:
    """Times kdt_knn: n_queries points drawn from the workload's distribution
    (another seed) against the tree whose level-order points are tree_pts."""
    import torch
    from balanced_tree_build_gb300.inputs import make_points
    n, k = tree_pts.shape
    q = torch.from_numpy(make_points(workload.dist, n_queries, k, workload.seed + 1000)).to(tree_pts.device)
    dims = kdt.node_dims(tree_pts, workload.mode, stream=stream) if workload.mode == 1 else None
    nodes = torch.empty((n_queries, K), dtype=torch.int32, device=q.device)
    d2 = torch.empty((n_queries, K), dtype=torch.float32, device=q.device)
    kdt.knn(tree_pts, q, K, dims=dims, out_nodes=nodes, out_dist2=d2, stream=stream)
    reps = 3
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(reps):
        kdt.knn(tree_pts, q, K, dims=dims, out_nodes=nodes, out_dist2=d2, stream=stream)
    e1.record(stream)
    torch.cuda.synchronize()
    if kdt.status(stream) != 0:
        raise SystemExit("device status after kNN queries")
    ms = e0.elapsed_time(e1) / reps
    return {"queries": n_queries, "K": K, "ms": ms, "queries_per_s": n_queries / (ms / 1e3),
            "tree_points": n, "api": "kdt_knn (one thread per query, stack-free descent and backtrack)"}


def time_steps(step, stream, n_steps: int) -> float:
    """Milliseconds for n_steps calls of step(), CUDA events on `stream`
    with a device synchronisation on both sides."""
    import torch
    torch.cuda.synchronize()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for _ in range(n_steps):
        step()
    ev1.record(stream)
    torch.cuda.synchronize()
    return ev0.elapsed_time(ev1)


def workload_rows(kdt, dev, stream, peak, names, steps: int, oracle_full: bool) -> list[dict]:
    """The smaller workloads, each timed like the headline one (device-resident
    points, caller workspace, CUDA events over `steps` builds after 3 warm-up
    builds), checked by the GPU verifier and, unless disabled, element by
    element against the CPU oracle run on the same full-size input (its
    single-threaded build time is reported beside the GPU's)."""
    import numpy as np
    import torch
    from balanced_tree_build_gb300.inputs import WORKLOADS
    rows = []
    for name in names:
        w = WORKLOADS[name]
        host = w.points()
        pts = torch.from_numpy(host).to(dev)
        perm = torch.empty(w.n, dtype=torch.int32, device=dev)
        ws = kdt.alloc_workspace(w.n, w.k, w.mode, device=dev)

        def step():
            kdt.build_tree(pts, w.mode, out=perm, workspace=ws, stream=stream)

        for _ in range(3):
            step()
        ms = time_steps(step, stream, steps) / steps
        rc = kdt.status(stream)
        if rc != 0:
            raise SystemExit(f"{name}: device status {rc}")
        if not kdt.verify_tree(pts, perm, w.mode, stream=stream):
            raise SystemExit(f"{name}: the GPU verifier rejected the tree")
        balg = b_alg(w.n)
        gbs = balg / (ms / 1e3) / 1e9
        row = {"workload": name, "N": w.n, "k": w.k, "split_mode": "round_robin" if w.mode == 0 else "widest",
               "ms_per_build": ms, "points_per_s": w.n / (ms / 1e3), "B_alg_bytes": balg,
               "frac_of_measured": gbs / peak, "frac_of_nominal_8TBps": gbs / NOMINAL_HBM_GBS,
               "builds_timed": steps, "verified": "gpu verifier"}
        if oracle_full:
            import oracle
            t0 = time.perf_counter()
            want = oracle.get().build_tree(host, w.mode)
            row["oracle_s"] = time.perf_counter() - t0
            row["oracle_points_per_s"] = w.n / row["oracle_s"]
            if not np.array_equal(perm.cpu().numpy(), want):
                raise SystemExit(f"{name}: the GPU tree differs from the oracle's")
            row["verified"] = "gpu verifier + bit-exact equal to the full-size oracle build"
        rows.append(row)
        del pts, perm, ws
    return rows


def balanced_extra(kdt, pts, workload, stream, steps: int = 5) -> dict:
    """Times kdt_build_balanced (the median-split tree of Brown's builder,
    round-robin split) on the bench workload's points, device-resident, with
    a caller workspace; CUDA events over `steps` builds after 2 warm-ups."""
    import torch
    n, k = pts.shape
    out = torch.empty(kdt.balanced_slots(n), dtype=torch.int32, device=pts.device)
    ws = torch.empty(kdt.balanced_workspace_bytes(n, k), dtype=torch.uint8, device=pts.device)

    def step():
        kdt.build_balanced(pts, out=out, workspace=ws, stream=stream)

    for _ in range(2):
        step()
    ms = time_steps(step, stream, steps) / steps
    if kdt.status(stream) != 0:
        raise SystemExit("device status after the balanced builds")
    nodes = int((out >= 0).sum().item())
    if nodes != n:
        raise SystemExit("balanced tree: occupied slots != N")
    balg = b_alg(n)
    return {"ms": ms, "points_per_s": n / (ms / 1e3), "slots": out.numel(), "split_rule": "round_robin",
            "frac_of_measured_B_alg": balg / (ms / 1e3) / 1e9 / measured_peaks()[0],
            "api": "kdt_build_balanced (lower median, heap-ordered slots)"}


def run_ours(args, workload):
    import torch
    import balanced_tree_build_gb300 as kdt

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    active = init_dist(world, "nccl" if world > 1 else "gloo")
    dev = torch.device("cuda", local)

    pts_host = workload.points()
    n, k = pts_host.shape
    pts = torch.from_numpy(pts_host).to(dev)
    perm = torch.empty(n, dtype=torch.int32, device=dev)
    ws = kdt.alloc_workspace(n, k, workload.mode, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        kdt.build_tree(pts, workload.mode, out=perm, workspace=ws, stream=stream)

    # clock samples: nvidia-smi starts now, so that it samples by the time
    # the timed region begins; only samples inside that region are kept
    sampler = ClockSampler(gpu_identifier(local))
    sampler.start()
    for _ in range(max(args.warmup, 0)):
        step()
    torch.cuda.synchronize(dev)
    rc = kdt.status(stream)
    if rc != 0:
        raise SystemExit(f"device status after warm-up: {rc}")

    # timed region: the library's per-kernel timing is off here
    kdt.profile_enable(False)
    barrier(active)
    torch.cuda.synchronize(dev)
    t_wall0 = time.time()
    ms = time_steps(step, stream, args.steps)
    t_wall1 = time.time()
    barrier(active)
    clocks = sampler.stop((t_wall0, t_wall1))
    ms_max = max_over_ranks(ms, active, dev if active else None)
    rc = kdt.status(stream)
    if rc != 0:
        raise SystemExit(f"device status after timed steps: {rc}")
    # the last timed build's output, checked on the GPU (every node against
    # every ancestor, plus the permutation check)
    if not kdt.verify_tree(pts, perm, workload.mode, stream=stream):
        raise SystemExit("the GPU verifier rejected the benchmarked tree")

    total_points = float(n) * args.steps * world
    value = total_points / (ms_max / 1e3)
    ms_step = ms_max / args.steps

    # separate profiled pass: per-kernel CUDA events on the build's stream
    prof_steps = max(1, min(args.steps, 5))
    kdt.profile_reset()
    kdt.profile_enable(True)
    prof_ms = time_steps(step, stream, prof_steps)
    kdt.profile_enable(False)
    stats = kdt.profile_read()
    kdt.profile_reset()

    peak, peak_src = measured_peaks()
    launches_per_build = sum(s["kernels"] for s in stats) / prof_steps
    dom = max(stats, key=lambda s: s["total_ms"]) if stats else None
    roofline = None
    if dom:
        avg_ms = dom["total_ms"] / dom["launches"]
        avg_bytes = dom["bytes_alg"] / dom["launches"]
        achieved = avg_bytes / (avg_ms / 1e3) / 1e9
        traffic = recorded_traffic(dom["name"]) if workload.name == "uniform_100m" else None
        roofline = {"bound": "hbm", "kernel": dom["name"], "achieved": achieved, "peak": peak,
                    "unit": "GB/s", "frac": achieved / peak, "peak_source": peak_src,
                    "traffic": traffic, "avg_launch_ms": avg_ms, "alg_bytes_per_launch": avg_bytes,
                    "timing": f"CUDA events around each launch on the build's stream, in a separate "
                              f"profiled pass of {prof_steps} builds after the timed region"}
    balg = b_alg(n)
    build_gbs = balg / (ms_step / 1e3) / 1e9
    build_roof = {"B_alg_bytes": balg, "achieved_GBps": build_gbs, "frac_of_measured": build_gbs / peak,
                  "frac_of_nominal_8TBps": build_gbs / NOMINAL_HBM_GBS}

    e2e = None
    if not args.no_e2e:
        pin_pts = torch.from_numpy(pts_host).pin_memory()
        pin_out = torch.empty(n, dtype=torch.int32).pin_memory()
        hws = kdt.alloc_workspace(n, k, workload.mode, device=dev, host=True)
        for _ in range(2):
            kdt.build_tree_host(pin_pts, workload.mode, out=pin_out, workspace=hws, stream=stream)
        e_steps = max(1, min(args.steps, 5))
        barrier(active)
        t0 = time.perf_counter()
        for _ in range(e_steps):
            kdt.build_tree_host(pin_pts, workload.mode, out=pin_out, workspace=hws, stream=stream)
        dt = time.perf_counter() - t0
        dt = max_over_ranks(dt, active, dev if active else None)
        if not torch.equal(pin_out, perm.cpu()):
            raise SystemExit("the host-buffer build differs from the device build")
        # the link on its own, for context: one pinned H2D copy of the points
        # and one D2H copy of the permutation (CUDA events)
        tmp = torch.empty_like(pts)
        h2d_ms = time_steps(lambda: tmp.copy_(pin_pts, non_blocking=True), stream, 3) / 3
        d2h_ms = time_steps(lambda: pin_out.copy_(perm, non_blocking=True), stream, 3) / 3
        del tmp
        e2e = {"value": float(n) * e_steps * world / dt, "unit": UNIT,
               "h2d_bytes_per_step": int(n * k * 4), "d2h_bytes_per_step": int(n * 4),
               "steps": e_steps, "ms_per_step": dt * 1e3 / e_steps,
               "api": "kdt_build_host (pinned host buffers)",
               "link_alone": {"h2d_ms": h2d_ms, "h2d_GBps": n * k * 4 / (h2d_ms / 1e3) / 1e9,
                              "d2h_ms": d2h_ms, "d2h_GBps": n * 4 / (d2h_ms / 1e3) / 1e9}}
        del hws

    extras = None
    if not args.no_extras:
        lo, tree_pts = level_order_extra(kdt, pts, perm, ws, workload, stream, peak)
        extras = {"level_order_points": lo, "knn": knn_extra(kdt, tree_pts, workload, stream)}
        del tree_pts
        if workload.mode == 0:
            extras["balanced_tree"] = balanced_extra(kdt, pts, workload, stream)
    if not args.no_workloads and rank == 0:
        del ws
        torch.cuda.empty_cache()
        extras = extras or {}
        extras["workloads"] = workload_rows(kdt, dev, stream, peak,
                                            ["uniform_1k", "uniform_pm1_1m", "mixture_dup_10m", "quant1024_k8_4m"],
                                            10, not args.no_oracle_full)

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline(workload)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": workload_config(workload, extra={"parallelism": f"replicas x{world}"}),
            "verified": True, "roofline": roofline, "build_roofline": build_roof, "cpu_baseline": cpu,
            "e2e": e2e, "gpu_launches": int(round(launches_per_build * args.steps)),
            "kernels": stats, "profiled_ms_per_step": prof_ms / prof_steps, "clocks": clocks, "extras": extras,
        }
        print(json.dumps(line), flush=True)
    if active:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="uniform_100m")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extras", action="store_true", help="skip the level-order points and kNN timings")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the rows for the four smaller workloads")
    ap.add_argument("--no-oracle-full", action="store_true",
                    help="skip the full-size oracle builds of the smaller workloads")
    ap.add_argument("--ref-sample", type=int, default=1 << 20,
                    help="points per step for --impl reference")
    ap.add_argument("--n", type=int, default=None,
                    help="build a sample of this many points of the workload's distribution "
                         "instead of the full workload (profiling runs)")
    args = ap.parse_args(argv)
    from balanced_tree_build_gb300.inputs import WORKLOADS, Workload
    workload = WORKLOADS[args.workload]
    if args.n is not None and args.n != workload.n:
        w = workload
        workload = Workload(f"{w.name}_sample{args.n}", args.n, w.k, w.mode, w.dist, w.seed)
    if args.impl == "reference":
        return run_reference(args, workload)
    return run_ours(args, workload)


if __name__ == "__main__":
    sys.exit(main())
