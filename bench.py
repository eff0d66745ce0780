"""Benchmark of the MPM transfer step (bin + P2G + grid update + G2P).

Default workload: 3D quadratic B-spline, 256^3 nodes, 16,777,216 particles in
64 Gaussian blobs (sigma 0.02), int64 fixed point.  Every timed step bins the
particles, checks the accumulator bound (its range taken from the records the
previous step's P2G and G2P wrote), scatters, updates the grid and gathers;
seven steps in eight gather in place and every eighth with the sorted G2P,
which writes the new state in bin order into the second particle buffer
(ping-pong), so the steps stay in the steady state of a simulation that keeps
its particles sorted.  The other workloads of the method's configurations (the
512^3 sphere as a full step, the dam break in int64 and float-atomic modes and
at S = 2^32, the 2D int32 MLS case, the blobs at S = 2^32) are timed the same
way as extra rows of the line.

Prints one JSON line.  ``--impl reference`` times the CPU oracle on a bounded
sample of the same workload instead.  Under torchrun (N > 1) every rank runs an
independent replica (the step does not shard); the reported value is the sum
over ranks of particles per second at the slowest rank's time.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "P2G+G2P particles/sec (3D 256^3, 16M clustered); % of HBM roofline"
UNIT = "particles/s"
WORKLOAD = "blobs3d: 3D quadratic B-spline MPM step, 256^3 nodes, 16,777,216 particles in 64 Gaussian blobs " \
           "(sigma 0.02), int64 fixed point"
# kernels per step: bin (keys, 3 scans, runs, 2 run sorts, emit), the P2G call (the bound, the two share
# paths of which one returns at once, the undo that returns at once unless a particle broke the recorded
# range), G2P with the grid update on load; the sorted G2P adds the copy of the particles outside the domain
LAUNCHES_PER_STEP = 13
# The timed steps gather in place (mpm_g2p: one warp per work item), and every SORT_PERIOD-th step with
# mpm_g2p_sorted, which moves the particles into bin order and rewrites the bank-class interleave that the
# in-place steps keep and wear down; every step bins, scatters, updates and gathers every particle.
SORT_PERIOD = 8


# DRAM traffic per particle (dram__bytes_read.sum + dram__bytes_write.sum of one launch, divided by the
# particles it processed) from an ncu capture of the timed steps' P2G (the 22-bit instance), taken on the
# 2M-particle sample of the workload (same density) and scaled to a full launch by the particle count.
# Each figure holds only while the kernel's sources are the ones it was measured on (sha256 of the files).
MEASURED_TRAFFIC = {
    "p2g": {"bytes_per_particle": 82.2, "files": ('p2g.cu', 'common.cuh', 'scatter.cuh', 'stress.cuh', 'range.cuh'),
            "sha256": "edefb99ca279822bf7d50777c3f5979f02f56619c303ded74ec937898b9c4b16"
                      "4b1028dc922c926810222c631f1419edb36b336f9f5cae2e932a541931a000b7"
                      "dd28ea0fe9334290303e9b5c221100014b52c7cea975b1d29b3d662a3330f405"
                      "0c768a7fc62f6362d0285363fbfdcf0a3b8aa8e57edfd3d35d19bd9133d859f2"
                      "02130a6b5dd5211e01db3ff2aad034b7816abc055a35d45fabd3753f8eeadc19"},
}


def measured_traffic(kernel: str, n: int):
    """Bytes per launch of `kernel` for n particles, or None if not measured on these sources."""
    rec = MEASURED_TRAFFIC.get(kernel)
    if rec is None:
        return None
    import hashlib
    csrc = os.path.join(ROOT, "material_point_particle_gb300", "csrc")
    digest = "".join(hashlib.sha256(open(os.path.join(csrc, f), "rb").read()).hexdigest() for f in rec["files"])
    return round(rec["bytes_per_particle"] * n) if digest == rec["sha256"] else None


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def aggregate_max(value: float, world: int, device=None) -> float:
    """Max of `value` over ranks (identity when world == 1)."""
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int, device=None):
    if world > 1:
        import torch.distributed as dist
        if device is not None:
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


def load_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi clock/throttle samples during the timed region."""

    FIELDS = "index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active," \
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown," \
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap"

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join(tempfile.gettempdir(), f"mpm_bench_clocks_{os.getpid()}_{gpu_index}.csv")

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "20"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(nm)
        try:
            os.remove(self.path)
        except OSError:
            pass
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def workload(W, n_particles, n_blobs=64):
    return W.blobs3d(n_particles=n_particles, n_blobs=n_blobs)


def inputs_sha256(cloud) -> str:
    """SHA-256 of the generated particle arrays (x, v, C, m as stored fp32, in that order): the inputs the
    GPU and the oracle are given."""
    import hashlib
    h = hashlib.sha256()
    for k in ("x", "v", "C", "m"):
        h.update(np.ascontiguousarray(cloud[k]).tobytes())
    return h.hexdigest()


def run_ours(args, rank, world, local):
    import torch
    from material_point_particle_gb300 import _lib as L
    from material_point_particle_gb300 import workloads as W
    from material_point_particle_gb300.system import MPMSystem

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    cloud = workload(W, args.particles, args.blobs)
    grid = cloud["grid"]
    n = cloud["x"].shape[1]
    inputs_sha = inputs_sha256(cloud)
    sys_ = MPMSystem(grid, n, dev).load(cloud["x"], cloud["v"], cloud["C"], cloud["m"]).enable_sorted()
    # touched nodes of the initial state (algorithmic grid bytes)
    sys_.bin()
    sys_.p2g()
    touched = int((sys_.acc[0] != 0).sum().item())
    sys_.grid_update()
    torch.cuda.synchronize()
    st = sys_.status()
    assert st[L.ST_FLAGS] == 0, f"status flags {st[:8]}"
    stream = torch.cuda.current_stream(dev)
    # warm-up steps: the sorted step also moves the particles into bin order,
    # so the timed steps start from (and stay in) the steady state.  The first
    # one starts from the generated (blob-major) order: the cold step.
    c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for k in range(args.warmup):
        if k == 0:
            c0.record(stream)
        sys_.step_sorted(stream)
        if k == 0:
            c1.record(stream)
    torch.cuda.synchronize()
    cold_ms = c0.elapsed_time(c1) if args.warmup > 0 else None
    # from here on the bound takes its range from the records the previous P2G and G2P wrote, and each
    # in-place G2P writes the next step's keys and tile histogram, which that step's binning takes
    sys_.use_range_records(True)
    sys_.use_next_keys(True)
    # timed region
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    clocks = ClockSampler(local)
    barrier(world, dev)
    clocks.start()
    torch.cuda.synchronize()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for k in range(args.steps):
        e = ev[k]
        e[0].record(stream)
        sys_.bin(stream, keys_from_g2p=k % SORT_PERIOD != 0)   # the steps after an in-place G2P
        e[1].record(stream)
        sys_.p2g(stream)
        e[2].record(stream)
        # the grid update applied as G2P loads each tile's accumulators (no velocity grid)
        if (k + 1) % SORT_PERIOD == 0:
            sys_.g2p_sorted_update(stream)
        else:
            sys_.g2p_update(stream)
        e[3].record(stream)
    t_end.record(stream)
    torch.cuda.synchronize()
    barrier(world, dev)
    total_ms = t_start.elapsed_time(t_end)
    parts_ms = np.array([[e[i].elapsed_time(e[i + 1]) for i in range(3)] for e in ev])
    median_ms = aggregate_max(float(np.median(parts_ms.sum(axis=1))), world, dev)
    eager_ms = aggregate_max(total_ms / args.steps, world, dev)
    # the same schedule again, as a CUDA graph replayed (the headline); the eager region above gives the
    # per-phase times, which a replay does not expose
    graph = measure_graph(args.steps, bench_schedule(sys_, next_keys=True), stream, world, dev)
    clk = clocks.stop()
    st = sys_.status()
    assert st[L.ST_FLAGS] == 0, f"status flags after timing {st[:8]}"
    share_path = int(st[L.ST_SHARE_PATH])
    bound_range = float(np.array([st[L.ST_RANGE]], np.uint32).view(np.float32)[0])
    ms_step = graph["ms_per_step"] if "ms_per_step" in graph else eager_ms
    value = n * world / (ms_step * 1e-3)
    graph["eager"] = {"ms_per_step": round(eager_ms, 4), "value": round(n * world / (eager_ms * 1e-3), 1),
                      "median_ms_per_step": round(median_ms, 4)}
    # the advective step bound of the state the last timed G2P wrote
    speed = float(np.array([st[L.ST_MAX_SPEED]], np.uint32).view(np.float32)[0])
    advective = {"max_speed": speed, "dt_limit": grid["dx"] / speed if speed > 0 else None, "dt": sys_.dt}

    # roofline of the dominant kernel
    mean_ms = parts_ms.mean(axis=0)
    names = ["bin", "p2g", "g2p_update"]
    alg_bytes = {
        "bin": n * 24.0,
        "p2g": n * 64.0 + touched * 4 * 8.0,
        # read the accumulators of the touched nodes, read x, write x v C (the clear folded in is not
        # algorithmic, nor the m and id copies of the sorted output)
        "g2p_update": n * 72.0 + touched * 4 * 8.0,
    }
    dom = names[int(np.argmax(mean_ms))]
    peak, peak_kind = load_peaks()
    achieved = alg_bytes[dom] / (mean_ms[names.index(dom)] * 1e-3) / 1e9
    step_bytes = n * 160.0 + touched * 64.0
    roofline = {"bound": "hbm", "kernel": dom, "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4), "traffic": measured_traffic(dom, n), "peak_kind": peak_kind,
                "step_frac": round(step_bytes / (ms_step * 1e-3) / 1e9 / peak, 4)}
    # the transfer alone (P2G + the grid update and G2P, binning reported apart):
    # 136 B per particle and 64 B per touched node must move
    tr_ms = aggregate_max(float(mean_ms[1:].sum()), world, dev)
    transfer = {"ms_per_step": round(tr_ms, 4), "value": round(n * world / (tr_ms * 1e-3), 1), "unit": UNIT,
                "frac": round((n * 136.0 + touched * 64.0) / (tr_ms * 1e-3) / 1e9 / peak, 4),
                "bin_ms": round(float(mean_ms[0]), 4)}

    elastic = volume = fused = loop = schedules = None
    if args.variant_steps > 0:
        elastic = measure_variant(args, cloud, dev, stream, world, peak, elastic=True, volume=False)
        volume = measure_variant(args, cloud, dev, stream, world, peak, elastic=False, volume=True)
        fused = measure_fused(args, cloud, dev, stream, world, peak, touched, float(mean_ms[0]))
        loop = measure_loop(args, cloud, dev, stream, world, peak)
        schedules = measure_schedules(args, cloud, dev, stream, world)

    # end to end through the host entry point (pinned host SoA, copies inside the timed region)
    e2e = None
    if not args.no_e2e:
        pin = lambda t: torch.from_numpy(t.cpu().numpy()).pin_memory()
        hx, hv, hC, hm, hid = pin(sys_.x), pin(sys_.v), pin(sys_.C), pin(sys_.m), pin(sys_.id)
        host = L.particles(hx, hv, hC, hm, hid)
        for _ in range(max(1, args.warmup)):
            L.mpm_step_host(sys_.desc, host, sys_.parts, sys_.parts2, sys_.bins, sys_.acc, sys_.vel, sys_.dt,
                            sys_.dtg, stream)
        torch.cuda.synchronize()
        barrier(world, dev)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(args.steps):
            L.mpm_step_host(sys_.desc, host, sys_.parts, sys_.parts2, sys_.bins, sys_.acc, sys_.vel, sys_.dt,
                            sys_.dtg, stream)
        b.record(stream)
        torch.cuda.synchronize()
        e2e_ms = aggregate_max(a.elapsed_time(b) / args.steps, world, dev)
        e2e = {"value": round(n * world / (e2e_ms * 1e-3), 1), "unit": UNIT,
               "h2d_bytes_per_step": n * 17 * 4, "d2h_bytes_per_step": n * 17 * 4,
               "ms_per_step": round(e2e_ms, 4)}

    rows = None
    if args.workload_steps > 0:
        del sys_
        torch.cuda.empty_cache()
        rows = measure_workloads(args, dev, stream, world, peak, rank)

    cpu = cpu_omp = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline(cloud, sample=args.cpu_sample)
        cpu_omp = cpu_baseline_omp(cloud, particles=args.cpu_omp_particles)

    out = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32+i64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "particles": n, "grid": grid["n"], "acc": "int64",
                   "scale_log2": grid["scale_log2"], "tile": grid["tile"], "touched_nodes": touched,
                   "particle_order": "in place between sorted steps: every 8th step's G2P moves the particles "
                                     "into bin order with the bank-class interleave (ping-pong), the others "
                                     "gather in place",
                   "grid_update": "applied as G2P loads each tile's accumulators (mpm_g2p_update, "
                                  "mpm_g2p_sorted_update); the consumed accumulators cleared as G2P goes; "
                                  "no velocity grid",
                   "bound": {"range_source": "records of the previous step's P2G (max |m|) and G2P "
                                             "(max(1, |v| + 1.5 dx sum |C|)), verified per particle",
                             "range": bound_range,
                             "share_path": "22-bit shares, one fma each" if share_path == 0
                             else "int64 shares (exact integer product)"},
                   "l2": "inputs larger than L2 (1.07 GB of particle state per step)",
                   "inputs_sha256": inputs_sha,
                   "parallelism": f"replicas x{world}"},
        "timing": "the timed steps twice: first eagerly with CUDA events between the phases (breakdown_ms, "
                  "transfer, roofline, median), then the same schedule as a CUDA graph of one 16-step period "
                  "replayed (ms_per_step, value; cuda_graph.eager holds the eager region's step time)",
        "cuda_graph": graph,
        "breakdown_ms": {k: round(float(v), 4) for k, v in zip(names, mean_ms)},
        "transfer": transfer,
        "median_ms_per_step": round(median_ms, 4),
        "cold_step_ms": round(cold_ms, 4) if cold_ms is not None else None,
        "roofline": roofline,
        "e2e": e2e,
        "gpu_launches": LAUNCHES_PER_STEP * args.steps + args.steps // SORT_PERIOD,
        "clocks": clk,
        "advective_step_bound": advective,
        "mls_stress": elastic,
        "volume_channel": volume,
        "fused_step": fused,
        "transfer_loop": loop,
        "g2p_schedules": schedules,
        "workloads": rows,
    }
    if cpu is not None:
        out["cpu_baseline"] = cpu
        out["cpu_baseline_openmp"] = cpu_omp
    return out


ELASTIC = {"fsig": 0.05, "ppc": 1.0, "mu": 1.0e9, "lambda": 1.0e9}


def measure_graph(steps, run, stream, world, dev):
    """A schedule captured as one CUDA graph and replayed.  run(count, s) issues `count` steps on stream s
    (None: the current stream) starting at the first step of a period of 2 * SORT_PERIOD steps, after which the
    ping-pong particle buffers are back where they started (two sorted G2P steps).  One period is captured on a
    side stream (capture runs nothing), then replayed steps // period times and the steps left over run
    eagerly, all timed together with CUDA events.  Every call's launches are the eager ones; only the launch
    overhead between them goes."""
    import torch
    period = 2 * SORT_PERIOD
    try:
        side = torch.cuda.Stream(dev)
        side.wait_stream(stream)
        g = torch.cuda.CUDAGraph()
        # thread_local: CUDA calls of other threads (a process group's watchdog) do not void the capture
        with torch.cuda.graph(g, stream=side, capture_error_mode="thread_local"):
            run(period, None)      # None: the capturing stream
        torch.cuda.synchronize()
    except Exception as exc:       # report the eager numbers instead
        return {"error": f"capture failed: {type(exc).__name__}: {exc}"}
    reps, rest = divmod(steps, period)
    barrier(world, dev)
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        t0.record(stream)
        for _ in range(reps):
            g.replay()
        run(rest, stream)
        t1.record(stream)
    torch.cuda.synchronize()
    barrier(world, dev)
    ms = aggregate_max(t0.elapsed_time(t1) / steps, world, dev)
    return {"ms_per_step": round(ms, 4), "period_steps": period, "replays": reps, "eager_steps": rest}


def bench_schedule(sys_, fixed: bool = True, next_keys: bool = False):
    """The bench's step schedule on sys_ as run(count, stream): bin, P2G, and G2P with the update on load
    (fixed point; float atomics: the separate grid update, then G2P), sorted every SORT_PERIOD-th step.
    next_keys (int64, sys_.use_next_keys set): each binning after an in-place G2P takes the keys that G2P
    wrote (MPM_BIN_KEYS_FROM_G2P); the first step of a period follows a sorted G2P and computes them."""
    def run(count, s):
        for k in range(count):
            sort = (k + 1) % SORT_PERIOD == 0
            sys_.bin(s, keys_from_g2p=next_keys and k % SORT_PERIOD != 0)
            sys_.p2g(s)
            if fixed:
                sys_.g2p_sorted_update(s) if sort else sys_.g2p_update(s)
            else:
                sys_.grid_update(s)
                sys_.g2p_sorted(s) if sort else sys_.g2p(s)
    return run


def measure_variant(args, cloud, dev, stream, world, peak, elastic: bool, volume: bool):
    """The same workload with the elastic state (F = I + N(0, 0.05), V0 = dx^3,
    Neo-Hookean mu = lambda = 1e9: the stress folded into P2G's affine matrix,
    F advanced in G2P) and/or the grid-recovered volume channel (rest volume
    V0 = dx^3 scattered and gathered back).  Timed like the main region (the same
    G2P schedule), in the steady state, per phase; then replayed as a CUDA graph (the step time)."""
    import torch
    from material_point_particle_gb300 import _lib as L
    from material_point_particle_gb300 import workloads as W
    from material_point_particle_gb300.system import MPMSystem

    steps = args.variant_steps
    grid = dict(cloud["grid"], volume_channel=1 if volume else 0)
    ecloud = W.with_elastic(cloud, seed=77, fsig=ELASTIC["fsig"], ppc=ELASTIC["ppc"], mu=ELASTIC["mu"],
                            lam=ELASTIC["lambda"])
    n = cloud["x"].shape[1]
    es = MPMSystem(grid, n, dev).load(cloud["x"], cloud["v"], cloud["C"], cloud["m"])
    if elastic:
        es.load_elastic(ecloud["F"], ecloud["vol"], ecloud["material"])
    else:
        es.load_volume(ecloud["vol"])
    es.enable_sorted()
    del ecloud
    for _ in range(max(3, args.warmup)):
        es.step_sorted(stream)
    es.use_range_records(True)   # (the elastic state always takes the range pass: its C is stress-folded)
    nk = not elastic   # the next keys from G2P (measured slower with the elastic state's G2P)
    es.use_next_keys(nk)
    torch.cuda.synchronize()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(steps)]
    barrier(world, dev)
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for k in range(steps):
        e = ev[k]
        e[0].record(stream)
        es.bin(stream, keys_from_g2p=nk and k % SORT_PERIOD != 0)
        e[1].record(stream)
        es.p2g(stream)
        e[2].record(stream)
        if (k + 1) % SORT_PERIOD == 0:
            es.g2p_sorted_update(stream)
        else:
            es.g2p_update(stream)
        e[3].record(stream)
    t1.record(stream)
    torch.cuda.synchronize()
    eager_ms = aggregate_max(t0.elapsed_time(t1) / steps, world, dev)
    # the same schedule replayed as a CUDA graph (the row's step time; the eager region gives the phases)
    graph = measure_graph(steps, bench_schedule(es, next_keys=nk), stream, world, dev)
    graph["eager_ms_per_step"] = round(eager_ms, 4)
    ms = graph.get("ms_per_step", eager_ms)
    st = es.status()
    assert st[L.ST_FLAGS] == 0, f"status flags {st[:8]}"
    parts = np.array([[e[i].elapsed_time(e[i + 1]) for i in range(3)] for e in ev]).mean(axis=0)
    names = ["bin", "p2g", "g2p_update"]
    es.bin(stream)
    es.p2g(stream)
    touched = int((es.acc[0] != 0).sum().item())
    es.grid_update(stream)
    torch.cuda.synchronize()
    # algorithmic bytes: P2G reads the record (64 B) plus F (36 B) and V0 (4 B) as used, and writes
    # 8 B per channel per touched node; G2P reads x (and F) and writes x v C (and F, and phi)
    ch = 4 + (1 if volume else 0)
    alg = {"p2g": n * (64.0 + (36.0 if elastic else 0.0) + 4.0) + touched * 8.0 * ch,
           "g2p_update": n * (72.0 + (72.0 if elastic else 0.0) + (4.0 if volume else 0.0)) + touched * 8.0 * ch}
    dom = "p2g" if parts[1] >= parts[2] else "g2p_update"
    achieved = alg[dom] / (parts[names.index(dom)] * 1e-3) / 1e9
    out = {"ms_per_step": round(ms, 4), "value": round(n * world / (ms * 1e-3), 1), "unit": UNIT, "steps": steps,
           "cuda_graph": graph,
           "breakdown_ms": {k: round(float(v), 4) for k, v in zip(names, parts)},
           "out_of_range": int(st[L.ST_N_OUT_OF_RANGE]),
           "roofline": {"bound": "hbm", "kernel": dom, "achieved": round(achieved, 1), "peak": peak,
                        "unit": "GB/s", "frac": round(achieved / peak, 4),
                        "traffic": None}}
    if elastic:
        out["material"] = {"mu": ELASTIC["mu"], "lambda": ELASTIC["lambda"], "F": "I + N(0, 0.05) per entry",
                           "V0": "dx^3"}
        out["degenerate"] = int(st[L.ST_N_DEGENERATE])
    if volume:
        phi = es.phi.float()
        out["volume_fraction"] = {"V0": "dx^3 (one cell)", "mean": round(float(phi.mean().item()), 4),
                                  "max": round(float(phi.max().item()), 4)}
    del es
    torch.cuda.empty_cache()
    return out


def measure_fused(args, cloud, dev, stream, world, peak, touched, bin_ms):
    """The same workload stepped by mpm_step_fused (bin, then one kernel for the grid
    update, G2P and the next P2G, then the clear of the grid it read), after sorted
    steps have written the bank-class interleave; `steps` fused steps in a row, then as many replayed as a
    CUDA graph (the step time)."""
    import torch
    from material_point_particle_gb300 import _lib as L
    from material_point_particle_gb300.system import MPMSystem

    steps = args.variant_steps
    n = cloud["x"].shape[1]
    fs = MPMSystem(cloud["grid"], n, dev).load(cloud["x"], cloud["v"], cloud["C"], cloud["m"]).enable_sorted()
    # the sorted steps write the bank-class interleave, which the fused steps' bin order keeps
    for _ in range(max(3, args.warmup)):
        fs.step_sorted(stream)
    fs.enable_fused()
    torch.cuda.synchronize()
    barrier(world, dev)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    ev[0].record(stream)
    for k in range(steps):
        fs.step_fused(stream)
        ev[k + 1].record(stream)
    torch.cuda.synchronize()
    per = [ev[k].elapsed_time(ev[k + 1]) for k in range(steps)]
    eager_ms = aggregate_max(ev[0].elapsed_time(ev[steps]) / steps, world, dev)

    def run(count, s):   # every fused step swaps both buffer pairs: a period of 16 ends where it began
        for _ in range(count):
            fs.step_fused(s)

    graph = measure_graph(steps, run, stream, world, dev)
    graph["eager_ms_per_step"] = round(eager_ms, 4)
    ms = graph.get("ms_per_step", eager_ms)
    st = fs.status()
    assert st[L.ST_FLAGS] == 0, f"status flags {st[:8]}"
    # algorithmic bytes of the fused kernel: read x, m, id (20 B) and write x, v, C, m, id (68 B) per
    # particle; read the accumulators R and write W (32 B each per touched node)
    kern_ms = ms - bin_ms
    achieved = (n * 88.0 + touched * 64.0) / (kern_ms * 1e-3) / 1e9
    q = max(1, steps // 10)
    out = {"ms_per_step": round(ms, 4), "value": round(n * world / (ms * 1e-3), 1), "unit": UNIT, "steps": steps,
           "cuda_graph": graph,
           "first_tenth_ms": round(float(np.mean(per[:q])), 4), "last_tenth_ms": round(float(np.mean(per[-q:])), 4),
           "escaped": int(st[L.ST_N_ESCAPED]), "out_of_range": int(st[L.ST_N_OUT_OF_RANGE]),
           "roofline": {"bound": "hbm", "kernel": "g2p2g + clear (step minus the main region's bin time)",
                        "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                        "frac": round(achieved / peak, 4), "traffic": None}}
    del fs
    torch.cuda.empty_cache()
    return out


def measure_schedules(args, cloud, dev, stream, world):
    """The G2P schedules on the same workload, after sorted steps have written the
    bank-class interleave, `steps` steps each: in place with every 4th, 8th (the main
    region's schedule) or 16th step sorted, in place only, in bin order (mpm_step_binned)
    with every 8th step sorted, in bin order only, and sorted only."""
    import torch
    from material_point_particle_gb300 import _lib as L
    from material_point_particle_gb300.system import MPMSystem

    steps = args.variant_steps
    n = cloud["x"].shape[1]
    out = {"unit": UNIT, "steps": steps}
    plans = (("in_place_sorted_every_4", "in_place", 4), ("in_place_sorted_every_8", "in_place", 8),
             ("in_place_sorted_every_16", "in_place", 16), ("in_place", "in_place", 0),
             ("bin_order_sorted_every_8", "bin_order", 8), ("bin_order", "bin_order", 0),
             ("sorted_every_step", "in_place", 1))
    for name, kind, period in plans:
        bs = MPMSystem(cloud["grid"], n, dev).load(cloud["x"], cloud["v"], cloud["C"], cloud["m"]).enable_sorted()
        for _ in range(max(3, args.warmup)):
            bs.step_sorted(stream)
        bs.use_range_records(True)
        torch.cuda.synchronize()
        barrier(world, dev)
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
        ev[0].record(stream)
        for k in range(steps):
            if period and (k + 1) % period == 0:
                bs.step_sorted(stream)
            elif kind == "bin_order":
                bs.step_binned(stream)
            else:
                bs.step(stream)
            ev[k + 1].record(stream)
        torch.cuda.synchronize()
        st = bs.status()
        assert st[L.ST_FLAGS] == 0, f"status flags {st[:8]}"
        per = [ev[k].elapsed_time(ev[k + 1]) for k in range(steps)]
        ms = aggregate_max(ev[0].elapsed_time(ev[steps]) / steps, world, dev)
        q = max(1, steps // 10)
        out[name] = {"ms_per_step": round(ms, 4), "value": round(n * world / (ms * 1e-3), 1),
                     "first_tenth_ms": round(float(np.mean(per[:q])), 4),
                     "last_tenth_ms": round(float(np.mean(per[-q:])), 4)}
        del bs
        torch.cuda.empty_cache()
    return out


LOOP_ITERATIONS = 5


def measure_loop(args, cloud, dev, stream, world, peak):
    """The position-based solver's transfer loop on the same workload (particles in the
    order three sorted steps leave them): LOOP_ITERATIONS rounds of P2G -> grid update
    (no gravity) -> G2P (no advection) at fixed positions, once as mpm_iterate (one fused
    kernel per iteration) and once as the separate calls; binning and the first P2G are
    outside both timings."""
    import torch
    from material_point_particle_gb300 import _lib as L
    from material_point_particle_gb300.system import MPMSystem

    n = cloud["x"].shape[1]
    # the particles in the steady-state order the sorted steps keep (three steps of the workload)
    ss = MPMSystem(cloud["grid"], n, dev).load(cloud["x"], cloud["v"], cloud["C"], cloud["m"]).enable_sorted()
    for _ in range(3):
        ss.step_sorted(stream)
    state = [t.cpu().numpy() for t in (ss.x, ss.v, ss.C, ss.m)]
    del ss
    grid = dict(cloud["grid"], g=[0.0, 0.0, 0.0], dt=0.0)
    ls = MPMSystem(grid, n, dev).load(*state)
    del state
    acc_b = torch.zeros_like(ls.acc)
    reps = max(1, args.variant_steps // LOOP_ITERATIONS)

    def fused():
        ls.use_range_records(False)
        ls.bin(stream)
        ls.p2g(stream)
        a.record(stream)
        L.mpm_iterate(ls.desc, ls.parts, ls.bins, ls.acc, acc_b, LOOP_ITERATIONS, stream)
        b.record(stream)

    def separate():
        ls.use_range_records(False)
        ls.bin(stream)
        ls.p2g(stream)
        ls.use_range_records(True)   # the later P2G calls take the range from the previous G2P and P2G
        a.record(stream)
        for it in range(LOOP_ITERATIONS):
            ls.grid_update(stream)
            ls.g2p(stream)
            if it + 1 < LOOP_ITERATIONS:
                ls.p2g(stream)
        b.record(stream)

    out = {"iterations": LOOP_ITERATIONS, "unit": "ms per iteration"}
    for name, fn in (("fused", fused), ("separate", separate)):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        for _ in range(2):
            fn()
        torch.cuda.synchronize()
        total = 0.0
        for _ in range(reps):
            fn()
            torch.cuda.synchronize()
            total += a.elapsed_time(b)
        out[name] = round(aggregate_max(total / reps / LOOP_ITERATIONS, world, dev), 4)
    st = ls.status()
    assert st[L.ST_FLAGS] == 0, f"status flags {st[:8]}"
    del ls, acc_b
    torch.cuda.empty_cache()
    return out


def measure_row(args, cloud, dev, stream, world, peak, steps, label):
    """One workload timed as the main region: three sorted warm-up steps (the first, from the generated
    order, is the cold step), then `steps` steps binning, checking the bound (range from the records in the
    fixed-point modes), scattering, updating and gathering (fixed point: the update applied as G2P loads the
    accumulators; float atomics: the separate grid update), in place with a sorted G2P every
    SORT_PERIOD-th step.  Per-phase CUDA events; then the same schedule as a CUDA graph replayed
    (measure_graph), whose step time is the row's.  The roofline of the dominant kernel and of the whole step
    from the algorithmic bytes: bin 24 B (2D 20 B) per particle; P2G 64 B (2D 36 B) per particle plus (dim+1)
    accumulator words per touched node; grid update (dim+1) words per touched node; G2P 72 B (2D 40 B)."""
    import torch
    from material_point_particle_gb300 import _lib as L
    from material_point_particle_gb300.system import MPMSystem

    grid = cloud["grid"]
    dim = grid["dim"]
    n = cloud["x"].shape[1]
    fixed = grid["acc_mode"] in (L.MPM_ACC_I32, L.MPM_ACC_I64)
    ws = MPMSystem(grid, n, dev).load(cloud["x"], cloud["v"], cloud["C"], cloud["m"]).enable_sorted()
    ws.bin(stream)
    ws.p2g(stream)
    touched = int((ws.acc[0] != 0).sum().item())
    ws.grid_update(stream)
    c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for k in range(max(3, args.warmup)):
        if k == 0:
            c0.record(stream)
        ws.step_sorted(stream)
        if k == 0:
            c1.record(stream)
    torch.cuda.synchronize()
    cold = c0.elapsed_time(c1)
    nk = grid["acc_mode"] == L.MPM_ACC_I64   # the in-place G2P writes the next keys (int64 only)
    if fixed:
        ws.use_range_records(True)
    if nk:
        ws.use_next_keys(True)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(steps)]
    barrier(world, dev)
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for k in range(steps):
        e = ev[k]
        sort = (k + 1) % SORT_PERIOD == 0
        e[0].record(stream)
        ws.bin(stream, keys_from_g2p=nk and k % SORT_PERIOD != 0)
        e[1].record(stream)
        ws.p2g(stream)
        e[2].record(stream)
        if fixed:   # the grid update applied as G2P loads the accumulators
            e[3].record(stream)
            ws.g2p_sorted_update(stream) if sort else ws.g2p_update(stream)
        else:       # float atomics: the separate grid update, then G2P
            ws.grid_update(stream)
            e[3].record(stream)
            ws.g2p_sorted(stream) if sort else ws.g2p(stream)
        e[4].record(stream)
    t1.record(stream)
    torch.cuda.synchronize()
    eager_ms = aggregate_max(t0.elapsed_time(t1) / steps, world, dev)
    # the same schedule replayed as a CUDA graph (the row's step time; the eager region gives the phases)
    graph = measure_graph(steps, bench_schedule(ws, fixed, nk), stream, world, dev)
    graph["eager_ms_per_step"] = round(eager_ms, 4)
    st = ws.status()
    assert st[L.ST_FLAGS] == 0, f"{label}: status flags {st[:8]}"
    ms = graph.get("ms_per_step", eager_ms)
    names = ["bin", "p2g", "grid_update", "g2p"]
    parts = np.array([[e[i].elapsed_time(e[i + 1]) for i in range(4)] for e in ev]).mean(axis=0)
    wacc = 8.0 if grid["acc_mode"] == L.MPM_ACC_I64 else 4.0
    node = touched * (dim + 1) * wacc
    # with the update on load the G2P phase also reads the accumulators (and the grid_update phase is empty)
    alg = {"bin": n * (24.0 if dim == 3 else 20.0), "p2g": n * (64.0 if dim == 3 else 36.0) + node,
           "grid_update": 0.0 if fixed else node, "g2p": n * (72.0 if dim == 3 else 40.0) + (node if fixed else 0.0)}
    dom = names[int(np.argmax(parts))]
    achieved = alg[dom] / (parts[names.index(dom)] * 1e-3) / 1e9
    step_bytes = sum(alg.values())
    out = {"workload": label, "particles": n, "grid": grid["n"][:dim], "touched_nodes": touched,
           "acc": {L.MPM_ACC_I32: "int32", L.MPM_ACC_I64: "int64", L.MPM_ACC_F32: "fp32 atomics"}[grid["acc_mode"]],
           "scale_log2": grid["scale_log2"] if fixed else None,
           "share_path": (("22-bit" if st[L.ST_SHARE_PATH] == 0 else "int64") if fixed else None),
           "steps": steps, "ms_per_step": round(ms, 4), "value": round(n * world / (ms * 1e-3), 1), "unit": UNIT,
           "cuda_graph": graph,
           "cold_step_ms": round(cold, 4),
           "breakdown_ms": {k: round(float(v), 4) for k, v in zip(names, parts)},
           "transfer_ms": round(float(parts[1:].sum()), 4),
           "roofline": {"bound": "hbm", "kernel": dom, "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                        "frac": round(achieved / peak, 4), "traffic": None,
                        "step_bytes": round(step_bytes), "step_frac": round(step_bytes / (ms * 1e-3) / 1e9 / peak, 4)}}
    del ws
    torch.cuda.empty_cache()
    return out


def row_cpu_baseline(cloud):
    """The CPU baseline of one row: the OpenMP build of the oracle's step on all host cores (fixed point),
    or the oracle itself on one core (float atomics), one step of the whole workload after a warm-up."""
    from oracle import cpu_omp
    from oracle import oracle as O
    grid = cloud["grid"]
    n = cloud["x"].shape[1]
    if grid["acc_mode"] != 2 and cpu_omp.available():
        bufs = cpu_omp.buffers(grid, n)
        times = []
        for _ in range(2):
            t0 = time.perf_counter()
            cpu_omp.step_fixed(grid, cloud["x"], cloud["v"], cloud["C"], cloud["m"], out=bufs)
            times.append(time.perf_counter() - t0)
        dt = times[-1]
        return {"value": round(n / dt, 1), "unit": UNIT, "cores": cpu_omp.max_threads(), "kind": "openmp",
                "sample": f"the whole workload, one step after a warm-up: {dt:.3f} s"}
    O.build()
    t0 = time.perf_counter()
    acc, _, _ = O.p2g_float(grid, cloud["x"], cloud["v"], cloud["C"], cloud["m"])
    vel = O.grid_update_float(grid, acc)
    O.g2p(grid, vel, cloud["x"], cloud["v"], cloud["C"])
    dt = time.perf_counter() - t0
    return {"value": round(n / dt, 1), "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"the whole workload, one oracle step (P2G in fp64 sums, grid update, G2P): {dt:.2f} s"}


def measure_workloads(args, dev, stream, world, peak, rank):
    """The other configurations of the method's workloads, each a row timed like the main region (see
    measure_row), with its CPU baseline on rank 0: the 512^3 sphere (67,108,864 particles) as a full step
    with binning; the 128^3 dam break (2,097,152 particles) in int64 (S = 2^21 and S = 2^32, the int64
    share path) and in float-atomic mode, the comparison the float variant is kept for; the 2D 128^2 MLS
    case (65,536 particles) with int32 accumulators; the blobs at S = 2^32 (int64 shares)."""
    from material_point_particle_gb300 import workloads as W
    steps = args.workload_steps
    plans = [("sphere3d", lambda: W.sphere3d(), max(10, steps // 2)),
             ("dambreak3d_int64", lambda: W.dambreak3d(), steps),
             ("dambreak3d_int64_S2^32", lambda: W.dambreak3d(scale_log2=32), steps),
             ("dambreak3d_float_atomic", lambda: W.dambreak3d(acc_mode=W.ACC_F32), steps),
             ("mls2d_int32", lambda: W.mls2d(), steps),
             ("blobs3d_int64_S2^32", lambda: W.blobs3d(scale_log2=32), steps)]
    if args.workloads:
        keep = set(args.workloads.split(","))
        unknown = keep - {label for label, _, _ in plans}
        if unknown:
            raise SystemExit(f"unknown workload rows: {sorted(unknown)}")
        plans = [pl for pl in plans if pl[0] in keep]
    out = {}
    for label, make, k in plans:
        cloud = make()
        row = measure_row(args, cloud, dev, stream, world, peak, k, label)
        if rank == 0 and not args.no_cpu_baseline and label != "blobs3d_int64_S2^32":
            row["cpu_baseline"] = row_cpu_baseline(cloud)
        out[label] = row
        del cloud
    if "sphere3d" in out:
        out["sphere3d"]["note"] = "full step (binning included), the roofline's step bytes 160 B per particle + " \
                                  "64 B per touched node"
    return out


def cpu_baseline(cloud, sample: int):
    """The oracle as it stands, timed on the host on the first `sample` particles."""
    from oracle import oracle as O
    grid = cloud["grid"]
    x, v, C, m = (cloud[k][..., :sample].copy() for k in ("x", "v", "C", "m"))
    O.build()
    t0 = time.perf_counter()
    O.step_fixed(grid, x, v, C, m)
    dt = time.perf_counter() - t0
    return {"value": round(sample / dt, 1), "unit": UNIT, "cores": 1, "kind": "oracle", "cpu": cpu_model(),
            "sample": f"first {sample} particles (storage order) of the same workload, full 256^3 grid, "
                      f"one full oracle step (bin, P2G, grid update, G2P): {dt:.2f} s"}


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else the machine type) and its core count."""
    import platform
    import subprocess
    name = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                name = line.split(":", 1)[1].strip()
                break
    except (OSError, subprocess.SubprocessError):
        pass
    if not name:
        try:
            for line in open("/proc/cpuinfo"):
                if line.lower().startswith("model name"):
                    name = line.split(":", 1)[1].strip()
                    break
        except OSError:
            pass
    return f"{name or platform.machine()}, {os.cpu_count()} cores"


def cpu_baseline_omp(cloud, particles: int):
    """The multi-core CPU baseline (OpenMP: the oracle's arithmetic, private per-thread int64 grids merged by
    integer add, outputs in bin order) on all host cores: one warm-up and two timed full steps of the first
    `particles` particles (all by default) on the full grid."""
    from oracle import cpu_omp
    if not cpu_omp.available():
        return {"unavailable": "the host compiler has no OpenMP"}
    grid = cloud["grid"]
    n = cloud["x"].shape[1] if particles <= 0 else min(particles, cloud["x"].shape[1])
    state = {k: np.ascontiguousarray(cloud[k][..., :n]) for k in ("x", "v", "C", "m")}
    bufs = [cpu_omp.buffers(grid, n), cpu_omp.buffers(grid, n)]   # ping-pong, as the GPU path
    times = []
    for k in range(3):
        t0 = time.perf_counter()
        state = cpu_omp.step_fixed(grid, state["x"], state["v"], state["C"], state["m"], out=bufs[k % 2])
        times.append(time.perf_counter() - t0)
    dt = min(times[1:])
    phases = cpu_omp.phase_seconds()
    return {"value": round(n / dt, 1), "unit": UNIT, "cores": cpu_omp.max_threads(), "kind": "openmp",
            "cpu": cpu_model(),
            "sample": f"{n} particles of the same workload, full 256^3 grid, one full step (bin, P2G with "
                      f"private per-thread int64 grids merged by integer add, grid update, G2P; outputs in bin "
                      f"order), best of 2 after a warm-up: {dt:.3f} s", "phases_s": phases}


def run_reference(args, rank, world):
    if rank != 0:
        return None
    from material_point_particle_gb300 import workloads as W
    from oracle import oracle as O
    cloud = W.blobs3d(n_particles=args.particles)
    grid = cloud["grid"]
    sample = args.ref_sample
    x, v, C, m = (cloud[k][..., :sample].copy() for k in ("x", "v", "C", "m"))
    O.build()
    for _ in range(args.warmup):
        O.step_fixed(grid, x, v, C, m)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        O.step_fixed(grid, x, v, C, m)
    dt = (time.perf_counter() - t0) / args.steps
    value = sample / dt
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32+i64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "particles": args.particles, "grid": grid["n"], "acc": "int64"},
        "cpu_baseline": {"value": round(value, 1), "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": f"first {sample} particles of the workload per step, full grid"},
        "e2e": {"value": round(value, 1), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--particles", type=int, default=16777216)
    ap.add_argument("--blobs", type=int, default=64, help="blobs (64 = the workload; fewer keeps the density "
                    "of a smaller sample, for profiling)")
    ap.add_argument("--cpu-sample", type=int, default=2097152)
    ap.add_argument("--cpu-omp-particles", type=int, default=0,
                    help="particles of the workload the OpenMP CPU baseline steps (0: all)")
    ap.add_argument("--ref-sample", type=int, default=262144)
    ap.add_argument("--variant-steps", type=int, default=50,
                    help="timed steps of the same workload with the Neo-Hookean stress, and with the "
                         "volume channel (0: skip both)")
    ap.add_argument("--workloads", default="",
                    help="comma-separated workload rows to time (default: all of them)")
    ap.add_argument("--workload-steps", type=int, default=50,
                    help="timed steps of each other workload row (sphere, dam break, mls2d, blobs at S = 2^32; "
                         "0: skip them)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        print("warning: fewer than 3 warm-up steps", file=sys.stderr)
    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if args.impl == "ours" else "gloo"
        if args.impl == "ours":
            import torch
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    if args.impl == "reference":
        out = run_reference(args, rank, world)
    else:
        out = run_ours(args, rank, world, local)
    if rank == 0 and out is not None:
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
