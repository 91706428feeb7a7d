"""Benchmark of libpk's persistent Jacobi sweep on one GB300 (or N replicas).

Default workload: Laplace fp32 on a 16384 x 16384 interior grid (two 1 GiB
ping-pong buffers, field uniform [0,1) from seed 3), 100 sweeps per step, run
as ONE persistent cooperative kernel per step (pk_run_sweeps).  The field is
2 GiB, larger than L2, so no flush is needed between steps.

Prints one JSON line (rank 0).  ``value`` is whole-job cell-updates/s from
CUDA events recorded on the launching stream around each kernel (libpk
records them; pk_run_info.device_us); ``e2e`` is the same metric through the
public C ABI with host buffers (pinned H2D copy of each step's field, the
sweeps, a D2H copy of its result) on the host clock, the steps run through
pk_run_batch, which overlaps one step's copies with the next one's sweeps.  ``roofline`` reports the
dominant kernel's algorithmic HBM bytes per launch over its event time,
against the measured copy bandwidth.  Each pass over the field reads the
current iterate once and writes the next one once (8 B per cell, 12 with a
Poisson source); a pass of a shape with D sweeps per pass (temporal
blocking) advances D sweeps for those 8 B, so the sweeps' compulsory
traffic is 8/D B per cell-update there (2.67 B at the default three).
``cpu_baseline`` times the CPU
oracle on a bounded sample of the same workload, single-threaded.

``--impl reference`` runs the CPU oracle arm instead (the only reference for
this method), on the same config and metric.

Under torchrun (N > 1) every rank runs an independent replica on its own GPU
(the method runs on one GPU; nothing is exchanged on the data path); host
timing is combined with a gloo max-reduction.
"""
import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "us/sweep (persistent vs per-launch) and cell-updates/s; HBM GB/s vs peak"
UNIT = "cell-updates/s"

WORKLOADS = {
    # name: (n, seed, sweeps, poisson, tol, check_every)
    "laplace-16384x16384-100sweeps": (16384, 3, 100, False, 0.0, 0),
    "poisson-4096x4096-2000sweeps-res10": (4096, 2, 2000, True, 1e-4, 10),
    "laplace-512x512-1000sweeps": (512, 1, 1000, False, 0.0, 0),
    "laplace-64x64-topedge-100sweeps": (64, None, 100, False, 0.0, 0),
    # profiling-sized cases: inputs larger than L2, short enough for ncu replays
    "laplace-8192x8192-10sweeps": (8192, 3, 10, False, 0.0, 0),
    # seven passes: checks at 0, 10 and 20 fall in stages 1, 2 and 3
    "poisson-4096x4096-21sweeps-res10": (4096, 2, 21, True, 1e-4, 10),
    "poisson-4096x4096-21sweeps": (4096, 2, 21, True, 0.0, 0),
    # the same for Laplace: checks at 0, 10 and 20 (tolerance below any residual)
    "laplace-8192x8192-21sweeps-res10": (8192, 3, 21, False, 1e-30, 10),
}
DEFAULT_WORKLOAD = "laplace-16384x16384-100sweeps"

# DRAM traffic of one launch of the dominant kernel, from the ncu capture
# summarised in profiles/ (dram__bytes_read.sum + dram__bytes_write.sum of
# one full-size launch: 16384^2, 100 sweeps); valid only while the kernel
# source hash and the STREAM shape match.
TRAFFIC = {"kernel_sha": "c47dbabb6dba974d", "stream_config": 10,
           "bytes_per_launch": 37.969e9 + 36.674e9}


# pk_options.stream_config shapes: (float4 groups per thread, ring depth, sweeps per pass,
# consumer threads per CTA)
SHAPES = {0: (1, 8, 1, 256), 1: (1, 16, 1, 256), 2: (2, 8, 1, 256), 3: (4, 4, 1, 256), 4: (4, 8, 1, 256),
          5: (2, 16, 1, 256), 6: (1, 8, 2, 256), 7: (2, 8, 2, 256), 8: (1, 16, 2, 256), 9: (2, 16, 2, 256),
          10: (1, 16, 3, 224), 11: (1, 8, 3, 224), 12: (1, 16, 3, 256), 13: (1, 16, 3, 128),
          14: (1, 16, 3, 128)}


def shape_label(info, poisson):
    if info["variant"] != 2:
        return {1: "k_persistent_direct", 3: "k_persistent_local"}[info["variant"]] + \
            ("2" if info["variant"] == 3 and info["sweeps_per_pass"] == 2 else "")
    q, ring, depth, cons = SHAPES[info["stream_config"]]
    return "k_persistent_stream<{%d float4/thread, %d-deep ring, %d sweep%s/pass, %d consumers}, %s>" % (
        q, ring, depth, "s" if depth > 1 else "", cons, "poisson" if poisson else "laplace")


def passes_of(info, sweeps, tol, check_every, exit_at=None):
    """Passes a persistent run over `sweeps` sweeps takes: (passes that
    store, check-only passes).  A shape of D sweeps per pass takes up to D
    sweeps per pass, never past the end; a pass of fewer than three sweeps
    stops at a residual check, while a three-sweep STREAM pass runs past one
    (the check is taken in its stage 2 or 3) when no second check falls
    inside it.  exit_at: the check at which the run stopped early (then a
    straddled check costs one more pass, which sweeps again to that
    iterate)."""
    checks = tol > 0 and check_every > 0
    depth = info["sweeps_per_pass"]
    straddle = checks and bool(info.get("straddle"))
    k, store_passes, check_only = 0, 0, 0
    while True:
        here = checks and k % check_every == 0
        if k == sweeps:
            check_only += 1 if here else 0
            break
        m, cs = sweeps - k, 1 if here else 0
        if checks:
            to_check = check_every - k % check_every
            if straddle and not here and to_check < depth and m >= depth \
                    and to_check + check_every >= depth:
                cs, m = to_check + 1, depth
            elif to_check < m:
                m = to_check
        store_passes += 1
        if cs and exit_at is not None and 0 < exit_at == k + cs - 1:
            store_passes += 1 if cs >= 2 else 0
            break
        k += min(m, depth)
    return store_passes, check_only


def algorithmic_bytes(info, cells, sweeps, poisson, tol, check_every):
    """Compulsory HBM bytes of one persistent run: every pass reads U (and g)
    once and, unless it only checks, writes U once."""
    done = info.get("sweeps_done", sweeps)
    exit_at = done if done < sweeps else None
    store_passes, check_only = passes_of(info, sweeps, tol, check_every, exit_at)
    src = 4.0 if poisson else 0.0
    return cells * (store_passes * (8.0 + src) + check_only * (4.0 + src))


def kernel_source_sha():
    """Hash of the headline kernel's sources, comments and blank lines
    removed, so that only a change to the code retires the traffic record."""
    h = hashlib.sha256()
    for name in ("pk_stream.cuh", "pk_stream_d3.cu", "pk_sweep.cuh", "pk_device.cuh", "pk_internal.h"):
        with open(os.path.join(ROOT, "iterative_stencil_solver_gb300", "csrc", name)) as fh:
            text = re.sub(r"/\*.*?\*/", "", fh.read(), flags=re.S)
        for line in text.splitlines():
            line = re.sub(r"//.*", "", line).rstrip()
            if line:
                h.update(line.encode() + b"\n")
    return h.hexdigest()[:16]


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as fh:
            d = json.load(fh)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def make_workload(name):
    from iterative_stencil_solver_gb300 import inputs
    n, seed, sweeps, poisson, tol, ce = WORKLOADS[name]
    if name.startswith("laplace-64x64-topedge"):
        w = inputs.workload_laplace_top_edge(n)
    elif poisson:
        w = inputs.workload_poisson_random_source(n, seed)
    else:
        w = inputs.workload_laplace_random(n, seed)
    w.update(sweeps=sweeps, tol=tol, check_every=ce)
    return w


# ---- distributed plumbing (replicas only) -------------------------------------

def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group("gloo", rank=rank, world_size=world)
    return world, rank, local


def dist_barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def dist_max(world, value):
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def dist_sum(world, value):
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# ---- clocks -------------------------------------------------------------------

class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        try:
            self.fh = tempfile.NamedTemporaryFile("w", prefix="pk_clocks_%d_" % self.index,
                                                  suffix=".csv", delete=False)
            self.path = self.fh.name
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.QUERY,
                 "--format=csv,noheader,nounits", "-lms", "50"], stdout=self.fh,
                stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
            return
        # wait (up to 5 s) for the sampler's first line, so that it is
        # running when the timed region starts
        t0 = time.time()
        while time.time() - t0 < 5.0 and self.proc.poll() is None:
            if os.path.getsize(self.path) > 0:
                break
            time.sleep(0.02)
        self.offset = 0

    def mark(self):
        """Start of the timed region: samples written before it are ignored."""
        if self.proc is not None:
            self.offset = os.path.getsize(self.path)

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        try:
            return self._summary()
        finally:
            os.unlink(self.path)

    def _summary(self):
        sm, smax, reasons = [], 0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        offset = getattr(self, "offset", 0)
        with open(self.path) as fh:
            before = fh.read(offset).splitlines()
            lines = fh.read().splitlines()
        # (a line the mark cut in two has fewer than nine fields on each side)
        window = "timed region"
        if not [l for l in lines if len(l.split(",")) >= 9]:
            # no sample fell inside a short timed region: the last one taken
            # before it, during the warm-up steps that ran just before
            lines = [l for l in before if len(l.split(",")) >= 9][-1:]
            window = "last warm-up sample (timed region shorter than the 50 ms period)"
        for line in lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = max(smax, float(parts[2]))
            except ValueError:
                continue
            for name, flag in zip(names, parts[5:9]):
                if flag.lower() == "active":
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(sm), "window": window}


# ---- CPU oracle timing ---------------------------------------------------------

def oracle_sample(w, target_s=10.0, max_rows=None, threads=1):
    """Time the oracle (single-threaded unless `threads` > 1: its OpenMP split
    of the row loop, bit-identical) on a band of the workload's rows.

    The band keeps the full row width; its top and bottom rows act as its
    ring.  Returns (cell-updates/s, description, seconds)."""
    import oracle
    nx = w["nx"]
    ny = w["ny"] if max_rows is None else min(w["ny"], max_rows)
    band = np.ascontiguousarray(w["u0"][:ny + 2])
    f = None if w["f"] is None else np.ascontiguousarray(w["f"][:ny])
    h2 = oracle.h2(nx)
    t0 = time.perf_counter()
    oracle.jacobi_run(band, f=f, n=2, h2v=h2, threads=threads)
    per_sweep = max((time.perf_counter() - t0) / 2.0, 1e-6)
    sweeps = int(max(1, min(w["sweeps"], target_s / per_sweep)))
    t0 = time.perf_counter()
    oracle.jacobi_run(band, f=f, n=sweeps, h2v=h2, threads=threads)
    dt = time.perf_counter() - t0
    updates = float(nx) * ny * sweeps
    desc = "%d sweeps over a %d x %d band of the %d x %d workload, %d thread%s" % (
        sweeps, nx, ny, w["nx"], w["ny"], threads, "s" if threads > 1 else "")
    return updates / dt, desc, dt


def reference_arm(args, world, rank):
    if rank != 0:
        return
    w = make_workload(args.workload)
    import oracle  # noqa: F401
    rows = min(w["ny"], max(1, int(4e7 // w["nx"])))  # ~4e7 cells per sweep sample
    values, secs = [], []
    for step in range(args.warmup + args.steps):
        v, desc, dt = oracle_sample(w, target_s=1.0, max_rows=rows)
        if step >= args.warmup:
            values.append(v)
            secs.append(dt)
    value = statistics.median(values)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        # a step here is one bounded sample (see cpu_baseline.sample)
        "ms_per_step": 1e3 * statistics.mean(secs), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": args.workload},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---- supplementary measurements (rank 0) ------------------------------------------

def barrier_spin(pk, w, sweeps, **opts):
    """Per-CTA time spent waiting between passes over one persistent run
    (%globaltimer around each wait, PK_FLAG_PROFILE_BARRIER): at the grid
    barrier, or for the pass counters of the CTAs a pass reads from."""
    flags = opts.pop("flags", pk.PK_FLAG_ALTERNATE_DIRECTION) | pk.PK_FLAG_PROFILE_BARRIER
    ctx = pk.pk_create(w["nx"], w["ny"], w["u0"], w["f"], pk.pk_options_default(flags=flags, **opts))
    try:
        pk.pk_run_sweeps(ctx, sweeps)
        info = pk.pk_run_sweeps(ctx, sweeps)
        waits = pk.pk_barrier_wait_ns(ctx).astype(np.float64)
    finally:
        pk.pk_destroy(ctx)
    passes = info["passes"]
    run_ns = info["device_us"] * 1e3
    return {"kernel": shape_label(info, w["f"] is not None), "grid": info["grid"],
            "pass_order": "pass counters" if info["pass_counters"] else "grid barrier",
            "passes": passes, "barriers": info["barriers"], "run_us": info["device_us"],
            "wait_us_per_pass_mean": float(waits.mean()) / passes / 1e3,
            "wait_us_per_pass_max_cta": float(waits.max()) / passes / 1e3,
            "wait_fraction_of_run_mean": float(waits.mean()) / run_ns}


def latency_extras(pk):
    """512^2 persistent vs per-launch (1000 sweeps), floors, barrier costs, and
    the task-queue round trip (10,000 tasks)."""
    from iterative_stencil_solver_gb300 import inputs
    out = {}
    w = inputs.workload_laplace_random(512, 1)
    ctx = pk.pk_create(512, 512, w["u0"], None)
    try:
        plan = pk.pk_get_plan(ctx)
        for _ in range(3):
            pk.pk_run_sweeps(ctx, 1000)
            pk.pk_run_sweeps_launch(ctx, 1000)
        pers = [pk.pk_run_sweeps(ctx, 1000)["device_us"] / 1000 for _ in range(5)]
        launch = [pk.pk_run_sweeps_launch(ctx, 1000)["device_us"] / 1000 for _ in range(5)]
        pk.pk_run_sweeps_graph(ctx, 1000)
        graph = [pk.pk_run_sweeps_graph(ctx, 1000)["device_us"] / 1000 for _ in range(5)]
        sync_each, queued = pk.pk_bench_launch_floor(ctx, 2000)
        nb = 10000

        def per_barrier(kind):
            b0 = pk.pk_bench_barrier(ctx, kind, 0, 0)
            return (pk.pk_bench_barrier(ctx, kind, 0, nb) - b0) / nb

        ours = per_barrier(2)          # monotonic-counter construction (default)
        gen = per_barrier(0)           # count + generation words
        cgs = per_barrier(1)           # cooperative_groups grid.sync
        p_med, l_med = statistics.median(pers), statistics.median(launch)
        out["laplace_512_1000sweeps"] = {
            "persistent_us_per_sweep": p_med, "launch_us_per_sweep": l_med,
            "graph_us_per_sweep": statistics.median(graph),
            "persistent_speedup": l_med / p_med,
            "persistent_speedup_vs_graph": statistics.median(graph) / p_med, "grid": plan["grid"],
            "variant": {1: "direct", 2: "stream", 3: "local"}[plan["variant"]],
            "persistent_cell_updates_per_s": 512 * 512 / (p_med * 1e-6),
            "floors_us": {"empty_launch_sync_each": sync_each, "empty_launch_queued": queued,
                          "grid_barrier_counter": ours, "grid_barrier_generation": gen,
                          "cg_grid_sync": cgs},
            "persistent_sweep_in_barriers": p_med / ours if ours > 0 else None,
            "persistent_sweep_in_queued_launches": p_med / queued if queued > 0 else None,
        }
    finally:
        pk.pk_destroy(ctx)
    w = inputs.workload_laplace_top_edge(64)
    ctx = pk.pk_create(64, 64, w["u0"], None)
    try:
        for _ in range(3):
            pk.pk_run_sweeps(ctx, 100)
            pk.pk_run_sweeps_launch(ctx, 100)
        pers = statistics.median(pk.pk_run_sweeps(ctx, 100)["device_us"] / 100 for _ in range(5))
        launch = statistics.median(pk.pk_run_sweeps_launch(ctx, 100)["device_us"] / 100
                                   for _ in range(5))
        pk.pk_run_sweeps_graph(ctx, 100)
        graph = statistics.median(pk.pk_run_sweeps_graph(ctx, 100)["device_us"] / 100
                                  for _ in range(5))
        out["laplace_64_topedge_100sweeps"] = {"persistent_us_per_sweep": pers,
                                               "launch_us_per_sweep": launch,
                                               "graph_us_per_sweep": graph,
                                               "persistent_speedup": launch / pers,
                                               "persistent_speedup_vs_graph": graph / pers}
    finally:
        pk.pk_destroy(ctx)
    # task queue: 10,000 tasks alternating 1-sweep Jacobi (256^2) and axpy (65,536)
    import torch
    w = inputs.workload_task_queue(256, 65536, 4)
    dev = torch.device("cuda", torch.cuda.current_device())
    x = torch.from_numpy(w["x"]).to(dev)
    y = torch.from_numpy(w["y"]).to(dev)
    torch.cuda.synchronize()
    tasks = [pk.make_task(pk.PK_TASK_JACOBI, n_sweeps=1),
             pk.make_task(pk.PK_TASK_AXPY, a=0.5, x=x.data_ptr(), y=y.data_ptr(),
                          length=x.numel())]
    # Floors: a NOP on a task kernel of one CTA is the host<->device handshake
    # alone (CTA 0 completes NOPs without the grid); the device-side
    # hand-out (distributed shared memory) + gather of one task across the
    # task kernel's cluster, no host involved.
    ctx1 = pk.pk_create(256, 256, w["u0"], None, pk.pk_options_default(task_grid=1))
    try:
        echo = pk.pk_bench_tasks(ctx1, 0, [pk.make_task(pk.PK_TASK_NOP)], 5100)[100:] / 1e3
    finally:
        pk.pk_destroy(ctx1)
    ctx = pk.pk_create(256, 256, w["u0"], None)
    try:
        n_h = 20000
        pk.pk_bench_handoff(ctx, 0, n_h)
        handoff = (pk.pk_bench_handoff(ctx, 0, n_h) - pk.pk_bench_handoff(ctx, 0, 0)) / n_h
        bar = (pk.pk_bench_barrier(ctx, 2, pk.pk_get_plan(ctx)["task_grid"], 10000)
               - pk.pk_bench_barrier(ctx, 2, pk.pk_get_plan(ctx)["task_grid"], 0)) / 10000
        mb = pk.pk_bench_tasks(ctx, 0, tasks, 10100)[100:] / 1e3
        nop = pk.pk_bench_tasks(ctx, 0, [pk.make_task(pk.PK_TASK_NOP)], 2100)[100:] / 1e3
        pk.pk_shutdown(ctx)
        ln = pk.pk_bench_tasks(ctx, 1, tasks, 10100)[100:] / 1e3
        lnop = pk.pk_bench_tasks(ctx, 1, [pk.make_task(pk.PK_TASK_NOP)], 2100)[100:] / 1e3
        echo50 = float(np.percentile(echo, 50))
        out["task_queue_10000"] = {
            "floors_us": {"echo_one_cta_p50": echo50,
                          "echo_one_cta_p99": float(np.percentile(echo, 99)),
                          "handout_gather_task_cluster": handoff,
                          "grid_barrier_task_grid": bar},
            "p50_over_echo_plus_barrier": float(np.percentile(mb, 50)) / (echo50 + bar),
            "mailbox_round_trip_us": {"p50": float(np.percentile(mb, 50)),
                                      "p99": float(np.percentile(mb, 99))},
            "launch_sync_round_trip_us": {"p50": float(np.percentile(ln, 50)),
                                          "p99": float(np.percentile(ln, 99))},
            "nop_mailbox_round_trip_us": {"p50": float(np.percentile(nop, 50)),
                                          "p99": float(np.percentile(nop, 99))},
            "nop_launch_sync_round_trip_us": {"p50": float(np.percentile(lnop, 50)),
                                              "p99": float(np.percentile(lnop, 99))},
            "task_cluster_ctas": pk.pk_get_plan(ctx)["task_grid"],
        }
    finally:
        pk.pk_destroy(ctx)
    # Red-black Gauss-Seidel: 512^2 time per iteration, and iterations to
    # convergence against Jacobi sweeps on a 64^2 Poisson problem
    w = inputs.workload_laplace_random(512, 1)
    ctx = pk.pk_create(512, 512, w["u0"], None)
    try:
        for _ in range(2):
            pk.pk_run_redblack(ctx, 500)
            pk.pk_run_redblack_launch(ctx, 500)
        rbp = statistics.median(pk.pk_run_redblack(ctx, 500)["device_us"] / 500 for _ in range(5))
        rbl = statistics.median(pk.pk_run_redblack_launch(ctx, 500)["device_us"] / 500
                                for _ in range(5))
    finally:
        pk.pk_destroy(ctx)
    w = inputs.workload_poisson_random_source(64, 5)
    ctx = pk.pk_create(64, 64, w["u0"], w["f"])
    try:
        jac = pk.pk_run_sweeps(ctx, 1000000, 1e-6, 10)
        pk.pk_set_field(ctx, w["u0"])
        rb = pk.pk_run_redblack(ctx, 1000000, 1e-6, 10)
    finally:
        pk.pk_destroy(ctx)
    out["redblack"] = {
        "laplace_512_us_per_iteration": {"persistent": rbp, "launch": rbl,
                                         "persistent_speedup": rbl / rbp},
        "poisson_64_tol1e-6_check10": {"jacobi_sweeps": jac["sweeps_done"],
                                       "redblack_iterations": rb["sweeps_done"],
                                       "jacobi_us": jac["device_us"], "redblack_us": rb["device_us"]},
    }
    # Temporal blocking: one, two and three sweeps per HBM pass, same bits (16384^2, 100 sweeps)
    w = make_workload(DEFAULT_WORKLOAD)
    tb = {}
    for name, cfg in (("one_sweep_per_pass", 3), ("two_sweeps_per_pass", 8),
                      ("three_sweeps_per_pass", 10)):
        ctx = pk.pk_create(16384, 16384, w["u0"], None, pk.pk_options_default(stream_config=cfg))
        try:
            for _ in range(2):
                pk.pk_run_sweeps(ctx, 100)
            runs = [pk.pk_run_sweeps(ctx, 100) for _ in range(5)]
            us = statistics.median(r["device_us"] / 100 for r in runs)
            tb[name] = {"stream_config": cfg, "us_per_sweep": us,
                        "cell_updates_per_s": 16384 * 16384 / (us * 1e-6),
                        "dram_bytes_per_sweep_algorithmic":
                            algorithmic_bytes(runs[0], 16384 * 16384, 100, False, 0, 0) / 100}
        finally:
            pk.pk_destroy(ctx)
    tb["speedup_two"] = tb["one_sweep_per_pass"]["us_per_sweep"] / tb["two_sweeps_per_pass"]["us_per_sweep"]
    tb["speedup_three"] = tb["one_sweep_per_pass"]["us_per_sweep"] / tb["three_sweeps_per_pass"]["us_per_sweep"]
    out["temporal_blocking_16384_100sweeps"] = tb
    # Pass counters against a grid barrier after every pass (the same bits):
    # the default three-sweep shape, and the 8-deep-ring shape that was the
    # default with the barrier
    pc = {}
    for label, cfg in (("ring16", 10), ("ring8", 11)):
        for mode, flags in (("pass_counters", pk.PK_FLAG_ALTERNATE_DIRECTION),
                            ("barrier_every_pass",
                             pk.PK_FLAG_ALTERNATE_DIRECTION | pk.PK_FLAG_BARRIER_EVERY_PASS)):
            ctx = pk.pk_create(16384, 16384, w["u0"], None,
                               pk.pk_options_default(stream_config=cfg, flags=flags))
            try:
                for _ in range(2):
                    pk.pk_run_sweeps(ctx, 100)
                runs = [pk.pk_run_sweeps(ctx, 100) for _ in range(5)]
                pc["%s_%s" % (label, mode)] = {
                    "stream_config": cfg, "us_per_sweep": statistics.median(r["device_us"] / 100 for r in runs),
                    "barriers": runs[0]["barriers"], "passes": runs[0]["passes"]}
            finally:
                pk.pk_destroy(ctx)
    out["pass_counters_laplace_16384_100sweeps"] = pc
    # A residual check every 10 sweeps (11 checks; tol below any residual, so
    # all 100 sweeps run): passes that straddle the checks (the default) and
    # passes that stop at them; the same bits
    lr = {}
    for mode, flags in (("straddled", pk.PK_FLAG_ALTERNATE_DIRECTION),
                        ("checks_end_passes",
                         pk.PK_FLAG_ALTERNATE_DIRECTION | pk.PK_FLAG_CHECKS_END_PASSES)):
        ctx = pk.pk_create(16384, 16384, w["u0"], None, pk.pk_options_default(flags=flags))
        try:
            runs = []
            for rep in range(4):  # the first is a warm-up; each run starts from the workload's field
                pk.pk_set_field(ctx, w["u0"])
                info = pk.pk_run_sweeps(ctx, 100, 1e-30, 10)
                if rep:
                    runs.append(info)
            info = min(runs, key=lambda r: r["device_us"])
            lr[mode] = {"us_per_sweep": info["device_us"] / 100, "kernel": shape_label(info, False),
                        "straddle": info["straddle"], "passes": info["passes"],
                        "passes_model": sum(passes_of(info, 100, 1e-30, 10)),
                        "barriers": info["barriers"], "n_checks": info["n_checks"],
                        "res_last": info["res_last"]}
        finally:
            pk.pk_destroy(ctx)
    out["laplace_16384_res10"] = lr
    # Barrier spin: the headline kernel (one barrier per pass) and
    # the barrier-per-sweep DIRECT kernel on the L2-resident 512^2 grid.
    out["barrier_spin"] = {
        "laplace_16384_100sweeps": barrier_spin(pk, w, 100),
        "laplace_512_1000sweeps_direct": barrier_spin(pk, inputs.workload_laplace_random(512, 1),
                                                      1000, variant=1),
    }
    del w
    # Poisson 4096^2 with the in-kernel residual every 10 sweeps: passes that
    # straddle the checks (default) and passes that stop at them
    w = make_workload("poisson-4096x4096-2000sweeps-res10")
    res10 = {}
    for name, flags in (("straddled", pk.PK_FLAG_ALTERNATE_DIRECTION),
                        ("checks_end_passes",
                         pk.PK_FLAG_ALTERNATE_DIRECTION | pk.PK_FLAG_CHECKS_END_PASSES)):
        ctx = pk.pk_create(4096, 4096, w["u0"], w["f"], pk.pk_options_default(flags=flags))
        try:
            runs = []
            for rep in range(4):  # the first is a warm-up; each run starts from the workload's field
                pk.pk_set_field(ctx, w["u0"])
                info = pk.pk_run_sweeps(ctx, 2000, 1e-4, 10)
                if rep:
                    runs.append(info)
            info = min(runs, key=lambda r: r["device_us"])
            done = info["sweeps_done"]
            model = info
            res10[name] = {
                "us_per_sweep": info["device_us"] / max(1, done), "sweeps_done": done,
                "res_ratio": info["res_last"] / info["res0"] if info["res0"] else None,
                "kernel": shape_label(info, True), "passes": info["passes"],
                "passes_model": sum(passes_of(model, 2000, 1e-4, 10,
                                              done if done < 2000 else None)),
                "hbm_gbs_algorithmic": algorithmic_bytes(model, 4096 * 4096, 2000, True, 1e-4, 10)
                                       / (info["device_us"] * 1e-6) / 1e9,
                "n_checks": info["n_checks"],
            }
        finally:
            pk.pk_destroy(ctx)
    out["poisson_4096_res10"] = res10
    return out


def e2e_buffers(pk, w):
    """The e2e leg's page-locked host buffers (pk_host_array: on transparent
    huge pages where the kernel grants them), one field in and two out.
    Made before the device-timed steps: the huge-page faults can wake the
    kernel's background memory compaction, which slows host-device copies
    while it runs."""
    host_in = pk.pk_host_array(w["u0"].shape)
    host_in[...] = w["u0"]
    host_out = [pk.pk_host_array(w["u0"].shape) for _ in range(2)]
    return host_in, host_out


def compaction_pages():
    """Pages the kernel's memory compaction has scanned or isolated so far
    (/proc/vmstat), or None where the file cannot be read."""
    try:
        total = 0
        with open("/proc/vmstat") as fh:
            for line in fh:
                key, val = line.split()
                if key in ("compact_migrate_scanned", "compact_free_scanned", "compact_isolated"):
                    total += int(val)
        return total
    except (OSError, ValueError):
        return None


def wait_compaction_idle(limit_s=20.0, quiet_s=0.5):
    """Wait until memory compaction has been idle for quiet_s (at most
    limit_s); returns (seconds waited, idle reached)."""
    t0 = time.perf_counter()
    last = compaction_pages()
    if last is None:
        return 0.0, None
    quiet_since = t0
    while time.perf_counter() - t0 < limit_s:
        time.sleep(0.1)
        cur = compaction_pages()
        now = time.perf_counter()
        if cur != last:
            last, quiet_since = cur, now
        elif now - quiet_since >= quiet_s:
            return now - t0, True
    return time.perf_counter() - t0, False


def wait_huge_pages(arrays, target, limit_s=20.0):
    """Wait until the arrays' huge-page share is back at `target` (their
    share when made), at most limit_s; returns (seconds waited, reached)."""
    t0 = time.perf_counter()
    if not target:
        return 0.0, None
    while True:
        cur = huge_page_fraction(arrays)
        if cur is None or cur >= 0.999 * target:
            return time.perf_counter() - t0, cur is not None
        if time.perf_counter() - t0 >= limit_s:
            return time.perf_counter() - t0, False
        time.sleep(0.1)


def e2e_steps(pk, ctx, w, args, world, torch, buffers):
    """The bench steps end to end through the public API (host buffers in and
    out); returns the e2e record and the serial set/run/get number."""
    cells = w["nx"] * w["ny"]
    sweeps = w["sweeps"]
    # e2e through the public API with page-locked host buffers on huge pages
    # (e2e_buffers): every step uploads its field, sweeps and downloads its
    # result.  pk_run_batch runs the steps as a pipeline (step i+1's upload
    # and step i-1's download overlap step i's sweeps).
    host_in, host_out = buffers
    huge_before = huge_page_fraction([host_in] + host_out)
    host_in_t, host_out_t = torch.from_numpy(host_in), [torch.from_numpy(a) for a in host_out]
    pk.pk_run_batch(ctx, [host_in] * 3, [host_out[q % 2] for q in range(3)], sweeps, w["tol"],
                    w["check_every"])
    # The host settled before the timed batches.  On the GB300 hosts the
    # first batch call of a process (its device buffers and mapped records
    # made after many other contexts came and went) has split every huge
    # page of these buffers, which the kernel rebuilt within a second or
    # so; timed in between, the copies ran at a third of their rate.  So:
    # the buffers back on huge pages, then no memory compaction running.
    huge_wait_s, huge_back = wait_huge_pages([host_in] + host_out, huge_before)
    settle_s, settled = wait_compaction_idle()
    dist_barrier(world)
    t0 = time.perf_counter()
    infos = pk.pk_run_batch(ctx, [host_in] * args.steps,
                            [host_out[q % 2] for q in range(args.steps)], sweeps, w["tol"],
                            w["check_every"])
    e2e_s = dist_max(world, time.perf_counter() - t0)
    e2e_updates = sum(cells * info["sweeps_done"] for info in infos)
    e2e_value = dist_sum(world, e2e_updates) / e2e_s
    e2e_launches = len(infos) * 3  # per step: ring copy, persistent kernel, result record
    # the same steps one call after another (set, run, get), for context
    pk.pk_set_field(ctx, host_in)
    pk.pk_run_sweeps(ctx, sweeps, w["tol"], w["check_every"])
    pk.pk_get_field(ctx, host_out[0])
    dist_barrier(world)
    serial_steps = min(args.steps, 10)
    serial_updates = 0
    t0 = time.perf_counter()
    for _ in range(serial_steps):
        pk.pk_set_field(ctx, host_in)
        info = pk.pk_run_sweeps(ctx, sweeps, w["tol"], w["check_every"])
        pk.pk_get_field(ctx, host_out[0])
        serial_updates += cells * info["sweeps_done"]
    serial_s = dist_max(world, time.perf_counter() - t0)
    serial_value = dist_sum(world, serial_updates) / serial_s
    link = host_link_gbs(torch, host_in_t, host_out_t[0])
    link["huge_page_fraction"] = huge_page_fraction([host_in] + host_out)
    link["huge_page_fraction_before"] = huge_before
    sweeps_ms = statistics.median(i["device_us"] for i in infos) / 1e3
    copy_ms = 2 * host_in_t.numel() * 4 / (link["both_gbs"] * 1e9) * 1e3
    return {"value": e2e_value, "seconds": e2e_s, "launches": e2e_launches,
            "sweeps_ms_median": sweeps_ms, "link": link,
            # a step can go no faster than its sweeps or than both copies at
            # this box's two-way link rate, whichever is longer
            "bound_value": cells * sweeps / (max(sweeps_ms, copy_ms) * 1e-3),
            "serial_value": serial_value, "serial_steps": serial_steps,
            "compaction_settle": {"waited_s": settle_s, "idle": settled},
            "huge_page_wait": {"waited_s": huge_wait_s, "restored": huge_back}}


def huge_page_fraction(arrays):
    """Share of the arrays' bytes that the kernel backs with transparent huge
    pages (AnonHugePages of their mappings in /proc/self/smaps), or None
    where that file cannot be read."""
    spans = [(a.ctypes.data, a.ctypes.data + a.nbytes) for a in arrays]
    total = sum(e - b for b, e in spans)
    try:
        huge, cur = 0, None
        with open("/proc/self/smaps") as fh:
            for line in fh:
                head = line.split()[0]
                if "-" in head and not head.endswith(":"):
                    lo, hi = (int(x, 16) for x in head.split("-"))
                    cur = (lo, hi) if any(lo < e and b < hi for b, e in spans) else None
                elif cur and line.startswith("AnonHugePages:"):
                    huge += int(line.split()[1]) * 1024
        return min(1.0, huge / total) if total else None
    except (OSError, ValueError):
        return None


def host_link_gbs(torch, host_in_t, host_out_t):
    """This machine's host link with the e2e buffers: one field up, one down, and
    both at once on two streams (GB/s, the best of three)."""
    dev = torch.device("cuda", torch.cuda.current_device())
    d_in = torch.empty_like(host_in_t, device=dev)
    d_out = torch.empty_like(host_out_t, device=dev)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    nbytes = host_in_t.numel() * 4
    best = {"h2d_gbs": 0.0, "d2h_gbs": 0.0, "both_gbs": 0.0}
    for _ in range(3):
        for key in best:
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            if key in ("h2d_gbs", "both_gbs"):
                with torch.cuda.stream(s1):
                    d_in.copy_(host_in_t, non_blocking=True)
            if key in ("d2h_gbs", "both_gbs"):
                with torch.cuda.stream(s2):
                    host_out_t.copy_(d_out, non_blocking=True)
            torch.cuda.synchronize()
            dt = time.perf_counter() - t0
            moved = nbytes * (2 if key == "both_gbs" else 1)
            best[key] = max(best[key], moved / dt / 1e9)
    del d_in, d_out
    return best


# ---- main arm ----------------------------------------------------------------------

def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["pk", "reference"], default="pk")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default=DEFAULT_WORKLOAD)
    ap.add_argument("--no-extras", action="store_true", help="skip the supplementary measurements")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true",
                    help="skip the end-to-end measurement (profiling runs)")
    ap.add_argument("--stream-config", type=int, default=-1,
                    help="STREAM shape index (include/pk.h pk_options.stream_config), -1 = default")
    ap.add_argument("--profile-handoff", action="store_true",
                    help="only run the task kernel's device-side hand-out (pk_bench_handoff, "
                         "10,000 made-up tasks) four times and print its cost per task: a "
                         "small command to profile the task kernel with")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    world, rank, local = dist_setup()
    if args.impl == "reference":
        reference_arm(args, world, rank)
        return

    import torch
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device (there is no CPU fallback)")
    torch.cuda.set_device(local)
    from iterative_stencil_solver_gb300 import build_ext
    build_ext.build()
    from iterative_stencil_solver_gb300 import pk

    if args.profile_handoff:
        from iterative_stencil_solver_gb300 import inputs
        hw = inputs.workload_laplace_random(512, 1)
        ctx = pk.pk_create(512, 512, hw["u0"], None)
        try:
            us = [pk.pk_bench_handoff(ctx, 0, 10000) / 10000 for _ in range(4)]
            print(json.dumps({"handoff_us_per_task": us, "task_cluster_ctas": pk.pk_get_plan(ctx)["task_grid"]}))
        finally:
            pk.pk_destroy(ctx)
        return

    w = make_workload(args.workload)
    nx, ny, sweeps = w["nx"], w["ny"], w["sweeps"]
    cells = nx * ny
    ctx = pk.pk_create(nx, ny, w["u0"], w["f"],
                       pk.pk_options_default(stream_config=args.stream_config))
    try:
        buffers = None if args.no_e2e else e2e_buffers(pk, w)
        plan = pk.pk_get_plan(ctx)
        clocks = ClockSampler(local)
        clocks.start()  # samples the warm-up too: a short timed region may hold none
        for _ in range(args.warmup):
            pk.pk_run_sweeps(ctx, sweeps, w["tol"], w["check_every"])
        dist_barrier(world)
        torch.cuda.synchronize()
        clocks.mark()
        dev_us, updates = [], 0
        t0 = time.perf_counter()
        for _ in range(args.steps):
            info = pk.pk_run_sweeps(ctx, sweeps, w["tol"], w["check_every"])
            run_info = info
            dev_us.append(info["device_us"])
            updates += cells * info["sweeps_done"]
        torch.cuda.synchronize()
        host_s = time.perf_counter() - t0
        dist_barrier(world)
        clk = clocks.stop()
        dev_s = sum(dev_us) * 1e-6
        dev_s_max = dist_max(world, dev_s)
        updates_all = dist_sum(world, updates)
        value = updates_all / dev_s_max
        ms_per_step = dev_s_max * 1e3 / args.steps
        us_per_sweep = dev_s * 1e6 / (updates / cells)
        line = None if rank != 0 else result_line(args, w, world, value, ms_per_step, us_per_sweep,
                                                  dev_us, run_info, host_s, clk)
        # The end-to-end leg runs last, after the extras and the CPU
        # baseline: the first run on a host that has just released a lot of
        # page-locked memory (another process's exit) copied at about half
        # speed for some seconds.
        e2e = None if args.no_e2e else e2e_steps(pk, ctx, w, args, world, torch, buffers)
        del buffers
    finally:
        pk.pk_destroy(ctx)

    if rank != 0:
        return
    line["e2e"] = None if e2e is None else {
        "value": e2e["value"], "unit": UNIT,
        "h2d_bytes_per_step": int(w["u0"].nbytes),
        "d2h_bytes_per_step": int(w["u0"].nbytes),
        "api": "pk_run_batch (pipelined: uploads and downloads overlap the sweeps); "
               "host buffers from pk_host_alloc (page-locked, on transparent huge pages where granted)",
        "steps": args.steps, "seconds": e2e["seconds"], "gpu_launches": e2e["launches"],
        "sweeps_ms_per_step_median": e2e["sweeps_ms_median"],
        "host_link": e2e["link"], "bound_value": e2e["bound_value"],
        "frac_of_bound": e2e["value"] / e2e["bound_value"],
        # untimed, before the timed batches: the buffers back on huge pages,
        # then the host's memory compaction idle
        "host_huge_page_wait": e2e["huge_page_wait"],
        "host_compaction_settle": e2e["compaction_settle"]}
    line["e2e_serial"] = None if e2e is None else {
        "value": e2e["serial_value"], "unit": UNIT, "steps": e2e["serial_steps"],
        "api": "pk_set_field + pk_run_sweeps + pk_get_field per step"}
    print(json.dumps(line), flush=True)


def result_line(args, w, world, value, ms_per_step, us_per_sweep, dev_us, run_info, host_s, clk):
    """Rank 0's JSON line without the end-to-end leg, with the CPU baseline
    and the extras (both measured here)."""
    from iterative_stencil_solver_gb300 import pk
    nx, ny, sweeps = w["nx"], w["ny"], w["sweeps"]
    cells = nx * ny
    peak, peak_kind = measured_peaks()
    launch_us = statistics.median(dev_us)
    alg_bytes = algorithmic_bytes(run_info, cells, run_info["sweeps_done"], w["f"] is not None,
                                  w["tol"], w["check_every"])
    achieved = alg_bytes / (launch_us * 1e-6) / 1e9
    traffic = (TRAFFIC["bytes_per_launch"]
               if TRAFFIC["kernel_sha"] == kernel_source_sha()
               and run_info["stream_config"] == TRAFFIC["stream_config"]
               and args.workload == DEFAULT_WORKLOAD else None)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": args.workload, "nx": nx, "ny": ny, "sweeps_per_step": sweeps,
                   "variant": {1: "direct", 2: "stream", 3: "local"}[run_info["variant"]],
                   "stream_config": run_info["stream_config"],
                   "pass_order": "pass counters" if run_info["pass_counters"] else "grid barrier",
                   "grid": run_info["grid"], "l2": "inputs larger than L2 (2 x field > 129 MB)"
                   if 2 * 4 * cells > 129e6 else "L2-resident",
                   "parallelism": "replicas" if world > 1 else "single-gpu"},
        "us_per_sweep": us_per_sweep,
        "hbm_gbs_algorithmic": achieved,
        "host_s": host_s,
        "gpu_launches": args.steps,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "peak_source": peak_kind,
                     "kernel": shape_label(run_info, w["f"] is not None),
                     "algorithmic_bytes_per_launch": alg_bytes},
        "clocks": clk,
    }
    if not args.no_cpu_baseline:
        v, desc, dt = oracle_sample(w, target_s=10.0, max_rows=min(ny, 2048))
        line["cpu_baseline"] = {"value": v, "unit": UNIT, "cores": 1, "kind": "oracle",
                                "sample": desc, "seconds": dt}
        # context: the same oracle with its OpenMP split of the row loop on
        # every host core (bit-identical per cell)
        import oracle
        ncpu = os.cpu_count() or 1
        if oracle.has_openmp() and ncpu > 1:
            va, desca, dta = oracle_sample(w, target_s=3.0, max_rows=min(ny, 2048), threads=ncpu)
            line["cpu_baseline"]["all_cores"] = {"value": va, "cores": ncpu, "sample": desca,
                                                 "seconds": dta}
    if not args.no_extras:
        line["extras"] = latency_extras(pk)
    return line


if __name__ == "__main__":
    main()
