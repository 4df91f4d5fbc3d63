#!/usr/bin/env python
"""Benchmark of the GB300 warp-level SIMT PTX interpreter.

Metric: simulated thread-instructions per second (sum over issued simulated
instructions of the active lanes, divided by device time). One step is one
pass of the whole hot path over the FFMA latency-probe pair (grid 132 x
block 128, 4096 outer iterations of 32 fma.rn.f32, one dependent-chain
kernel and one with 8 rotating accumulators), i.e. two interpreter launches.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload ffma_pair|vector_add|gather_sS|divergent_kK|fuzz|smem_reduce]
                  [--cache [--cache-cap C] [--cache-form auto|replay|reinterpret]]
                  [--sched [--sched-sms S]]

--cache runs every launch with the L1/L2 hit model (ks_simulate_cached: a
logging pass, the sorted levels, then either a value-free replay of each
warp's issued runs or a checked second interpretation: the replay for large
grids by default, the second interpretation for small grids, kernels with
shared memory and --cache-form reinterpret); --sched with the
SM-level issue model (ks_simulate_sched: the interpreter logging each warp's
issued runs, then one replay warp per simulated SM).

The default run (headline workload, one GPU) also measures every benchmark
configuration at its stated size on its own and adds them to the line as
"per_config": vector_add, the FFMA pair, the strided gather at s = 1, 8, 32
(roofline against HBM), the divergent workload at k = 2, 4, 32, the 64 fuzz
kernels and the shared-memory reduction, each with the median, minimum and
mean over --config-reps timed repetitions (L2 flushed before each) and the
oracle's rate on all host cores and on one core.

Prints one JSON line (rank 0). N > 1 runs N independent replicas, one per
GPU (weak scaling; the path has no exchange step).
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

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = "simulated thread-instructions/sec"
UNIT = "thread-inst/s"
KERNEL_SRC = [os.path.join(ROOT, "simt_ptx_interpretation_gb300", "csrc", f)
              for f in ("ks_interp_kernel.cuh", "ks_interp.cu", "ks_batch.cu", "ks_interp_split.cu", "ks_decode.cpp",
                        "ks_internal.h")]
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")
NCU_FILE = os.path.join(ROOT, "profiles", "ncu_full_size.json")
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK_SM_MHZ = 2070.0


# The configurations measured by the per-configuration suite: every benchmark
# configuration at its stated size (vector_add; the FFMA probe pair; the
# strided gather at s = 1, 8, 32; the divergent workload at k = 2, 4, 32; the
# 64 fuzz kernels) and the shared-memory reduction.
SUITE = ("vector_add", "ffma_pair", "gather_s1", "gather_s8", "gather_s32", "divergent_k2", "divergent_k4",
         "divergent_k32", "fuzz", "smem_reduce")


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default="ffma_pair")
    p.add_argument("--e2e-steps", type=int, default=5)
    p.add_argument("--no-e2e", action="store_true", help="skip the end-to-end leg (profiling runs)")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--iters", type=int, default=4096, help="FFMA outer iterations (smaller cases for profiling)")
    p.add_argument("--cache", action="store_true", help="simulate with the L1/L2 hit model")
    p.add_argument("--cache-cap", type=int, default=0,
                   help="logged global accesses per warp (--cache); 0: the largest count of a plain run, "
                        "rounded up to a power of two")
    p.add_argument("--cache-form", choices=["auto", "replay", "reinterpret"], default="auto",
                   help="second half of the hit model (--cache): replay the logged runs (kernels without shared "
                        "memory; the run log is sized from an untimed logging run) or interpret again; auto: "
                        "replay when every launch of the step has at least 32 simulated warps per SM (the replay "
                        "walks a warp's log with one thread, so a small grid leaves it few real warps)")
    p.add_argument("--layout", choices=["auto", "pair", "split"], default="auto",
                   help="register-file layout of every launch (auto: the library's choice per kernel)")
    p.add_argument("--sched", action="store_true", help="simulate with the SM-level issue model")
    p.add_argument("--sched-sms", type=int, default=152, help="simulated SMs (--sched)")
    p.add_argument("--streams", type=int, default=0,
                   help="CUDA streams the step's independent calls are spread over (0: one per launch, at most 8, "
                        "with --sched; else 1)")
    p.add_argument("--no-batch", action="store_true",
                   help="one ks_simulate per launch instead of one ks_simulate_batch per step")
    p.add_argument("--scale", type=int, default=1,
                   help="divide the gather outputs, divergent threads or fuzz kernels (smaller cases for profiling)")
    p.add_argument("--no-per-config", action="store_true",
                   help="skip the per-configuration suite that the default run adds to its line")
    p.add_argument("--config-reps", type=int, default=50, help="timed repetitions per configuration (suite)")
    p.add_argument("--config-warmup", type=int, default=3, help="warm-up repetitions per configuration (suite)")
    p.add_argument("--configs", default=",".join(SUITE),
                   help="comma-separated configurations of the suite (default: all)")
    return p.parse_args()


def workloads(name: str, iters: int = 4096, scale: int = 1):
    from simt_ptx_interpretation_gb300 import workloads as wl
    if scale < 1 or scale & (scale - 1):
        raise SystemExit("--scale must be a power of two")
    if name == "ffma_pair":
        return [wl.ffma(acc=1, iters=iters), wl.ffma(acc=8, iters=iters)], {
            "workload": "ffma_probe_pair", "grid": 132, "block": 128, "iters": iters, "fma_per_iter": 32,
            "accumulators": [1, 8], "seed": 2}
    if name == "vector_add":
        return [wl.vector_add()], {"workload": "vector_add", "n": 4000, "grid": 16, "block": 256, "seed": 0}
    if name.startswith("gather_s"):
        s = int(name[len("gather_s"):])
        n_out = max(256, (1 << 24) // scale)
        return [wl.gather(s, n_out=n_out)], {"workload": name, "n_out": n_out, "stride": s, "block": 256, "seed": 1}
    if name.startswith("divergent_k"):
        k = int(name[len("divergent_k"):])
        n = max(128, (1 << 20) // scale)
        return [wl.divergent(k, n=n)], {"workload": name, "threads": n, "block": 128, "k": k, "seed": 3}
    if name == "smem_reduce":
        n = max(256, (1 << 22) // scale)
        return [wl.smem_reduce(n=n, block=256)], {"workload": "smem_reduce", "n": n, "block": 256, "seed": 5}
    if name == "fuzz":
        nk = max(1, 64 // scale)
        return [wl.fuzz(i) for i in range(nk)], {"workload": "fuzz64" if nk == 64 else f"fuzz{nk}", "grid": 1024,
                                                 "block": 256, "kernels": nk, "seed": "1000+i, data 4"}
    raise SystemExit(f"unknown workload {name}")


def dist_init():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        import torch
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend=backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu: int):
        self.gpu = gpu
        self.proc = None
        self.path = None

    def __enter__(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (FileNotFoundError, OSError):
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if not self.path or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        os.unlink(self.path)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


def kernel_sha() -> str:
    """Hash of the interpreter kernel's sources (the kernel and its launchers)."""
    h = hashlib.sha256()
    for f in KERNEL_SRC:
        h.update(open(f, "rb").read())
    return h.hexdigest()[:16]


def traffic_for(workload: str):
    """DRAM bytes per launch from the committed ncu capture, if it was taken
    on the current kernel source; else None."""
    try:
        t = json.load(open(TRAFFIC_FILE))
    except (OSError, ValueError):
        return None
    if t.get("kernel_sha") != kernel_sha():
        return None
    return t.get("workloads", {}).get(workload)


def ncu_figures(workload: str):
    """Per-launch ncu figures of a full-size workload (DRAM bytes, issue and
    warp activity) from the committed capture, if it was taken on the current
    kernel source; else None."""
    try:
        t = json.load(open(NCU_FILE))
    except (OSError, ValueError):
        return None
    if t.get("kernel_sha") != kernel_sha():
        return None
    return t.get("workloads", {}).get(workload)


def sm_peak_mhz():
    try:
        return float(json.load(open(PEAKS_FILE)).get("sm_max_mhz", FALLBACK_SM_MHZ)), "measured"
    except (OSError, ValueError):
        return FALLBACK_SM_MHZ, "fallback"


# ---------------------------------------------------------------- ours ----

def most_runs(jobs, n_sm, dev, stream) -> int:
    """The largest count of issued runs of any warp of the jobs, from one
    untimed logging run of each (the SM model's issue log, whose runs the
    hit model's replay form logs too), rounded up to a power of two."""
    import simt_ptx_interpretation_gb300 as ks
    import torch
    runs = 1
    for j in jobs:
        w = j["w"]
        probe = ks.SchedConfig(n_sm=n_sm, max_runs_per_warp=1 << 16)
        tmp = torch.empty(ks.sched_workspace_bytes(w.grid, w.block, probe), dtype=torch.uint8, device=dev)
        sw = torch.empty(w.warps * ks.SCHED_WARP_DTYPE.itemsize, dtype=torch.uint8, device=dev)
        ss = torch.empty(n_sm * 32, dtype=torch.uint8, device=dev)
        ks.simulate_sched(j["mod"], w.kernel, w.grid, w.block, w.params, j["bufs"], j["st"], sw, ss, tmp, j["tr"],
                          j["cfg"], probe, stream)
        torch.cuda.synchronize(dev)
        runs = max(runs, int(tmp[:w.warps * 4].view(torch.int32).max().item()))
        del tmp
    return 1 << (runs - 1).bit_length()


def run_ours(args, world, rank, local):
    import torch
    import simt_ptx_interpretation_gb300 as ks
    from simt_ptx_interpretation_gb300 import _build

    if not _build.up_to_date():
        _build.build_native()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    ws, config = workloads(args.workload, args.iters, args.scale)
    stream = torch.cuda.current_stream(dev)

    # inputs resident in HBM; outputs preallocated
    jobs = []
    for w in ws:
        mod = ks.Module(w.ptx)
        host = [b.data for b in w.fresh_buffers()]
        bufs = [(b.sim_base, torch.from_numpy(h.view(np.uint8)).to(dev)) for b, h in zip(w.buffers, host)]
        cfg = ks.Config(max_ts=w.max_ts, layout=args.layout)
        st = torch.empty(ks.stats_bytes(w.grid, w.block), dtype=torch.uint8, device=dev)
        tr = (torch.empty(ks.trace_bytes(w.grid, w.block, w.max_ts, mod.record_bytes(w.kernel)), dtype=torch.uint8,
                          device=dev) if w.max_ts else None)
        jobs.append(dict(w=w, mod=mod, bufs=bufs, cfg=cfg, st=st, tr=tr))
    if args.layout != "auto":
        config = dict(config, layout=args.layout)
    # The step's launches are independent simulations (own buffers, stats and
    # trace). Plain runs go to the GPU as one batch (ks_simulate_batch: their
    # warps share one real grid). With the SM model, whose calls hold the
    # GPU with a small replay grid, they may be spread over streams forked
    # from and joined to `stream`.
    batch = not (args.cache or args.sched or args.no_batch) and len(jobs) > 1
    cache_batch = None  # the cached batches' items (--cache, several launches a step)
    cache_ws = None  # the workspaces of single cached calls (--cache, --no-batch or one launch a step)
    n_streams = args.streams if args.streams > 0 else (min(len(jobs), 8) if args.sched else 1)
    n_streams = max(1, min(n_streams, len(jobs)))
    streams = [stream] + [torch.cuda.Stream(dev) for _ in range(n_streams - 1)]
    cap = args.cache_cap
    if args.cache and cap <= 0:  # size the log from an untimed plain run
        most = 1
        for j in jobs:
            w = j["w"]
            ks.simulate(j["mod"], w.kernel, w.grid, w.block, w.params, j["bufs"], j["st"], j["tr"], j["cfg"], stream)
            a = ks.stats_array(j["st"])
            most = max(most, int((a["ld_req"] + a["st_req"]).max()))
        cap = 1 << (most - 1).bit_length()
    cache = None
    cache_form = args.cache_form
    if args.cache and cache_form == "auto":
        sms = torch.cuda.get_device_properties(dev).multi_processor_count
        cache_form = "replay" if all(j["w"].warps >= 32 * sms for j in jobs) else "reinterpret"
    if args.cache:
        runs = most_runs(jobs, args.sched_sms, dev, stream) if cache_form == "replay" else 0
        cache = ks.CacheConfig(max_accesses_per_warp=cap, max_runs_per_warp=runs)
    if cache:  # one workspace, sized for the largest grid
        wmax = max(jobs, key=lambda j: j["w"].warps)["w"]
        nbytes = ks.cache_workspace_bytes(wmax.grid, wmax.block, cache)
        if nbytes == 0:
            raise SystemExit("invalid cache configuration")
        # a step of several launches goes as cached batches of at most 16
        # items (their passes share real grids or run side by side, their
        # replays too), each item with a workspace of its own; a single
        # launch as one ks_simulate_cached call
        if not args.no_batch and len(jobs) > 1:
            items = [ks.CachedBatchItem(
                ks.BatchItem(j["mod"], j["w"].kernel, j["w"].grid, j["w"].block, j["w"].params, j["bufs"], j["st"],
                             j["tr"], j["cfg"]), cache,
                torch.empty(ks.cache_workspace_bytes(j["w"].grid, j["w"].block, cache), dtype=torch.uint8,
                            device=dev)) for j in jobs]
            cache_batch = [items[i:i + 16] for i in range(0, len(items), 16)]
        else:
            cache_ws = [torch.empty(nbytes, dtype=torch.uint8, device=dev) for _ in range(n_streams)]
        config = dict(config, cache_model={"l1_lines": cache.l1_lines, "l2_lines": cache.l2_lines,
                                           "lat_l1": cache.lat_l1, "lat_l2": cache.lat_l2,
                                           "max_accesses_per_warp": cache.max_accesses_per_warp,
                                           "form": cache_form + (" (kernels with shared memory or bar.sync: "
                                                                 "reinterpret)" if cache_form == "replay" else ""),
                                           "max_runs_per_warp": cache.max_runs_per_warp})

    sched = ks.SchedConfig(n_sm=args.sched_sms) if args.sched else None
    if sched:
        if cache:
            raise SystemExit("--cache and --sched run separately")
        wmax = max(jobs, key=lambda j: j["w"].warps)["w"]
        sched = ks.SchedConfig(n_sm=args.sched_sms, max_runs_per_warp=most_runs(jobs, args.sched_sms, dev, stream))
        nbytes = ks.sched_workspace_bytes(wmax.grid, wmax.block, sched)
        sched_ws = [torch.empty(nbytes, dtype=torch.uint8, device=dev) for _ in range(n_streams)]
        sched_w = [torch.empty(wmax.warps * ks.SCHED_WARP_DTYPE.itemsize, dtype=torch.uint8, device=dev)
                   for _ in range(n_streams)]
        sched_s = [torch.empty(args.sched_sms * 32, dtype=torch.uint8, device=dev) for _ in range(n_streams)]
        config = dict(config, sm_model={"n_sm": sched.n_sm, "schedulers_per_sm": sched.schedulers_per_sm,
                                        "ctas_per_sm": "fill 32 warps", "max_runs_per_warp": sched.max_runs_per_warp})

    def launch(i):
        j, q = jobs[i], i % n_streams
        w, s = j["w"], streams[q]
        if sched:
            ks.simulate_sched(j["mod"], w.kernel, w.grid, w.block, w.params, j["bufs"], j["st"], sched_w[q],
                              sched_s[q], sched_ws[q], j["tr"], j["cfg"], sched, s)
        elif cache:
            ks.simulate_cached(j["mod"], w.kernel, w.grid, w.block, w.params, j["bufs"], j["st"], cache_ws[q], j["tr"],
                               j["cfg"], cache, s)
        else:
            ks.simulate(j["mod"], w.kernel, w.grid, w.block, w.params, j["bufs"], j["st"], j["tr"], j["cfg"], s)

    def fork():
        if n_streams > 1:
            e = torch.cuda.Event()
            e.record(stream)
            for s in streams[1:]:
                s.wait_event(e)

    def join():
        for s in streams[1:]:
            e = torch.cuda.Event()
            e.record(s)
            stream.wait_event(e)

    batch_launches = [0]  # real kernel launches of the last batch call

    def launch_batch():
        batch_launches[0] = ks.simulate_batch(
            [ks.BatchItem(j["mod"], j["w"].kernel, j["w"].grid, j["w"].block, j["w"].params, j["bufs"], j["st"],
                          j["tr"], j["cfg"]) for j in jobs], stream)

    def launch_cached_batch():
        batch_launches[0] = sum(ks.simulate_cached_batch(c, stream) for c in cache_batch)

    def step(lev=None):
        if cache_batch:
            if lev:
                lev[0][0].record(stream)
            launch_cached_batch()
            if lev:
                lev[0][1].record(stream)
            return
        if batch:
            if lev:
                lev[0][0].record(stream)
            launch_batch()
            if lev:
                lev[0][1].record(stream)
            return
        fork()
        for i in range(len(jobs)):
            if lev:
                lev[i][0].record(streams[i % n_streams])
            launch(i)
            if lev:
                lev[i][1].record(streams[i % n_streams])
        join()

    # work per step (deterministic): one run, reduce totals, check statuses
    step()
    insts, launch_insts = 0, []
    for j in jobs:
        t = ks.read_stats(j["st"], j["w"].warps, stream)
        if t.status != 0:
            raise SystemExit(f"simulation status {t.status} on {j['w'].name}")
        insts += t.thread_insts
        launch_insts.append(t.thread_insts)

    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)  # > 129 MB L2
    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize(dev)

    n_launch = 1 if (batch or cache_batch) else len(jobs)  # timed calls per step
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    lev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_launch)]
           for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize(dev)
    with ClockSampler(local) as clk:
        t_wall0 = time.perf_counter()
        for k in range(args.steps):
            flush.zero_()
            evs[k][0].record(stream)
            step(lev[k])
            evs[k][1].record(stream)
        torch.cuda.synchronize(dev)
        t_wall = time.perf_counter() - t_wall0
    barrier(world)
    step_ms = [evs[k][0].elapsed_time(evs[k][1]) for k in range(args.steps)]
    launch_ms = [[lev[k][i][0].elapsed_time(lev[k][i][1]) for k in range(args.steps)] for i in range(n_launch)]
    dev_s = sum(step_ms) / 1e3
    dev_s = max_over_ranks(dev_s, world)
    value = insts * args.steps * world / dev_s
    clocks = clk.summary()

    # roofline of the interpreter kernel (every launch is ks_interp_kernel)
    mhz, peak_src = sm_peak_mhz()
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    peak = sms * 4 * 32 * mhz * 1e6 / 1e9  # G thread-inst/s: 4 warp-issues per SM per clock, 32 lanes
    # Every kernel of a step is a ks_interp_kernel launch (plus, with the
    # models, their own kernels): the launches of one step may run
    # concurrently, so the roofline takes the step's algorithmic units over
    # the span from the first launch's start to the last one's end (the
    # step's events; nothing else runs inside them).
    span_s = sum(step_ms) / args.steps / 1e3
    # with the cache model a call interprets the launch twice (and sorts in
    # between): charge the whole call to the two interpreter passes
    # (the replay form and the SM model interpret once per call)
    passes = 2 if cache and not cache.max_runs_per_warp else 1
    achieved = passes * insts / span_s / 1e9
    # the stored counters are for the full-size workloads only
    traffic = traffic_for(config["workload"]) if args.scale == 1 and args.iters == 4096 else None
    roofline = {"bound": "alu", "achieved": round(achieved, 3), "peak": round(peak, 1), "unit": "Gthread-inst/s",
                "frac": round(achieved / peak, 5), "traffic": traffic,
                "measure": "simulated thread-instructions per second against the GPU's issue peak in "
                           "thread-instructions (1.0 would be one simulated instruction per real issue slot)",
                "peak_source": f"{sms} SMs x 4 issue/clk x 32 lanes x {mhz:.0f} MHz ({peak_src})",
                "algorithmic_units_per_launch": [int(x) for x in launch_insts],
                "launch_ms_mean": [round(sum(x) / len(x), 4) for x in launch_ms],
                "streams": n_streams, "batched": bool(batch or cache_batch),
                "timed_over": "each step's span (its launches may overlap)"}
    ncu = ncu_figures(config["workload"]) if args.scale == 1 and args.iters == 4096 and not (cache or sched) else None
    if ncu:  # the interpreter's own instruction stream on this kernel source, per ncu
        roofline["ncu"] = {k: v for k, v in ncu.items() if k != "dram_bytes"}
        roofline["ncu"]["measure"] = ("sm__inst_issued.avg.pct_of_peak_sustained_active: the share of the SMs' issue "
                                      "slots the interpreter's own instructions use")
    if cache and cache.max_runs_per_warp:
        roofline["note"] = ("each call runs ks_interp_kernel once (logging accesses and issued runs), the level "
                            "kernels and radix sorts, then cache_replay_kernel; achieved counts the simulated "
                            "thread-instructions over the whole call's time")
    elif cache:
        roofline["note"] = ("each call runs ks_interp_kernel twice plus the level kernels and radix sorts; "
                            "achieved counts both passes over the whole call's time")
    if sched:
        roofline["note"] = ("each call runs ks_interp_kernel once and ks_sched_kernel once; achieved counts the "
                            "simulated thread-instructions over the whole call's time")

    # end to end through the public API with pinned host buffers
    e2e = None if args.no_e2e else run_e2e(args, jobs, insts, dev, streams, launch, fork, join,
                                           launch_batch if batch else
                                           launch_cached_batch if cache_batch
                                           else None)

    line = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(sum(step_ms) / len(step_ms), 4),
        "ms_per_step_median": round(statistics.median(step_ms), 4), "ms_per_step_min": round(min(step_ms), 4),
        "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32+u32/u64 (simulated)", "data": "synthetic (seeded)",
        "config": dict(config, l2="flushed between steps (256 MiB write)", parallelism=f"replicas{world}",
                       streams=n_streams, batched=bool(batch or cache_batch)),
        # our kernels per call: the interpreter, or (cache model) the four level
        # kernels between either two interpreter passes or one pass and the
        # replay (the radix sorts and the scan are library code)
        "roofline": roofline, "e2e": e2e,
        # (a batch call reports its real launches)
        "gpu_launches": args.steps * (batch_launches[0] if (batch or cache_batch)
                                      else n_launch * (6 if cache else 2 if sched else 1)),
        "clocks": clocks,
        "wall_s_timed_region": round(t_wall, 3), "kernel_sha": kernel_sha(),
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = (cpu_baseline_cached(ws, cache) if cache else cpu_baseline_sched(ws, sched) if sched
                                else cpu_baseline(ws, sample_warps=None))
    # the default run (headline workload, plain model, one GPU) adds every
    # configuration measured on its own
    if (world == 1 and not args.no_per_config and args.workload == "ffma_pair" and not (cache or sched)
            and args.scale == 1 and args.iters == 4096):
        torch.cuda.empty_cache()
        line["per_config"] = run_suite(args, dev, stream)
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_e2e(args, jobs, insts, dev, streams, launch, fork, join, launch_batch=None):
    """The same step through the public API from pinned host memory: each
    launch's inputs are copied in, it runs, and its outputs, stats and trace
    are copied out, all on the launch's own stream (a batch: every input in,
    the batch, every output out)."""
    import torch
    pinned_in, pinned_out = [], []
    h2d = d2h = 0
    for j in jobs:
        ins, outs = [], []
        for b, (_, t) in zip(j["w"].buffers, j["bufs"]):
            h = torch.from_numpy(b.data.view(np.uint8)).pin_memory()
            if b.output:
                outs.append((t, torch.empty_like(h).pin_memory()))
                d2h += h.numel()
            else:
                ins.append((h, t))
                h2d += h.numel()
        outs.append((j["st"], torch.empty(j["st"].numel(), dtype=torch.uint8).pin_memory()))
        d2h += j["st"].numel()
        if j["tr"] is not None:
            outs.append((j["tr"], torch.empty(j["tr"].numel(), dtype=torch.uint8).pin_memory()))
            d2h += j["tr"].numel()
        pinned_in.append(ins)
        pinned_out.append(outs)
    times = []
    for k in range(args.e2e_steps):
        torch.cuda.synchronize(dev)
        t0 = time.perf_counter()
        if launch_batch is not None:
            with torch.cuda.stream(streams[0]):
                for ins in pinned_in:
                    for h, t in ins:
                        t.copy_(h, non_blocking=True)
                launch_batch()
                for outs in pinned_out:
                    for t, h in outs:
                        h.copy_(t, non_blocking=True)
            streams[0].synchronize()
            times.append(time.perf_counter() - t0)
            continue
        fork()
        for i, (ins, outs) in enumerate(zip(pinned_in, pinned_out)):
            with torch.cuda.stream(streams[i % len(streams)]):
                for h, t in ins:
                    t.copy_(h, non_blocking=True)
                launch(i)
                for t, h in outs:
                    h.copy_(t, non_blocking=True)
        join()
        streams[0].synchronize()
        times.append(time.perf_counter() - t0)
    mean = sum(times) / len(times)
    return {"value": round(insts / mean, 1), "unit": UNIT, "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(d2h), "steps": args.e2e_steps}


def cpu_baseline(ws, sample_warps=None, max_warps_per_kernel=None, threads=None, buffers=None):
    """The oracle, as it stands, on the host cores over a bounded sample of the
    workload: the first `n` warps of every kernel (whole CTAs for kernels with
    shared memory or barriers, every one of which is counted), on `threads`
    host threads (default: every core). `buffers`: per kernel, buffers to run
    on (default: a fresh copy of the kernel's inputs)."""
    import oracle
    cores = threads or os.cpu_count() or 1
    n = max_warps_per_kernel or 40 * cores
    total_i, total_s, desc = 0, 0.0, []
    for i, w in enumerate(ws):
        warps = list(range(min(n, w.warps)))
        bufs = buffers[i] if buffers is not None else w.fresh_buffers()
        t0 = time.perf_counter()
        r = oracle.run(w.ptx, w.kernel, w.grid, w.block, w.params, [(b.sim_base, b.data) for b in bufs],
                       max_ts=w.max_ts, trace=bool(w.max_ts), warps=warps, threads=cores)
        total_s += time.perf_counter() - t0
        ran = r.stats["warp_insts"] > 0
        total_i += int(r.stats["thread_insts"][ran].sum())
        desc.append(f"{w.name}: warps 0..{int(np.nonzero(ran)[0].max())} of {w.warps}")
    return {"value": round(total_i / total_s, 1), "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": "; ".join(desc), "thread_insts": total_i, "seconds": round(total_s, 3)}


def cpu_baseline_suite(ws, target_s: float = 2.0):
    """The oracle on a bounded sample of one configuration, on every host core
    and on one core: the first n warps of every kernel (of every eighth kernel
    when there are more than eight, so that each call's set-up stays small
    against its warps), n grown from a small probe until a leg takes about
    target_s (or covers every warp). The oracle's stores are idempotent for
    these workloads (no kernel reads what it stores), so the probes share one
    copy of the inputs."""
    cores = os.cpu_count() or 1
    if len(ws) > 8:
        ws = ws[::8]
    bufs = [w.fresh_buffers() for w in ws]
    most = max(w.warps for w in ws)
    legs = {}
    for label, threads in (("all_cores", cores), ("one_core", 1)):
        n = min(most, 2 * threads)
        r = cpu_baseline(ws, max_warps_per_kernel=n, threads=threads, buffers=bufs)
        while r["seconds"] < target_s / 3 and n < most:
            n = min(most, max(n + 1, int(n * min(64.0, target_s / max(r["seconds"], 1e-4)))))
            r = cpu_baseline(ws, max_warps_per_kernel=n, threads=threads, buffers=bufs)
        legs[label] = r
    a, o = legs["all_cores"], legs["one_core"]
    return {"value": a["value"], "unit": UNIT, "cores": cores, "kind": "oracle", "sample": a["sample"],
            "thread_insts": a["thread_insts"], "seconds": a["seconds"],
            "one_core": {"value": o["value"], "cores": 1, "sample": o["sample"], "thread_insts": o["thread_insts"],
                         "seconds": o["seconds"]}}


def hbm_peak():
    try:
        return float(json.load(open(PEAKS_FILE))["hbm_gbs"]), "measured"
    except (OSError, ValueError, KeyError):
        return 6800.0, "fallback"


def gather_bytes(w, s: int) -> int:
    """Algorithmic DRAM bytes of one strided-gather launch: per warp, min(32,
    4s) sectors of 32 bytes read (sector-granular), one 128-byte store and its
    96-byte statistics record."""
    return w.warps * (min(32, 4 * s) * 32 + 128 + 96)


def issue_peak(dev):
    """G thread-inst/s the GPU issues at most: SMs x 4 warp-instructions per
    clock x 32 lanes x the measured maximum SM clock."""
    import torch
    mhz, src = sm_peak_mhz()
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    return sms * 4 * 32 * mhz * 1e6 / 1e9, f"{sms} SMs x 4 issue/clk x 32 lanes x {mhz:.0f} MHz ({src})"


def measure_config(name: str, reps: int, warmup: int, dev, stream, flush, cpu: bool = True):
    """One configuration at its stated size: plain simulations (one
    ks_simulate_batch call when it has several launches), `warmup` untimed
    repetitions, then `reps` timed ones with the L2 flushed before each,
    CUDA events on the launching stream around each; median, minimum and
    mean, the roofline of the interpreter launch and the oracle's rate."""
    import torch
    import simt_ptx_interpretation_gb300 as ks
    ws, config = workloads(name)
    jobs = []
    for w in ws:
        mod = ks.Module(w.ptx)
        bufs = [(b.sim_base, torch.from_numpy(b.data.view(np.uint8)).to(dev)) for b in w.buffers]
        cfg = ks.Config(max_ts=w.max_ts)
        st = torch.empty(ks.stats_bytes(w.grid, w.block), dtype=torch.uint8, device=dev)
        tr = (torch.empty(ks.trace_bytes(w.grid, w.block, w.max_ts, mod.record_bytes(w.kernel)), dtype=torch.uint8,
                          device=dev) if w.max_ts else None)
        jobs.append((w, mod, bufs, cfg, st, tr))
    items = [ks.BatchItem(mod, w.kernel, w.grid, w.block, w.params, bufs, st, tr, cfg)
             for (w, mod, bufs, cfg, st, tr) in jobs]
    launched = [0]

    def step():
        if len(items) > 1:
            launched[0] = ks.simulate_batch(items, stream)
        else:
            w, mod, bufs, cfg, st, tr = jobs[0]
            ks.simulate(mod, w.kernel, w.grid, w.block, w.params, bufs, st, tr, cfg, stream)
            launched[0] = 1

    step()
    insts = 0
    for (w, mod, bufs, cfg, st, tr) in jobs:
        t = ks.read_stats(st, w.warps, stream)
        if t.status != 0:
            raise SystemExit(f"simulation status {t.status} on {w.name}")
        insts += t.thread_insts
    for _ in range(warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize(dev)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
    with ClockSampler(dev.index or 0) as clk:
        for k in range(reps):
            flush.zero_()
            evs[k][0].record(stream)
            step()
            evs[k][1].record(stream)
        torch.cuda.synchronize(dev)
    ms = [a.elapsed_time(b) for a, b in evs]
    med, mn, mean = statistics.median(ms), min(ms), sum(ms) / len(ms)
    entry = {"config": config, "reps": reps, "warmup": warmup, "ms_median": round(med, 5), "ms_min": round(mn, 5),
             "ms_mean": round(mean, 5), "value": round(insts / (med / 1e3), 1),
             "value_at_min": round(insts / (mn / 1e3), 1), "unit": UNIT, "thread_insts_per_step": int(insts),
             "gpu_launches_per_step": launched[0], "l2": "flushed before each repetition (256 MiB write)",
             "clocks": clk.summary()}
    ncu = ncu_figures(config["workload"])
    traffic = ncu["dram_bytes"] if ncu else traffic_for(config["workload"])
    if name.startswith("gather_s"):
        s_ = int(name[len("gather_s"):])
        nbytes = gather_bytes(ws[0], s_)
        hbm, src = hbm_peak()
        achieved = nbytes / (med / 1e3) / 1e9
        entry["roofline"] = {"bound": "hbm", "achieved": round(achieved, 2), "peak": hbm, "unit": "GB/s",
                             "frac": round(achieved / hbm, 5), "traffic": traffic,
                             "algorithmic_bytes_per_launch": int(nbytes),
                             "peak_source": f"copy bandwidth, MEASURED_PEAKS.json ({src})",
                             "timed_over": "the median launch"}
        if traffic:  # what the GPU actually moved (whole lines when the stride leaves sectors unused)
            dram = traffic / (med / 1e3) / 1e9
            entry["roofline"].update(dram_gbs=round(dram, 2), dram_frac=round(dram / hbm, 5))
    else:
        peak, src = issue_peak(dev)
        achieved = insts / (med / 1e3) / 1e9
        entry["roofline"] = {"bound": "alu", "achieved": round(achieved, 3), "peak": round(peak, 1),
                             "unit": "Gthread-inst/s", "frac": round(achieved / peak, 5), "traffic": traffic,
                             "measure": "simulated thread-instructions per second against the GPU's issue peak "
                                        "in thread-instructions (1.0 would be one simulated instruction per real "
                                        "issue slot)",
                             "peak_source": src, "timed_over": "the median step"}
    if ncu:  # the interpreter's own instruction stream, per ncu on this kernel source
        entry["roofline"]["ncu"] = {k: v for k, v in ncu.items() if k != "dram_bytes"}
    if cpu:
        entry["cpu_baseline"] = cpu_baseline_suite(ws)
    del jobs, items
    return entry


def run_suite(args, dev, stream):
    """Every configuration of SUITE (or --configs) measured in turn."""
    import torch
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)  # > 129 MB L2
    out = {}
    for name in [c for c in args.configs.split(",") if c]:
        out[name] = measure_config(name, args.config_reps, args.config_warmup, dev, stream, flush,
                                   cpu=not args.no_cpu_baseline)
        torch.cuda.empty_cache()
    return out


def cpu_baseline_cached(ws, cache, warps_per_kernel=16):
    """The oracle's cache-model stepper (one host thread: the caches are
    global state) on a bounded sample: each kernel on a grid cut down to about
    `warps_per_kernel` warps."""
    import oracle
    total_i, total_s, desc = 0, 0.0, []
    for w in ws:
        wpc = (w.block + 31) // 32
        grid = max(1, min(w.grid, warps_per_kernel // wpc))
        bufs = w.fresh_buffers()
        t0 = time.perf_counter()
        r = oracle.run_cached(w.ptx, w.kernel, grid, w.block, w.params, [(b.sim_base, b.data) for b in bufs],
                              max_ts=w.max_ts, trace=bool(w.max_ts), l1_lines=cache.l1_lines,
                              l2_lines=cache.l2_lines, lat_l1=cache.lat_l1, lat_l2=cache.lat_l2, log_cap=1)
        total_s += time.perf_counter() - t0
        total_i += int(r.stats["thread_insts"].sum())
        desc.append(f"{w.name}: grid {grid} of {w.grid}")
    return {"value": round(total_i / total_s, 1), "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": "; ".join(desc), "thread_insts": total_i, "seconds": round(total_s, 3)}


def cpu_baseline_sched(ws, sched, warps_per_kernel=16):
    """The oracle's cycle-by-cycle SM model (one host thread) on a bounded
    sample: each kernel on a grid cut down to about `warps_per_kernel` warps,
    on as many SMs as it has CTAs."""
    import oracle
    total_i, total_s, desc = 0, 0.0, []
    for w in ws:
        wpc = (w.block + 31) // 32
        grid = max(1, min(w.grid, warps_per_kernel // wpc))
        bufs = w.fresh_buffers()
        t0 = time.perf_counter()
        st = np.zeros(grid * wpc, dtype=oracle.STATS_DTYPE)
        oracle.run_sched(w.ptx, w.kernel, grid, w.block, w.params, [(b.sim_base, b.data) for b in bufs],
                         n_sm=min(grid, sched.n_sm), schedulers=sched.schedulers_per_sm, stats=st)
        total_s += time.perf_counter() - t0
        total_i += int(st["thread_insts"].sum())
        desc.append(f"{w.name}: grid {grid} of {w.grid}")
    return {"value": round(total_i / total_s, 1), "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": "; ".join(desc), "thread_insts": total_i, "seconds": round(total_s, 3)}


# ----------------------------------------------------------- reference ----

def run_reference(args, world, rank):
    if rank != 0:
        return
    ws, config = workloads(args.workload, args.iters, args.scale)
    cores = os.cpu_count() or 1
    per = max(4, min(64, 2 * cores))
    if args.cache:
        from simt_ptx_interpretation_gb300.api import CacheConfig
        cache = CacheConfig(max_accesses_per_warp=args.cache_cap)
        per = 8
        config = dict(config, cache_model={"l1_lines": cache.l1_lines, "l2_lines": cache.l2_lines,
                                           "lat_l1": cache.lat_l1, "lat_l2": cache.lat_l2})
        cores = 1

        def sample(n):
            return cpu_baseline_cached(ws, cache, warps_per_kernel=n)
    elif args.sched:
        from simt_ptx_interpretation_gb300.api import SchedConfig
        sc = SchedConfig(n_sm=args.sched_sms)
        per = 8
        config = dict(config, sm_model={"n_sm": sc.n_sm, "schedulers_per_sm": sc.schedulers_per_sm})
        cores = 1

        def sample(n):
            return cpu_baseline_sched(ws, sc, warps_per_kernel=n)
    else:
        def sample(n):
            return cpu_baseline(ws, max_warps_per_kernel=n)
    for _ in range(args.warmup):
        sample(4)
    times, insts = [], 0
    for _ in range(args.steps):
        t0 = time.perf_counter()
        b = sample(per)
        times.append(time.perf_counter() - t0)
        insts = b["thread_insts"]
    value = insts * len(times) / sum(times)
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * sum(times) / len(times), 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32+u32/u64 (simulated)",
        "data": "synthetic (seeded)", "config": dict(config, sample_warps_per_kernel=per),
        "cpu_baseline": {"value": round(value, 1), "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": (f"each kernel on a grid of about {per} warps per step"
                                    if args.cache or args.sched else f"first {per} warps of each kernel per step")},
        "e2e": {"value": round(value, 1), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    world, rank, local = dist_init()
    try:
        if args.impl == "reference":
            run_reference(args, world, rank)
        else:
            run_ours(args, world, rank, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
