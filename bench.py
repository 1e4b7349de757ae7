"""Benchmark of the all-reduce fusion epilogue on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl arf|reference]
                    [--workload NAME] [--sweep-out FILE]

One step = one pass of the whole hot path over one batch: a kAllReduce call
and a kARResidualRMSNorm call on the workload's partials. The default
workload is the largest one-GPU configuration, the 80 MiB-per-partial TP4
payload (W=4, M=5851, H=7168, bf16). The L2 is flushed before every step,
outside the timed events: a write of twice its size, then a read of another
buffer of twice its size. The read evicts the flush's own dirty lines, so
their write-back to HBM is not charged to the timed kernels.
Metric: achieved HBM GB/s = algorithmic bytes / device time, where the
algorithmic bytes read every partial and the residual once, gamma once and
write each output once. Rank 0 prints one JSON line, the last line of
standard output. --sweep-out writes the per-configuration table (every
workload, pattern and K3 row count) to a JSON file instead.

N > 1 (torchrun, one process per GPU): every rank runs its own replica of the
workload (the path has no exchange step on one GPU); value = bytes of all
ranks / the slowest rank's time.

--impl reference times the CPU oracle (single-threaded C) on the host cores,
on a bounded sample of the same workload, for the same metric.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "µs/call and achieved HBM GB/s (% of GB300 roofline) vs M, per W and pattern"
FALLBACK_HBM_GBS = 6800.0
PATTERNS = ("allreduce", "rmsnorm")
# the kARResidualRMSNorm kernel of each plan path (arf_path_t order)
KERNEL_OF_PATH = {0: "ar_flat_kernel", 1: "rms_kernel", 2: "rms_kernel", 3: "rms_async_kernel", 4: "rms_elem_kernel",
                  5: "rms_bulk_kernel"}
AR_KERNEL_OF_PATH = {0: "ar_flat_kernel", 4: "ar_elem_kernel", 5: "rms_bulk_kernel"}
CSRC = os.path.join(ROOT, "all_reduce_residual_gb300", "csrc")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=("arf", "reference"), default="arf")
    ap.add_argument("--workload", default="tp4_80mib")
    ap.add_argument("--sweep-out", default=None,
                    help="also time every workload, pattern and K3 row count and write the table to this JSON file")
    ap.add_argument("--no-sweep", action="store_true",
                    help="accepted for older command lines; the sweep runs only with --sweep-out")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU-oracle baseline leg")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the cold per-call fractions of the other configurations of 8 MiB and more")
    ap.add_argument("--m", type=int, default=None, help="override the workload's row count M (for profiling)")
    ap.add_argument("--pattern", choices=PATTERNS, default=None,
                    help="time only this pattern of the workload (for profiling one kernel)")
    ap.add_argument("--plan", default=None,
                    help="explicit launch plan path,threads,vpt,cluster,grid,w_spec,stages for the step's calls "
                         "(arf_plan_check rules; for profiling a kernel shape the planner does not pick)")
    return ap.parse_args()


# ---------------------------------------------------------------------------
# distributed plumbing (replicas only)
# ---------------------------------------------------------------------------


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return rank, world, local


def init_dist(world: int, backend: str):
    import torch.distributed as dist

    if world > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend)


def barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def aggregate(units: float, seconds: float, world: int):
    """(total units over ranks, slowest rank's seconds). Replicas: each rank
    contributes its own units; the job takes as long as its slowest rank."""
    if world == 1:
        return units, seconds
    import torch
    import torch.distributed as dist

    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    u = torch.tensor([units], dtype=torch.float64, device=dev)
    t = torch.tensor([seconds], dtype=torch.float64, device=dev)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(u.item()), float(t.item())


# ---------------------------------------------------------------------------
# measurement helpers
# ---------------------------------------------------------------------------


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def source_digests(kernel: str) -> dict:
    """SHA-256 of each source file that defines `kernel`."""
    files = ["arf_kernels.cuh"] + (["arf_bulk.cuh"] if kernel == "rms_bulk_kernel" else []) + \
        (["arf_elem.cuh"] if kernel.endswith("_elem_kernel") else [])
    return {f: hashlib.sha256(open(os.path.join(CSRC, f), "rb").read()).hexdigest() for f in files}


def recorded_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel source (else None)."""
    try:
        with open(TRAFFIC_FILE) as f:
            rec = json.load(f)
        e = rec.get(f"{kernel}/{workload}")
        if e and e.get("kernel_sources_sha256") == source_digests(kernel):
            return int(e["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 200 ms."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
                self.lines = [ln for ln in out.splitlines() if ln.strip()]
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ln in getattr(self, "lines", []):
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 8:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


class L2Flush:
    """Leaves the L2 holding none of the benchmark's data: write `nbytes`
    (twice the L2), then read another `nbytes` so that the L2 ends up full
    of clean lines (no write-back pending when the timed kernels start).
    zero_(dirty_only=True) skips the read: the plain write flush.

    It ends with a spin of a random 0-4095 SM cycles (under 2 us, touching
    no memory). The GPU's event clock advances in steps of about 2 us and
    the flush takes a fixed time, so without it the timed call would start at
    nearly the same phase of that clock every time and the mean of many
    timings would carry up to a step of bias; with it the phase is random
    and the mean is unbiased."""

    def __init__(self, nbytes, dev, seed=12345):
        import random

        import torch

        self.w = torch.empty(nbytes, dtype=torch.uint8, device=dev)
        self.r = torch.zeros(nbytes // 4, dtype=torch.int32, device=dev)
        self.nbytes = nbytes
        self.rng = random.Random(seed)

    def zero_(self, dirty_only=False):
        import torch

        self.w.zero_()
        if not dirty_only:
            self.sink = torch.amax(self.r)  # one read pass, no temporary
        torch.cuda._sleep(self.rng.randrange(4096))

    def describe(self):
        mib = self.nbytes >> 20
        return f"flush before each step: write {mib} MiB, read another {mib} MiB, random 0-2 us spin"


# ---------------------------------------------------------------------------
# the GPU arm
# ---------------------------------------------------------------------------


def run_arf(args):
    import torch

    import all_reduce_residual_gb300 as arf
    from all_reduce_residual_gb300 import build as arf_build
    from all_reduce_residual_gb300 import workloads as wl

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    init_dist(world, "nccl")
    arf_build.build()
    ws = arf.Workspace(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream(dev)
    w = {**wl.WORKLOADS, **wl.EXTRA_WORKLOADS}[args.workload]
    if args.m is not None:
        w = w.with_m(args.m)
    pats = [p for p in PATTERNS if p in w.patterns and (args.pattern is None or p == args.pattern)]
    inp = wl.make_inputs(w)
    P = [p.to(dev) for p in inp.partials]
    R, G = inp.residual.to(dev), inp.gamma.to(dev)
    plan = None
    if args.plan:
        f = [int(x) for x in args.plan.split(",")]
        plan = arf.Plan(path=f[0], threads=f[1], vpt=f[2], cluster=f[3], grid=f[4], w_spec=f[5],
                        stages=f[6] if len(f) > 6 else 0)
    ptrs = arf.pointer_array(P, dev)
    outs = {p: torch.empty_like(R) for p in pats}
    ro = torch.empty_like(R)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = L2Flush(max(2 * l2, 256 << 20), dev)
    bytes_call = {p: w.bytes_per_call(p) for p in pats}
    step_bytes = sum(bytes_call.values())

    def call(p):
        arf.run(ws, p, P, R, G, w.eps, out=outs[p], residual_out=ro if p == "rmsnorm" else None, ptrs=ptrs,
                plan=plan)

    def step():
        flush.zero_()
        for p in pats:
            call(p)

    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(pats) + 1)] for _ in range(K)]
    with ClockSampler(local) as clk:
        for _ in range(args.warmup):
            step()
        torch.cuda.synchronize()
        barrier(world)
        torch.cuda.synchronize()
        t_timed = time.perf_counter()
        for k in range(K):
            flush.zero_()
            ev[k][0].record(stream)
            for i, p in enumerate(pats):
                call(p)
                ev[k][i + 1].record(stream)
        torch.cuda.synchronize()
        barrier(world)
        t_timed = time.perf_counter() - t_timed
        # nvidia-smi samples every 200 ms: a timed region shorter than a
        # second is followed by untimed repetitions of the same step, so that
        # the clock record holds samples taken under this load
        t_extra = time.perf_counter()
        while t_timed + (time.perf_counter() - t_extra) < 1.0:
            for _ in range(20):
                step()
            torch.cuda.synchronize()
    per_call = {p: [ev[k][i].elapsed_time(ev[k][i + 1]) for k in range(K)] for i, p in enumerate(pats)}
    step_ms = [ev[k][0].elapsed_time(ev[k][-1]) for k in range(K)]
    total_s = sum(step_ms) / 1e3
    units, slowest = aggregate(step_bytes * K, total_s, world)
    value = units / slowest / 1e9

    peak, peak_src = measured_peak()
    dom = "rmsnorm" if "rmsnorm" in pats else pats[0]
    dom_s = statistics.mean(per_call[dom]) / 1e3
    achieved = bytes_call[dom] / dom_s / 1e9
    dt_torch = torch.bfloat16 if w.dtype == "bf16" else torch.float16
    plans = {p: (plan if plan is not None else ws.plan(p, w.W, w.M, w.H, dt_torch)) for p in pats}
    kname = (KERNEL_OF_PATH if dom == "rmsnorm" else AR_KERNEL_OF_PATH)[plans[dom].path]
    traffic = recorded_traffic(kname, w.name if args.m is None else None)
    steady_us = steady_state_us(lambda: call(dom), dev, stream)
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4), "traffic": traffic, "kernel": kname,
                "algorithmic_bytes_per_launch": bytes_call[dom],
                "peak_source": f"{peak_src} hbm_gbs (copy)",
                "frac_basis": "cold mean per launch",
                "steady_frac": round(bytes_call[dom] / (steady_us * 1e-6) / 1e9 / peak, 4),
                "steady_us": round(steady_us, 3),
                "steady_basis": "20 back-to-back in a graph",
                "dram_over_algorithmic": round(traffic / bytes_call[dom], 4) if traffic else None}

    result = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(statistics.mean(step_ms), 6), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic: seeded N(0,s) partials, N(0,1) residual, U(0.5,1.5) gamma",
        "config": {"workload": f"{w.name}: W={w.W} M={w.M} H={w.H} {w.dtype}, one {' + one '.join(pats)} call per step",
                   "W": w.W, "M": w.M, "H": w.H, "io_dtype": w.dtype,
                   "bytes_per_step": step_bytes, "l2": flush.describe(), "parallelism": f"replicas x{world}",
                   "plans": {p: plan_str(plans[p]) for p in pats},
                   **({"plan_source": "explicit (--plan)"} if plan is not None else {})},
        "us_per_call": {p: round(statistics.mean(v) * 1e3, 3) for p, v in per_call.items()},
        "frac_per_call": {p: round(bytes_call[p] / (statistics.mean(v) * 1e-3) / 1e9 / peak, 4)
                          for p, v in per_call.items()},
        "roofline": roofline,
        "gpu_launches": len(pats) * K,
        "clocks": {**clk.summary(),
                   "window": "warm-up, timed" + (", padded to 1 s" if t_timed < 1.0 else "")},
    }
    if not args.no_e2e:
        result["e2e"] = e2e_leg(ws, w, inp, pats, flush, dev, K, world)
    result["roofline_context"] = roofline_context(ws, dev, flush, w, dom, per_call[dom])
    if world == 1 and not args.no_configs and args.m is None and plan is None:
        result["frac_other_configs"] = other_configs(ws, dev, flush, peak, skip=w.name)
    if rank == 0 and world == 1 and not args.no_cpu:
        result["cpu_baseline"] = cpu_baseline(w, inp, budget_s=10.0)
    if args.sweep_out and world == 1:  # the scaling runs (N > 1) time the headline only
        rows = sweep(ws, dev, flush, peak)
        with open(args.sweep_out, "w") as f:
            json.dump({"peak_gbs": peak, "peak_source": peak_src, "clocks": result["clocks"], "rows": rows}, f,
                      indent=1)
    if rank == 0:
        print(json.dumps(result, separators=(",", ":")), flush=True)
    ws.close()
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


def plan_str(p) -> str:
    """A launch plan in one short string: path threads x chunks per thread
    (bulk: ring slots), cluster, grid."""
    names = {0: "flat", 1: "row", 2: "cluster", 3: "async", 4: "elem", 5: "bulk"}
    s = f"{names.get(p.path, p.path)} {p.threads}x{p.vpt}"
    if p.cluster > 1:
        s += f" c{p.cluster}"
    if p.stages:
        s += f" s{p.stages}"
    return s + f" g{p.grid} w{p.w_spec}"


def steady_state_us(fn, dev, stream, n=20):
    """Per-call time of fn in a CUDA graph of n back-to-back calls, fastest of
    5 replays: the sustained rate, where each call also pays the write-backs
    the previous one left in L2."""
    import torch

    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream(dev)
    s.wait_stream(stream)
    with torch.cuda.stream(s):
        fn()  # plan made outside the capture
        with torch.cuda.graph(g, stream=s):
            for _ in range(n):
                fn()
    stream.wait_stream(s)
    torch.cuda.synchronize()
    best = None
    for _ in range(5):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        g.replay()
        b.record(stream)
        b.synchronize()
        t = a.elapsed_time(b) * 1e3 / n
        best = t if best is None else min(best, t)
    del g
    return best


def e2e_leg(ws, w, inp, pats, flush, dev, K, world):
    """The same step on page-locked host buffers, all data movement inside
    the timed events. Headline: arf_run_host (copies of the step's inputs in,
    the kernels, copies of its outputs back). Beside it, zero-copy: arf_run on
    the host buffers themselves, the kernels reading and writing host memory
    over NVLink-C2C."""
    st = _e2e(ws, w, inp, pats, flush, dev, K, world, zero_copy=False)
    zc = _e2e(ws, w, inp, pats, flush, dev, K, world, zero_copy=True)
    st["zero_copy"] = {k: zc[k] for k in ("value", "ms_per_step", "api")}
    return st


def _e2e(ws, w, inp, pats, flush, dev, K, world, zero_copy):
    import torch

    import all_reduce_residual_gb300 as arf

    dt = inp.partials[0].dtype
    P = [p.pin_memory() for p in inp.partials]
    R, G = inp.residual.pin_memory(), inp.gamma.pin_memory()
    outs = {p: torch.empty_like(inp.residual).pin_memory() for p in pats}
    ro = torch.empty_like(inp.residual).pin_memory()
    runners = {p: arf.HostRunner(ws, p, w.W, w.M, w.H, dt, zero_copy=zero_copy) for p in pats}
    stream = torch.cuda.current_stream(dev)
    n = min(K, 500)

    def step():
        for p in pats:
            runners[p](P, R, G, w.eps, outs[p], ro)

    for _ in range(5):
        step()
    torch.cuda.synchronize()
    times = []
    barrier(world)
    for _ in range(n):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        step()
        b.record(stream)
        b.synchronize()
        times.append(a.elapsed_time(b) / 1e3)
    barrier(world)
    step_bytes = sum(w.bytes_per_call(p) for p in pats)
    units, slowest = aggregate(step_bytes * n, sum(times), world)
    plane = w.M * w.H * 2
    h2d = sum((w.W * plane) + ((plane + w.H * 2) if p == "rmsnorm" else 0) for p in pats)
    d2h = sum(plane * (2 if p == "rmsnorm" else 1) for p in pats)
    api = ("arf_run on pinned host buffers, no copies" if zero_copy else
           "arf_run_host: H2D copies, kernels, D2H copies")
    return {"value": round(units / slowest / 1e9, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": n, "ms_per_step": round(statistics.mean(times) * 1e3, 4),
            "api": api}


def cold_event_us(fn, flush, stream, n=50):
    """Mean CUDA-event time of fn() with the L2 flushed clean before each call."""
    import torch

    for _ in range(5):
        fn()
    ts = []
    for _ in range(n):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        b.synchronize()
        ts.append(a.elapsed_time(b) * 1e3)
    return statistics.mean(ts)


def roofline_context(ws, dev, flush, w, pattern, call_ms):
    """For the dominant call: the same-bytes device copy and the read-only
    pass over its reads, timed like the call (cold). At decode sizes all three
    sit at the launch-and-first-touch floor, which the HBM fraction cannot show."""
    import torch

    import all_reduce_residual_gb300 as arf

    stream = torch.cuda.current_stream(dev)
    nbytes, nread = w.bytes_per_call(pattern), w.read_bytes_per_call(pattern)
    half = max(16, nbytes // 2 // 16 * 16)
    src = torch.empty(half, dtype=torch.uint8, device=dev)
    dst = torch.empty(half, dtype=torch.uint8, device=dev)
    n16 = max(16, (nread + 15) // 16 * 16)
    buf = torch.zeros(n16, dtype=torch.uint8, device=dev)

    def read_pass():
        st = arf.arf_read_pass(ws.handle, buf.data_ptr(), n16, stream.cuda_stream)
        if st != arf.ARF_OK:
            raise arf.ArfError(st, "arf_read_pass")

    copy_us = cold_event_us(lambda: dst.copy_(src), flush, stream)
    read_us = cold_event_us(read_pass, flush, stream)
    call_us = statistics.mean(call_ms) * 1e3
    return {"call_us": round(call_us, 3), "copy_same_bytes_us": round(copy_us, 3),
            "read_only_pass_same_reads_us": round(read_us, 3)}


# The configurations of 8 MiB and more per partial besides the headline's,
# with the M values the 80 % target covers: k3_tp8 at M = 1024 and 2048
# (14 and 28 MiB per partial), tp4_80mib and tp16_8mib (8 MiB, fp16).
OTHER_CONFIGS = (("k3_tp8", 1024), ("k3_tp8", 2048), ("tp4_80mib", None), ("tp16_8mib", None))


def other_configs(ws, dev, flush, peak, skip):
    """Cold per-call fraction of the measured copy rate for each pattern of
    the other 8 MiB+ configurations, timed like the headline's calls (clean
    L2 flush and a random 0-2 us spin before each call; mean of 50). The
    first calls on freshly made inputs read slower (tp16_8mib: 39.6 us over
    its first 20 cold calls, 29.5 us after), so each pattern is first run 30
    times, each time after a flush."""
    import torch

    import all_reduce_residual_gb300 as arf
    from all_reduce_residual_gb300 import workloads as wl

    stream = torch.cuda.current_stream(dev)
    out = {}
    for name, M in OTHER_CONFIGS:
        if name == skip:
            continue
        w = wl.WORKLOADS[name].with_m(M) if M else wl.WORKLOADS[name]
        inp = wl.make_inputs(w, device=dev)
        P, R, G = inp.partials, inp.residual, inp.gamma
        ptrs = arf.pointer_array(P, dev)
        o, ro = torch.empty_like(R), torch.empty_like(R)
        key = f"{name} M={w.M}"
        out[key] = {}
        for pat in w.patterns:
            def fn():
                arf.run(ws, pat, P, R, G, w.eps, out=o, residual_out=ro if pat == "rmsnorm" else None, ptrs=ptrs)

            for _ in range(30):
                flush.zero_()
                fn()
            us = cold_event_us(fn, flush, stream)
            out[key]["ar" if pat == "allreduce" else "rms"] = round(w.bytes_per_call(pat) / us / 1e3 / peak, 4)
        del inp, P, R, G, ptrs, o, ro
        torch.cuda.empty_cache()
    return out


def sweep(ws, dev, flush, peak):
    """µs/call and GB/s for every workload, pattern and (k3_tp8) M, beside a
    device-to-device copy of the same bytes timed the same way, through
    arf_run (planner's plan; and the plan arf_workspace_autotune picks, in a
    workspace of its own) and through arf_run_ex with partials by value + PDL: cold
    (L2 flushed clean before each call, mean of 50 CUDA-event timings: the event
    clock ticks in steps of about 2 µs here, and the mean of many samples
    taken at random phases is unbiased where a median is not) and warm (a
    CUDA graph of 20 back-to-back calls, per-call time of the fastest of 5
    replays)."""
    import torch

    import all_reduce_residual_gb300 as arf
    from all_reduce_residual_gb300 import workloads as wl

    rows = []
    stream = torch.cuda.current_stream(dev)
    ws_tuned = arf.Workspace(dev.index if dev.index is not None else 0)  # autotuned plans live here

    def copy_cold_us(nbytes):
        """A plain device-to-device copy moving the same bytes (nbytes/2 read,
        nbytes/2 written), timed like the calls: the practical peak at this size."""
        half = max(16, nbytes // 2 // 16 * 16)
        src = torch.empty(half, dtype=torch.uint8, device=dev)
        dst = torch.empty(half, dtype=torch.uint8, device=dev)
        for _ in range(5):
            dst.copy_(src)
        ts = []
        for _ in range(50):
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            dst.copy_(src)
            b.record(stream)
            b.synchronize()
            ts.append(a.elapsed_time(b) * 1e3)
        return statistics.mean(ts)

    def read_cold_us(nbytes):
        """arf_read_pass over as many bytes as the call reads, timed like the
        calls: the read-only reference (on this GPU reads alone stream slower
        than a copy's mix of reads and writes at these sizes)."""
        n16 = max(16, (nbytes + 15) // 16 * 16)
        buf = torch.zeros(n16, dtype=torch.uint8, device=dev)

        def one():
            st = arf.arf_read_pass(ws.handle, buf.data_ptr(), n16, stream.cuda_stream)
            if st != arf.ARF_OK:
                raise arf.ArfError(st, "arf_read_pass")

        for _ in range(5):
            one()
        ts = []
        for _ in range(50):
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            one()
            b.record(stream)
            b.synchronize()
            ts.append(a.elapsed_time(b) * 1e3)
        return statistics.mean(ts)

    for name, w in list(wl.WORKLOADS.items()) + list(wl.EXTRA_WORKLOADS.items()):
        Ms = wl.K3_M_SWEEP if name == "k3_tp8" else (w.M,)
        for M in Ms:
            inp = wl.make_inputs(w, device=dev, M=M)
            ww = w.with_m(M)
            P, R, G = inp.partials, inp.residual, inp.gamma
            ptrs = arf.pointer_array(P, dev)
            out, ro = torch.empty_like(R), torch.empty_like(R)
            for pat in w.patterns:
                tuned_plan, tuned_us = ws_tuned.autotune(pat, P, R, G, w.eps, out=out,
                                                         residual_out=ro if pat == "rmsnorm" else None, ptrs=ptrs)

                def call(opt=False, wsx=None):
                    arf.run(wsx or ws, pat, P, R, G, w.eps, out=out, residual_out=ro if pat == "rmsnorm" else None,
                            ptrs=ptrs, by_value=opt, pdl=True if opt else None)

                def cold_us(opt, dirty=False):
                    for _ in range(10):
                        call(opt)
                    ts = []
                    for _ in range(50):
                        flush.zero_(dirty_only=dirty)
                        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                        a.record(stream)
                        call(opt)
                        b.record(stream)
                        b.synchronize()
                        ts.append(a.elapsed_time(b) * 1e3)
                    return statistics.mean(ts)

                def warm_us(opt, wsx=None):
                    g = torch.cuda.CUDAGraph()
                    s = torch.cuda.Stream(dev)
                    s.wait_stream(stream)
                    with torch.cuda.stream(s):
                        with torch.cuda.graph(g, stream=s):
                            for _ in range(20):
                                call(opt, wsx)
                    stream.wait_stream(s)
                    torch.cuda.synchronize()
                    best = None
                    for _ in range(5):
                        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                        a.record(stream)
                        g.replay()
                        b.record(stream)
                        b.synchronize()
                        t = a.elapsed_time(b) * 1e3 / 20
                        best = t if best is None else min(best, t)
                    del g
                    return best

                us, us_opt, us_dirty = cold_us(False), cold_us(True), cold_us(False, dirty=True)
                us_copy = copy_cold_us(ww.bytes_per_call(pat))
                us_read = read_cold_us(ww.read_bytes_per_call(pat))
                warm, warm_opt, warm_tuned = warm_us(False), warm_us(True), warm_us(False, ws_tuned)
                nbytes = ww.bytes_per_call(pat)
                plan = ws.plan(pat, w.W, M, w.H, torch.bfloat16 if w.dtype == "bf16" else torch.float16)
                rows.append({"workload": name, "extra": name in wl.EXTRA_WORKLOADS,
                             "W": w.W, "M": M, "H": w.H, "dtype": w.dtype, "pattern": pat,
                             "bytes": nbytes, "us_cold": round(us, 3), "us_warm_graph": round(warm, 3),
                             "gbs_cold": round(nbytes / us / 1e3, 1), "frac_cold": round(nbytes / us / 1e3 / peak, 4),
                             "us_cold_byvalue_pdl": round(us_opt, 3), "us_warm_graph_byvalue_pdl": round(warm_opt, 3),
                             "us_cold_write_only_flush": round(us_dirty, 3),
                             "us_cold_copy_same_bytes": round(us_copy, 3),
                             "us_cold_read_only_same_reads": round(us_read, 3),
                             "us_warm_graph_autotuned": round(warm_tuned, 3),
                             "autotuned_plan": [tuned_plan.path, tuned_plan.threads, tuned_plan.vpt, tuned_plan.cluster,
                                                tuned_plan.grid, tuned_plan.w_spec, tuned_plan.stages],
                             "plan": [plan.path, plan.threads, plan.vpt, plan.cluster, plan.grid, plan.w_spec,
                                      plan.stages]})
            del inp, P, R, G, out, ro, ptrs
            torch.cuda.empty_cache()
    ws_tuned.close()
    return rows


# ---------------------------------------------------------------------------
# the CPU oracle legs
# ---------------------------------------------------------------------------


def _oracle_step(oracle, w, codes, rows, pats):
    P = [c[:rows] for c in codes["P"]]
    dt = oracle.BF16 if w.dtype == "bf16" else oracle.FP16
    for p in pats:
        if p == "allreduce":
            oracle.run(oracle.ALLREDUCE, P, dtype=dt)
        else:
            oracle.run(oracle.AR_RESIDUAL_RMSNORM, P, codes["R"][:rows], codes["G"], w.eps, dtype=dt)


def _codes(inp):
    from all_reduce_residual_gb300 import workloads as wl

    return {"P": [wl.codes(p) for p in inp.partials], "R": wl.codes(inp.residual), "G": wl.codes(inp.gamma)}


def _bytes(w, rows, pats):
    return sum(w.with_m(rows).bytes_per_call(p) for p in pats)


def cpu_baseline(w, inp, budget_s=10.0):
    """The oracle as it stands, single-threaded, repeated on the full workload
    step until about budget_s of CPU time has run."""
    import oracle

    pats = [p for p in PATTERNS if p in w.patterns]
    codes = _codes(inp)
    oracle.default()
    done, t0 = 0, time.perf_counter()
    while True:
        _oracle_step(oracle, w, codes, w.M, pats)
        done += 1
        el = time.perf_counter() - t0
        if el >= budget_s:
            break
    gbs = _bytes(w, w.M, pats) * done / el / 1e9
    return {"value": round(gbs, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"{done} full steps of {w.name} ({' + '.join(pats)}, M={w.M}) in {el:.1f} s, "
                      f"single-threaded C oracle"}


def run_reference(args):
    """The reference arm: the CPU oracle on the host cores, same metric. Under
    torchrun only rank 0 runs; the others exit at once."""
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import oracle
    from all_reduce_residual_gb300 import workloads as wl

    w = {**wl.WORKLOADS, **wl.EXTRA_WORKLOADS}[args.workload]
    if args.m is not None:
        w = w.with_m(args.m)
    pats = [p for p in PATTERNS if p in w.patterns and (args.pattern is None or p == args.pattern)]
    inp = wl.make_inputs(w)
    codes = _codes(inp)
    oracle.default()
    t0 = time.perf_counter()
    _oracle_step(oracle, w, codes, w.M, pats)
    full = time.perf_counter() - t0
    budget = 90.0  # seconds for the whole timed run
    rows = max(1, min(w.M, int(w.M * budget / max(1e-9, full * max(1, args.steps)))))
    for _ in range(args.warmup):
        _oracle_step(oracle, w, codes, rows, pats)
    times = []
    for _ in range(args.steps):
        a = time.perf_counter()
        _oracle_step(oracle, w, codes, rows, pats)
        times.append(time.perf_counter() - a)
    total = sum(times)
    value = _bytes(w, rows, pats) * args.steps / total / 1e9
    sample = f"{rows} of {w.M} rows of {w.name} per step ({' + '.join(pats)}), single-threaded C oracle"
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(total / args.steps * 1e3, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic (same seeded inputs as the GPU arm)",
            "config": {"workload": f"{w.name}: W={w.W} M={w.M} H={w.H} {w.dtype}, one {' + one '.join(pats)} call per step",
                       "W": w.W, "M": w.M, "H": w.H, "io_dtype": w.dtype, "sample_rows": rows},
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_arf(args)


if __name__ == "__main__":
    main()
