"""Measured launch-plan table for the planner.

    python -m all_reduce_residual_gb300.plan_table [--out FILE] [--reps N]

Runs on one GPU. For every (pattern, dtype, W, H) of the table's shape list
and a ladder of row counts M, it times candidate launch plans cold, the way
the benchmark times a call: the L2 is flushed clean before each call (a write
of twice its size, then a read of another buffer of that size, then a spin of
random length so that the call starts at a random phase of the event clock)
and the call is timed with CUDA events on its stream. The fastest plan at each measured M
is kept. Neighbouring row counts with the same winner merge into one range,
and the ranges split at the geometric mean of the measured row counts. The
result is written as C initialisers to ``csrc/arf_plan_table.inc``, which the
library's planner (arf_plan_for_caps) consults before its closed-form rules,
for devices whose capabilities equal those the table was measured on.

The shapes follow the launch-configuration story of the source pages: the
launch shape comes from the device (flashinfer PR #1507 "update allreduce to
match trtllm", Highlights: threads per block and cluster size from the SM
count), chosen per shape (vLLM PR #53318 "Tune FlashInfer all-reduce selection
on SM103", Scope: a selection table by device and world size).

Each table row gives a plan shape and a grid rule, so that one row serves a
range of M:
  GRID_ROWS      grid = M * cluster            (one CTA or cluster per row)
  GRID_RESIDENT  grid = min(M, per_sm * SMs / cluster) * cluster
  GRID_CHUNKS    grid = ceil(M * H / 8 / (threads * vpt))   (flat kAllReduce)
  GRID_TILES     grid = min(ceil(H / threads) * M, per_sm * SMs)  (elementwise kAllReduce)
"""
from __future__ import annotations

import argparse
import math
import os
import random
import statistics
import sys
import time

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

OUT_DEFAULT = os.path.join(os.path.dirname(os.path.abspath(__file__)), "csrc", "arf_plan_table.inc")

GRID_ROWS, GRID_RESIDENT, GRID_CHUNKS, GRID_TILES = 0, 1, 2, 3
PATH_FLAT, PATH_ROW, PATH_CLUSTER, PATH_ASYNC, PATH_ELEM, PATH_BULK = 0, 1, 2, 3, 4, 5
COMPILED_W = (1, 2, 4, 8, 12, 16)
MAX_THREADS = 512

# (W, H, dtype, patterns): the five benchmark workloads' shapes and the extra
# shapes that reach the other kernels.
KEYS = [
    (2, 1024, "bf16", ("rmsnorm", "allreduce")),
    (2, 4096, "bf16", ("allreduce", "rmsnorm")),
    (8, 7168, "bf16", ("allreduce", "rmsnorm")),
    (4, 7168, "bf16", ("allreduce", "rmsnorm")),
    (16, 7168, "fp16", ("rmsnorm", "allreduce")),
    (3, 7168, "bf16", ("rmsnorm",)),
    (12, 7168, "fp16", ("rmsnorm",)),
    (4, 7168, "fp16", ("rmsnorm",)),
    (4, 32768, "bf16", ("rmsnorm",)),
    (1, 7168, "fp16", ("rmsnorm",)),
    (2, 32776, "bf16", ("rmsnorm",)),
    (2, 4098, "bf16", ("allreduce", "rmsnorm")),
]
M_LADDER = (1, 2, 4, 8, 16, 32, 64, 128, 256, 512, 1024, 2048, 4096)
# the workloads' own row counts, measured besides the ladder
EXTRA_M = {(4, 7168, "bf16"): (5851,), (16, 7168, "fp16"): (585,), (3, 7168, "bf16"): (2000,),
           (12, 7168, "fp16"): (585,), (4, 7168, "fp16"): (5851,), (1, 7168, "fp16"): (4972,)}
MAX_BYTES = 2 << 30  # largest input set measured per shape


def grid_for(kind, per_sm, caps, M, H, threads, vpt, cluster):
    """The grid a table row gives at M rows (the library computes the same)."""
    if kind == GRID_ROWS:
        g = M * cluster
    elif kind == GRID_RESIDENT:
        g = min(M, max(1, per_sm * caps.num_sms // cluster)) * cluster
    elif kind == GRID_CHUNKS:
        g = -(-(M * H // 8) // (threads * vpt))
    else:
        g = min(-(-H // threads) * M, per_sm * caps.num_sms)
    return int(max(1, min(g, (2 ** 31 - 1) // cluster * cluster)))


def candidates(caps, pattern, W, H):
    """Plan shapes to try: (path, threads, vpt, cluster, w_spec, stages, kind, per_sm)."""
    out = []
    ws = W if W in COMPILED_W else 0  # the compiled rank count where there is one
    if H % 8 != 0:
        if pattern == "allreduce":
            # the flat kernel over the contiguous [M,H] as one range of chunks
            # (arf_plan_check admits it where M * H is a multiple of 8)
            for t in (128, 256, 512):
                for u in (1, 2, 4):
                    if u == 1 or (u == 2 and ws <= 8) or (u == 4 and ws <= 4):
                        out.append((PATH_FLAT, t, u, 1, ws, 0, GRID_CHUNKS, 0))
        for t in (64, 128, 256, 512):
            if pattern == "allreduce":
                for per in (2, 4, 8):
                    if per * t <= caps.max_threads_per_sm:
                        out.append((PATH_ELEM, t, 1, 1, 0, 0, GRID_TILES, per))
            else:
                out.append((PATH_ELEM, t, 1, 1, 0, 0, GRID_ROWS, 0))
                for per in (1, 2, 4, 8):
                    if per * t <= caps.max_threads_per_sm:
                        out.append((PATH_ELEM, t, 1, 1, 0, 0, GRID_RESIDENT, per))
        return out
    C = H // 8
    if pattern == "allreduce":
        for t in (128, 256, 512):
            for u in (1, 2, 4):
                if u == 1 or (u == 2 and ws <= 8) or (u == 4 and ws <= 4):
                    out.append((PATH_FLAT, t, u, 1, ws, 0, GRID_CHUNKS, 0))
        return out

    def threads_for(chunks, vpt):
        return max(32, -(-(-(-chunks // vpt)) // 32) * 32)

    # one CTA per row: the fewest chunks per thread that fit 512 threads, and two and four times that
    v0 = next((v for v in (1, 2, 4, 8) if threads_for(C, v) <= MAX_THREADS), None)
    for vpt in sorted({v for v in ((v0, 2 * v0, 4 * v0) if v0 else ()) if v <= 8}):
        t = threads_for(C, vpt)
        out.append((PATH_ROW, t, vpt, 1, ws, 0, GRID_ROWS, 0))
        for per in (1, 2, 3, 4):
            if per * t <= caps.max_threads_per_sm:
                out.append((PATH_ROW, t, vpt, 1, ws, 0, GRID_RESIDENT, per))
    # a row over a cluster, one or two chunks per thread
    for cs in (2, 4, 8, 16):
        if cs > caps.max_cluster:
            continue
        for vpt in (1, 2):
            t = threads_for(-(-C // cs), vpt)
            if t > MAX_THREADS:
                continue
            out.append((PATH_CLUSTER, t, vpt, cs, ws, 0, GRID_ROWS, 0))
            for per in (1, 2, 4):
                if per * t <= caps.max_threads_per_sm:
                    out.append((PATH_CLUSTER, t, vpt, cs, ws, 0, GRID_RESIDENT, per))
    # the bulk-copy ring: a resident grid walking the rows, or one CTA per row
    for t in (128, 256, 512):
        for st in (2, 3, 4):
            out.append((PATH_BULK, t, 1, 1, ws, st, GRID_ROWS, 0))
            for per in (1, 2):
                out.append((PATH_BULK, t, 1, 1, ws, st, GRID_RESIDENT, per))
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--out", default=OUT_DEFAULT)
    ap.add_argument("--reps", type=int, default=80, help="cold timings per finalist")
    ap.add_argument("--keys", default=None,
                    help="comma-separated indices into KEYS: measure only these shapes and keep the other rows "
                         "of the existing table (default: measure all and write a new table)")
    args = ap.parse_args()

    import torch

    import all_reduce_residual_gb300 as arf
    from all_reduce_residual_gb300 import build as arf_build
    from all_reduce_residual_gb300 import workloads as wl

    arf_build.build()
    dev = torch.device("cuda", 0)
    ws = arf.Workspace(0)
    caps = ws.caps
    stream = torch.cuda.current_stream(dev)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    nflush = max(2 * l2, 256 << 20)
    fw = torch.empty(nflush, dtype=torch.uint8, device=dev)
    fr = torch.zeros(nflush // 4, dtype=torch.int32, device=dev)

    rng = random.Random(4321)

    def flush():
        # then a spin of a random 0-4095 SM cycles: the timed call starts at a
        # random phase of the event clock (which advances in steps of about
        # 2 us), so that means of many cold timings are unbiased
        fw.zero_()
        torch.amax(fr)
        torch.cuda._sleep(rng.randrange(4096))

    def time_cold(fn, n):
        ts = []
        for _ in range(n):
            flush()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            b.synchronize()
            ts.append(a.elapsed_time(b) * 1e3)
        return ts

    keys = KEYS if args.keys is None else [KEYS[int(i)] for i in args.keys.split(",")]
    rows = []  # (pattern, dtype, W, H, M, winner tuple, us, library plan us)
    t_start = time.time()
    for W, H, dts, pats in keys:
        dcode = arf.ARF_BF16 if dts == "bf16" else arf.ARF_FP16
        Ms = sorted(set(M_LADDER) | set(EXTRA_M.get((W, H, dts), ())))
        Ms = [M for M in Ms if (W + 3) * M * H * 2 <= MAX_BYTES]
        for M in Ms:
            w = wl.custom(W, M, H, dts, 0.5, 1e-6, config_id=950)
            inp = wl.make_inputs(w, device=dev)
            P, R, G = inp.partials, inp.residual, inp.gamma
            ptrs = arf.pointer_array(P, dev)
            out, ro = torch.empty_like(R), torch.empty_like(R)
            for pattern in pats:
                pat = arf.PATTERNS[pattern]
                rms = pattern == "rmsnorm"
                lib_plan = ws.plan(pattern, W, M, H, wl.TORCH_DTYPE[dts])
                cands = []
                for c in candidates(caps, pattern, W, H):
                    path, t, vpt, cs, wsp, st, kind, per = c
                    pl = arf.Plan(path=path, threads=t, vpt=vpt, cluster=cs,
                                  grid=grid_for(kind, per, caps, M, H, t, vpt, cs), w_spec=wsp, stages=st)
                    if arf.arf_plan_check(caps, pl, pat, W, M, H, dcode) != arf.ARF_OK:
                        continue
                    cands.append((c, pl))
                lp = (lib_plan.path, lib_plan.threads, lib_plan.vpt, lib_plan.cluster, lib_plan.grid,
                      lib_plan.w_spec, lib_plan.stages)
                cands.append((None, lib_plan))

                def runner(pl):
                    def f():
                        arf.run(ws, pat, P, R, G, w.eps, out=out, residual_out=ro if rms else None, ptrs=ptrs,
                                plan=pl)
                    return f

                # The first cold calls on freshly made inputs read slower (on
                # GB300, W = 16 fp16 M = 585: 39.6 us over the first 20, 29.5
                # us after): warm up on the library's plan before scoring.
                warm = runner(lib_plan)
                for _ in range(30):
                    flush()
                    warm()
                scored = []
                for c, pl in cands:
                    f = runner(pl)
                    try:
                        f()
                        f()
                        torch.cuda.synchronize()
                    except arf.ArfError:
                        continue  # a shape this device cannot hold
                    scored.append((statistics.mean(time_cold(f, 10)), c, pl))
                scored.sort(key=lambda x: x[0])
                finals = scored[:6]
                if not any(c is None for _, c, _ in finals):
                    finals += [s for s in scored if s[1] is None]
                means = {id(x): [] for x in finals}
                for _ in range(4):  # interleaved rounds against drift
                    for x in finals:
                        means[id(x)] += time_cold(runner(x[2]), max(1, args.reps // 4))
                res = sorted(((statistics.mean(means[id(x)]), x[1], x[2]) for x in finals), key=lambda y: y[0])
                lib_us = next(m for m, c, _ in res if c is None)
                best_us, best_c, best_pl = res[0]
                if best_c is None:  # the library's own plan won: record it as a table shape
                    best_c = shape_of(best_pl, caps, M, H)
                rows.append((pattern, dts, W, H, M, best_c, best_us, lib_us, lp))
                print(f"{pattern:9s} {dts} W={W:2d} H={H:5d} M={M:5d}: best {fmt(best_c)} {best_us:8.3f} us; "
                      f"library plan {lp} {lib_us:8.3f} us  [{time.time() - t_start:6.0f} s]", flush=True)
            del inp, P, R, G, ptrs, out, ro
            torch.cuda.empty_cache()
    keep = []
    if args.keys is not None and os.path.exists(args.out):
        measured = {(0 if k[3] == "allreduce" else 1, 0 if k[2] == "bf16" else 1, k[0], k[1])
                    for W, H, dts, pats in keys for k in [(W, H, dts, p) for p in pats]}
        keep = [ln for ln in open(args.out) if ln.startswith("{") and
                tuple(int(x) for x in ln[1:ln.index("}")].split(",")[4:8]) not in measured]
    write_table(args.out, caps, rows, torch.cuda.get_device_name(dev), keep)
    ws.close()


FIELDS = ("num_sms", "max_cluster", "max_threads_per_sm", "max_smem_per_block", "pattern", "dtype", "W", "H", "m_lo",
          "m_hi", "path", "threads", "vpt", "cluster", "w_spec", "stages", "grid_rule", "per_sm")


def read_table(path=OUT_DEFAULT):
    """The rows of a written table, as dicts keyed by FIELDS."""
    import re

    rows = []
    for ln in open(path):
        m = re.match(r"\s*\{([-0-9, ]+)\},", ln)
        if m:
            vals = [int(x) for x in m.group(1).split(",")]
            assert len(vals) == len(FIELDS), ln
            rows.append(dict(zip(FIELDS, vals)))
    return rows


class _Caps:
    def __init__(self, num_sms):
        self.num_sms = num_sms


def row_plan_fields(row, M):
    """(path, threads, vpt, cluster, grid, w_spec, stages) a table row gives at M."""
    g = grid_for(row["grid_rule"], row["per_sm"], _Caps(row["num_sms"]), M, row["H"], row["threads"], row["vpt"],
                 row["cluster"])
    return (row["path"], row["threads"], row["vpt"], row["cluster"], g, row["w_spec"], row["stages"])


def shape_of(pl, caps, M, H):
    """The table shape of an explicit plan measured at M rows: its grid rule
    is whichever rule reproduces its grid."""
    for kind, per in ((GRID_ROWS, 0), (GRID_CHUNKS, 0), (GRID_RESIDENT, 1), (GRID_RESIDENT, 2), (GRID_RESIDENT, 3),
                      (GRID_RESIDENT, 4), (GRID_TILES, 2), (GRID_TILES, 4), (GRID_TILES, 8)):
        if grid_for(kind, per, caps, M, H, pl.threads, pl.vpt, pl.cluster) == pl.grid:
            return (pl.path, pl.threads, pl.vpt, pl.cluster, pl.w_spec, pl.stages, kind, per)
    per = max(1, -(-pl.grid // caps.num_sms))  # nearest resident rule
    return (pl.path, pl.threads, pl.vpt, pl.cluster, pl.w_spec, pl.stages, GRID_RESIDENT, per)


def fmt(c):
    names = {0: "flat", 1: "row", 2: "cluster", 3: "async", 4: "elem", 5: "bulk"}
    kinds = {0: "rows", 1: "resident", 2: "chunks", 3: "tiles"}
    path, t, vpt, cs, wsp, st, kind, per = c
    return f"{names[path]} {t}x{vpt} c{cs} w{wsp} s{st} {kinds[kind]}{per if kind in (1, 3) else ''}"


def write_table(path, caps, rows, device_name, keep=()):
    """Merge the measured points into M ranges and write the C initialisers
    (after `keep`: rows of an earlier table for shapes not measured now)."""
    by_key = {}
    for r in rows:
        by_key.setdefault((r[0], r[1], r[2], r[3]), []).append(r)
    lines = [
        "// Launch-plan table of the planner (arf_plan_for_caps), written by",
        "// all_reduce_residual_gb300/plan_table.py from cold timings (L2 flushed before",
        f"// each call) on {device_name}. Regenerate it with that script; do not edit.",
        "// Fields: num_sms, max_cluster, max_threads_per_sm, max_smem_per_block, pattern,",
        "// dtype, W, H, M_lo, M_hi, path, threads, vpt, cluster, w_spec, stages, grid rule,",
        "// CTAs per SM (resident and tiles rules). Comments: the measured row counts,",
        "// the winner's time and the time of the plan the library chose before.",
    ] + [ln.rstrip("\n") for ln in keep]
    for (pattern, dts, W, H), pts in sorted(by_key.items()):
        pts.sort(key=lambda r: r[4])
        m_max = (1 << 40) // H
        ranges = []
        for i, r in enumerate(pts):
            lo = 1 if i == 0 else int(math.floor(math.sqrt(pts[i - 1][4] * r[4]))) + 1
            hi = m_max if i == len(pts) - 1 else int(math.floor(math.sqrt(r[4] * pts[i + 1][4])))
            if ranges and ranges[-1][2] == r[5]:
                ranges[-1][1] = hi
                ranges[-1][3].append(r)
            else:
                ranges.append([lo, hi, r[5], [r]])
        pc = 0 if pattern == "allreduce" else 1
        dc = 0 if dts == "bf16" else 1
        for lo, hi, c, rs in ranges:
            kpath, t, vpt, cs, wsp, st, kind, per = c
            note = "; ".join(f"M={r[4]} {r[6]:.2f} us (before {r[7]:.2f})" for r in rs)
            lines.append(f"{{{caps.num_sms}, {caps.max_cluster}, {caps.max_threads_per_sm}, {caps.max_smem_per_block}, "
                         f"{pc}, {dc}, {W}, {H}, {lo}, {hi}, {kpath}, {t}, {vpt}, {cs}, {wsp}, {st}, {kind}, {per}}},"
                         f"  // {note}")
    with open(path, "w") as f:
        f.write("\n".join(lines) + "\n")
    print(f"wrote {path}: {sum(ln.startswith('{') for ln in lines)} rows")


if __name__ == "__main__":
    main()
