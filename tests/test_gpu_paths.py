"""Every kernel shape, ragged and edge sizes, and the call semantics of
arf_run on the GPU, each checked against the CPU oracle.

Covers: every launch plan shape (flat unroll factors, row and cluster paths
with 2..16 CTAs, every chunks-per-thread count, grids smaller than the work),
generic and specialised rank counts, W up to 64 and H up to 524288, ragged
sizes, M = 0, in-place residual, input preservation, guard bands around the
outputs, run-to-run determinism, rank-order permutations, the hand-worked
rows, non-finite inputs, rejected calls, workspace churn, CUDA-graph replay
and the host-buffer entry point (plain and pipelined, pinned and pageable,
from two threads, under graph capture)."""
import ctypes

import numpy as np
import pytest
import torch

import all_reduce_residual_gb300 as arf
import oracle
import pins
from all_reduce_residual_gb300 import workloads as wl
from gpu_util import DT, assert_parity, bitwise_equal, gpu_run, oracle_run, to_device

pytestmark = pytest.mark.gpu
RMS, AR = arf.ARF_AR_RESIDUAL_RMSNORM, arf.ARF_ALLREDUCE


@pytest.fixture(scope="module")
def ws():
    with arf.Workspace(0) as w:
        yield w


def inputs(W, M, H, dtype="bf16", sigma=1.0, eps=1e-6, cid=900):
    return wl.make_inputs(wl.custom(W, M, H, dtype, sigma, eps, config_id=cid))


def check(ws, pattern, inp, plan=None, in_place=False, what=""):
    P, R, G = to_device(inp)
    got = gpu_run(ws, pattern, P, R, G, inp.workload.eps, plan=plan, in_place=in_place)
    ref = oracle_run(pattern, inp)
    assert_parity(DT[inp.workload.dtype], pattern, got, ref, what)
    return got


def rms_plans(ws, W, M, H, grids=("full", 1)):
    """Every legal RMS plan shape for these sizes on this device."""
    caps = ws.caps
    C = H // 8
    plans = []
    for cs in (1, 2, 4, 8, 16):
        if cs > caps.max_cluster:
            continue
        slice_ = -(-C // cs)
        for vpt in (1, 2, 4, 8):
            per_thread = -(-slice_ // vpt)
            threads = max(32, -(-per_thread // 32) * 32)
            if threads > 512:
                continue
            for g in grids:
                nclus = min(M, 2 * caps.num_sms) if g == "full" else g
                for w_spec in {0, W if W in arf.COMPILED_W else 0}:
                    p = arf.Plan(path=arf.ARF_PATH_ROW if cs == 1 else arf.ARF_PATH_CLUSTER, threads=threads,
                                 vpt=vpt, cluster=cs, grid=max(1, nclus) * cs, w_spec=w_spec)
                    assert arf.arf_plan_check(caps, p, RMS, W, M, H, arf.ARF_BF16) == arf.ARF_OK, p
                    plans.append(p)
    if W in arf.COMPILED_W:  # the streaming kernel, every ring depth that fits
        for stages in range(2, 9):
            for g in ("full", 1, 3):
                grid = min(M, caps.num_sms) if g == "full" else g
                p = arf.Plan(path=arf.ARF_PATH_ASYNC, threads=256, vpt=1, cluster=1, grid=grid, w_spec=W,
                             stages=stages)
                if arf.arf_plan_check(caps, p, RMS, W, M, H, arf.ARF_BF16) == arf.ARF_OK:
                    plans.append(p)
    return plans


@pytest.mark.parametrize("W,M,H,dtype", [(3, 37, 1000, "bf16"), (8, 5, 7168, "bf16"), (16, 3, 4096, "fp16"),
                                         (1, 9, 8, "bf16"), (64, 2, 256, "fp16"), (5, 4, 32768, "bf16"),
                                         (2, 19, 2056, "bf16"), (4, 41, 7176, "bf16"), (16, 23, 7168, "fp16"),
                                         (8, 13, 32768, "bf16"), (1, 300, 264, "fp16"), (12, 7, 7168, "fp16"),
                                         (12, 3, 1000, "bf16")])
def test_every_rms_plan(ws, W, M, H, dtype):
    inp = inputs(W, M, H, dtype)
    ref = oracle_run(RMS, inp)
    P, R, G = to_device(inp)
    ro_first = None
    ran = 0
    for plan in rms_plans(ws, W, M, H):
        try:
            got = gpu_run(ws, RMS, P, R, G, inp.workload.eps, plan=plan)
        except arf.ArfError as e:  # a cluster or ring shape this device cannot keep resident
            assert e.status == arf.ARF_ERR_UNSUPPORTED and (plan.cluster > 1 or plan.stages > 0), e
            continue
        ran += 1
        assert_parity(DT[dtype], RMS, got, ref, f"{plan}")
        if ro_first is None:
            ro_first = got[1]
        assert np.array_equal(got[1], ro_first)
    assert ran >= 4


@pytest.mark.parametrize("W,M,H,dtype", [(3, 37, 1000, "bf16"), (2, 1, 8, "bf16"), (16, 11, 2056, "fp16"),
                                         (8, 3, 7168, "bf16"), (4, 5, 264, "fp16"), (1, 7, 24, "bf16"),
                                         (12, 9, 7168, "fp16")])
def test_every_flat_plan(ws, W, M, H, dtype):
    inp = inputs(W, M, H, dtype)
    ref = oracle_run(AR, inp)
    P, R, G = to_device(inp)
    specs = {0, W if W in arf.COMPILED_W else 0}
    for w_spec in specs:
        for u in (1, 2, 4):
            for threads in (32, 256, 512):
                for grid in (1, 7, 1000):
                    p = arf.Plan(path=arf.ARF_PATH_FLAT, threads=threads, vpt=u, cluster=1, grid=grid, w_spec=w_spec)
                    if arf.arf_plan_check(ws.caps, p, AR, W, M, H, DT[dtype]) != arf.ARF_OK:
                        continue
                    got = gpu_run(ws, AR, P, R, G, 0.0, plan=p)
                    assert_parity(DT[dtype], AR, got, ref, f"{p}")


@pytest.mark.parametrize("W", [3, 5, 6, 7, 9, 12, 17, 31, 32, 33, 63, 64])
@pytest.mark.parametrize("pattern", [AR, RMS])
def test_generic_rank_counts(ws, W, pattern):
    check(ws, pattern, inputs(W, 3, 264, "bf16" if W % 2 else "fp16", sigma=0.3), what=f"W={W}")


@pytest.mark.parametrize("M,H", [(1, 8), (1, 32768), (2500, 64), (5000, 8), (3, 7176), (3, 32776), (2, 65536),
                                 (40, 40960), (80, 32776), (2, 262144), (1, 524288)])
@pytest.mark.parametrize("pattern", [AR, RMS])
def test_ragged_and_extreme_shapes(ws, M, H, pattern):
    check(ws, pattern, inputs(4, M, H), what=f"M={M} H={H}")
    if pattern == RMS and M == 80:  # rows of 4097 chunks for half the SMs: the bulk ring
        assert ws.plan(RMS, 4, M, H, torch.bfloat16).path == arf.ARF_PATH_BULK


@pytest.mark.parametrize("W,M,H,dtype", [(64, 2, 524288, "bf16"), (64, 300, 7168, "fp16"), (64, 1, 524288, "fp16"),
                                         (1, 3, 524288, "bf16")])
@pytest.mark.parametrize("pattern", [AR, RMS])
def test_maximum_sizes(ws, pattern, W, M, H, dtype):
    """The build's limits together: ARF_MAX_W ranks, rows of ARF_MAX_H
    elements (split over the largest cluster or the elementwise path), and
    the generic rank count over many rows."""
    assert W <= arf.ARF_MAX_W and H <= arf.ARF_MAX_H
    check(ws, pattern, inputs(W, M, H, dtype, sigma=0.2), what=f"W={W} M={M} H={H} {dtype}")


def test_zero_rows_launch_nothing(ws):
    P = [torch.zeros((0, 64), dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    out = torch.full((16,), 7, dtype=torch.int16, device="cuda")
    st = arf.arf_run(ws.handle, RMS, 2, arf.pointer_array(P).data_ptr(), out.data_ptr(), out.data_ptr(), 1e-6,
                     out.data_ptr(), out.data_ptr() + 16, 0, 64, arf.ARF_BF16, torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert st == arf.ARF_OK
    assert (out == 7).all()


def _guarded(M, H, dt, pad=2048):
    buf = torch.full((M * H + 2 * pad,), -12345, dtype=torch.int16, device="cuda")
    return buf, buf[pad:pad + M * H].view(dt).view(M, H)


@pytest.mark.parametrize("pattern", [AR, RMS])
def test_guard_bands_and_input_preservation(ws, pattern):
    inp = inputs(8, 33, 7168)
    P, R, G = to_device(inp)
    copies = [p.clone() for p in P] + [R.clone(), G.clone()]
    ob, out = _guarded(33, 7168, torch.bfloat16)
    rb, ro = _guarded(33, 7168, torch.bfloat16)
    arf.run(ws, pattern, P, R, G, 1e-6, out=out, residual_out=ro if pattern == RMS else None)
    torch.cuda.synchronize()
    for buf in (ob, rb):
        assert (buf[:2048] == -12345).all() and (buf[-2048:] == -12345).all(), "write outside the output"
    for a, b in zip(P + [R, G], copies):
        assert torch.equal(a, b), "an input was modified"
    ref = oracle_run(pattern, inp)
    got = (wl.codes(out.cpu()), wl.codes(ro.cpu()) if pattern == RMS else None)
    assert_parity(oracle.BF16, pattern, got, ref)


def test_in_place_residual(ws):
    inp = inputs(8, 70, 7168)
    P, R, G = to_device(inp)
    for plan in rms_plans(ws, 8, 70, 7168, grids=("full",))[:6] + [None]:
        a = gpu_run(ws, RMS, P, R, G, 1e-6, plan=plan)
        b = gpu_run(ws, RMS, P, R, G, 1e-6, plan=plan, in_place=True)
        assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    assert_parity(oracle.BF16, RMS, b, oracle_run(RMS, inp))


def test_run_to_run_determinism(ws):
    inp = inputs(8, 64, 7168, sigma=0.25)
    P, R, G = to_device(inp)
    first = gpu_run(ws, RMS, P, R, G, 1e-6)
    outs = []
    ro = torch.empty_like(R)
    for _ in range(100):
        o, _ = arf.run(ws, RMS, P, R, G, 1e-6, residual_out=ro)
        outs.append(o)
    torch.cuda.synchronize()
    for o in outs:
        assert np.array_equal(wl.codes(o.cpu()), first[0])
    assert np.array_equal(wl.codes(ro.cpu()), first[1])


def test_rank_order_permutations(ws):
    inp = inputs(8, 16, 1024, sigma=2.0)
    P, R, G = to_device(inp)
    for order in ([7, 6, 5, 4, 3, 2, 1, 0], [3, 1, 4, 0, 5, 2, 7, 6]):
        Pp = [P[i] for i in order]
        got = gpu_run(ws, RMS, Pp, R, G, 1e-6)
        assert_parity(oracle.BF16, RMS, got, oracle_run(RMS, inp, order=order), f"order {order}")
    same = [P[0]] * 8
    a = gpu_run(ws, RMS, same, R, G, 1e-6)
    b = gpu_run(ws, RMS, same[::-1], R, G, 1e-6)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    two = inputs(2, 16, 1024, sigma=3.0)
    P2, R2, G2 = to_device(two)
    a = gpu_run(ws, RMS, P2, R2, G2, 1e-6)
    b = gpu_run(ws, RMS, P2[::-1], R2, G2, 1e-6)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_worked_rows_on_gpu(ws):
    for case in pins.load_golden():
        dtype = DT[case["dtype"]]
        pat = AR if case["pattern"] == "allreduce" else RMS
        W = sum(1 for k in case if k.startswith("p") and k[1:].isdigit())
        dt = torch.bfloat16 if dtype == oracle.BF16 else torch.float16
        dname = case["dtype"]
        P = [wl.from_codes(pins.exact_codes(dtype, case[f"p{r}"])[None, :], dname).cuda() for r in range(W)]
        R = G = None
        eps = 0.0
        if pat == RMS:
            R = wl.from_codes(pins.exact_codes(dtype, case["residual"])[None, :], dname).cuda()
            G = wl.from_codes(pins.exact_codes(dtype, case["gamma"]), dname).cuda()
            eps = float(case["eps"])
        out, ro = arf.run(ws, pat, P, R, G, eps)
        torch.cuda.synchronize()
        want = pins.exact_codes(dtype, case["expect_out"])
        got = wl.codes(out.cpu())[0]
        assert out.dtype == dt
        if pat == RMS:
            assert np.array_equal(wl.codes(ro.cpu())[0], pins.exact_codes(dtype, case["expect_residual_out"])), \
                case["case"]
        assert np.array_equal(got, want), (case["case"], got, want)


def test_non_finite_inputs_propagate(ws):
    H = 64
    p0 = torch.zeros((2, H), dtype=torch.bfloat16)
    p1 = torch.zeros((2, H), dtype=torch.bfloat16)
    p0[0, 0], p1[0, 0] = float("inf"), float("-inf")   # inf + -inf = NaN
    p0[0, 1] = float("nan")
    p0[1, 0] = float("inf")                            # inf row: inf * 0 in the norm
    R = torch.zeros((2, H), dtype=torch.bfloat16)
    G = torch.ones((H,), dtype=torch.bfloat16)
    P = [p0.cuda(), p1.cuda()]
    out, ro = arf.run(ws, RMS, P, R.cuda(), G.cuda(), 1e-6)
    torch.cuda.synchronize()
    ref = oracle.run(oracle.AR_RESIDUAL_RMSNORM, [wl.codes(p0), wl.codes(p1)], wl.codes(R), wl.codes(G), 1e-6)
    assert bitwise_equal(oracle.BF16, wl.codes(ro.cpu()), ref[1]).all()
    assert bitwise_equal(oracle.BF16, wl.codes(out.cpu()), ref[0]).all()
    assert torch.isnan(ro[0, 0].float()) and torch.isnan(ro[0, 1].float()) and torch.isinf(ro[1, 0].float())


def test_zero_rows_and_eps(ws):
    P = [torch.zeros((3, 64), dtype=torch.bfloat16, device="cuda")] * 2
    R = torch.zeros((3, 64), dtype=torch.bfloat16, device="cuda")
    G = torch.ones((64,), dtype=torch.bfloat16, device="cuda")
    out, _ = arf.run(ws, RMS, P, R, G, 1e-6)
    assert (out.float() == 0).all()
    out, _ = arf.run(ws, RMS, P, R, G, 0.0)  # 0 * rsqrt(0) = 0 * inf = NaN, as the formula says
    assert torch.isnan(out.float()).all()


def test_rejected_calls_write_nothing(ws):
    M, H = 4, 64
    P = [torch.randn((M, H), device="cuda").to(torch.bfloat16) for _ in range(2)]
    R = torch.randn((M, H), device="cuda").to(torch.bfloat16)
    G = torch.ones((H,), device="cuda", dtype=torch.bfloat16)
    ptrs = arf.pointer_array(P)
    out = torch.full((M * H + 8,), 99, dtype=torch.int16, device="cuda")
    ro = torch.full((M * H + 8,), 99, dtype=torch.int16, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    o, r = out.data_ptr(), ro.data_ptr()

    def call(pattern=RMS, W=2, pp=ptrs.data_ptr(), res=R.data_ptr(), g=G.data_ptr(), eps=1e-6, oo=o, rr=r, m=M,
             h=H, dt=arf.ARF_BF16):
        return arf.arf_run(ws.handle, pattern, W, pp, res, g, eps, oo, rr, m, h, dt, s)

    assert call(W=0) == arf.ARF_ERR_UNSUPPORTED
    assert call(W=65) == arf.ARF_ERR_UNSUPPORTED
    assert call(h=0) == arf.ARF_ERR_INVALID_ARG
    assert call(h=-8) == arf.ARF_ERR_INVALID_ARG
    assert call(h=524296) == arf.ARF_ERR_UNSUPPORTED
    assert call(m=-1) == arf.ARF_ERR_INVALID_ARG
    assert call(pp=None) == arf.ARF_ERR_INVALID_ARG
    assert call(res=None) == arf.ARF_ERR_INVALID_ARG
    assert call(g=None) == arf.ARF_ERR_INVALID_ARG
    assert call(rr=None) == arf.ARF_ERR_INVALID_ARG
    assert call(oo=None) == arf.ARF_ERR_INVALID_ARG
    assert call(eps=float("nan")) == arf.ARF_ERR_INVALID_ARG
    assert call(eps=float("inf")) == arf.ARF_ERR_INVALID_ARG
    assert call(eps=-1e-6) == arf.ARF_ERR_INVALID_ARG
    assert call(rr=o) == arf.ARF_ERR_INVALID_ARG                 # out == residual_out
    assert call(oo=o + 1) == arf.ARF_ERR_UNSUPPORTED             # odd address (2-byte offsets run elementwise)
    assert call(rr=r + 9) == arf.ARF_ERR_UNSUPPORTED             # odd residual_out
    assert call(res=R.data_ptr() + 3) == arf.ARF_ERR_UNSUPPORTED
    assert call(pattern=7) == arf.ARF_ERR_INVALID_ARG
    assert call(dt=5) == arf.ARF_ERR_INVALID_ARG
    bad = arf.Plan(path=arf.ARF_PATH_ROW, threads=48, vpt=1, cluster=1, grid=1, w_spec=2)  # not whole warps
    assert arf.arf_run_planned(ws.handle, bad, RMS, 2, ptrs.data_ptr(), R.data_ptr(), G.data_ptr(), 1e-6, o, r, M, H,
                               arf.ARF_BF16, s) == arf.ARF_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert (out == 99).all() and (ro == 99).all()
    assert call() == arf.ARF_OK
    torch.cuda.synchronize()
    assert not (out[:M * H] == 99).all()


def test_device_mismatch_on_wrong_current_device():
    # Only one device is visible: a workspace for a device that does not exist fails cleanly.
    h = ctypes.c_void_p()
    assert arf.arf_workspace_create(torch.cuda.device_count(), h) == arf.ARF_ERR_CUDA
    assert arf.arf_workspace_create(-1, h) == arf.ARF_ERR_CUDA


def test_workspace_churn(ws):
    inp = inputs(2, 4, 64)
    P, R, G = to_device(inp)
    for _ in range(100):
        with arf.Workspace(0) as w:
            out, _ = arf.run(w, AR, P)
    torch.cuda.synchronize()
    assert_parity(oracle.BF16, AR, (wl.codes(out.cpu()), None), oracle_run(AR, inp))


@pytest.mark.parametrize("warm", [True, False])
@pytest.mark.parametrize("pattern", [AR, RMS])
def test_cuda_graph_replay(ws, pattern, warm):
    """Capture once, replay with new values in the same buffers: results
    match the oracle and the inputs are preserved across replays. warm=False:
    the first call for the shape happens under capture."""
    W, M, H = (4, 64, 4096) if warm else (4, 24, 4104)
    first = inputs(W, M, H, cid=910)
    P, R, G = to_device(first)
    ptrs = arf.pointer_array(P)
    out = torch.empty_like(R)
    ro = torch.empty_like(R)
    if warm:  # memoise the plan outside capture
        arf.run(ws, pattern, P, R, G, 1e-6, out=out, residual_out=ro if pattern == RMS else None, ptrs=ptrs)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            arf.run(ws, pattern, P, R, G, 1e-6, out=out, residual_out=ro if pattern == RMS else None, ptrs=ptrs)
    for k in range(3):
        inp = inputs(W, M, H, cid=920 + k)
        for dst, src in zip(P + [R, G], inp.partials + [inp.residual, inp.gamma]):
            dst.copy_(src)
        keep = [t.clone() for t in P + [R, G]]
        g.replay()
        torch.cuda.synchronize()
        got = (wl.codes(out.cpu()), wl.codes(ro.cpu()) if pattern == RMS else None)
        assert_parity(oracle.BF16, pattern, got, oracle_run(pattern, inp), f"replay {k}")
        for a, b in zip(P + [R, G], keep):
            assert torch.equal(a, b)


@pytest.mark.parametrize("pinned", [True, False])
@pytest.mark.parametrize("name,pattern", [("small", RMS), ("llama_tp2", AR), ("llama_tp2", RMS)])
def test_host_buffer_entry_point(ws, name, pattern, pinned):
    w = wl.WORKLOADS[name]
    inp = wl.make_inputs(w)
    pin = (lambda t: t.pin_memory()) if pinned else (lambda t: t.clone())
    P = [pin(p) for p in inp.partials]
    R, G = pin(inp.residual), pin(inp.gamma)
    out = pin(torch.empty_like(inp.residual))
    ro = pin(torch.empty_like(inp.residual))
    runner = arf.HostRunner(ws, pattern, w.W, w.M, w.H, torch.bfloat16)
    for _ in range(2):
        runner(P, R, G, w.eps, out, ro)
        torch.cuda.synchronize()
        got = (wl.codes(out), wl.codes(ro) if pattern == RMS else None)
        assert_parity(DT[w.dtype], pattern, got, oracle_run(pattern, inp))


# Tensors of 8 MiB and more take arf_run_host's pipelined form (one row block
# per 4 MiB, at most 8, rows per block rounded up to a multiple of 8): W = 4,
# M = 1501 gives 5 blocks of 304 rows, the last of 285; tp16_8mib's shape 2
# blocks (296 and 289 rows); H = 4098 (not a multiple of 8) 2 blocks of 552
# and 548 rows.
PIPELINED = [(4, 1501, 7168, "bf16", 0.7), (16, 585, 7168, "fp16", 0.1), (2, 1100, 4098, "bf16", 0.5)]


@pytest.mark.parametrize("W,M,H,dtype,sigma", PIPELINED)
def test_host_buffer_pipelined(ws, W, M, H, dtype, sigma):
    """The pipelined host-buffer form (copies on the workspace's two copy
    streams, kernels per row block on the caller's stream): both patterns
    match the oracle, twice in a row, on a side stream, in place (residual_out
    is the residual buffer) and with out written over the first partial."""
    inp = inputs(W, M, H, dtype, sigma=sigma, cid=910)
    d = DT[dtype]
    tdt = wl.TORCH_DTYPE[dtype]
    P = [p.pin_memory() for p in inp.partials]
    R, G = inp.residual.pin_memory(), inp.gamma.pin_memory()
    side = torch.cuda.Stream()
    for pat in (AR, RMS):
        ref = oracle_run(pat, inp)
        out = torch.empty_like(R).pin_memory()
        ro = torch.empty_like(R).pin_memory()
        runner = arf.HostRunner(ws, pat, W, M, H, tdt)
        for k in range(2):
            out.fill_(0)
            ro.fill_(0)
            runner(P, R, G, 1e-6, out, ro, stream=side)
            side.synchronize()
            got = (wl.codes(out), wl.codes(ro) if pat == RMS else None)
            assert_parity(d, pat, got, ref, f"pipelined call {k}")
    # in place: residual_out written over the residual's host buffer
    Rin = inp.residual.clone().pin_memory()
    out = torch.empty_like(R).pin_memory()
    arf.HostRunner(ws, RMS, W, M, H, tdt)(P, Rin, G, 1e-6, out, Rin)
    torch.cuda.synchronize()
    assert_parity(d, RMS, (wl.codes(out), wl.codes(Rin)), oracle_run(RMS, inp), "pipelined in place")
    # kAllReduce into the first partial's host buffer
    P2 = [p.clone().pin_memory() for p in inp.partials]
    arf.HostRunner(ws, AR, W, M, H, tdt)(P2, None, None, 0.0, P2[0], None)
    torch.cuda.synchronize()
    assert_parity(d, AR, (wl.codes(P2[0]), None), oracle_run(AR, inp), "pipelined out = partial 0")


@pytest.mark.parametrize("pattern", [AR, RMS])
def test_host_buffer_pipelined_pageable(ws, pattern):
    """The pipelined form on pageable (not page-locked) host buffers, where
    the copies may block the calling thread: same results as the oracle."""
    W, M, H = 4, 1501, 7168
    inp = inputs(W, M, H, sigma=0.7, cid=914)
    P = [p.clone() for p in inp.partials]
    R, G = inp.residual.clone(), inp.gamma.clone()
    out, ro = torch.empty_like(R), torch.empty_like(R)
    arf.HostRunner(ws, pattern, W, M, H, torch.bfloat16)(P, R, G, 1e-6, out, ro)
    torch.cuda.synchronize()
    got = (wl.codes(out), wl.codes(ro) if pattern == RMS else None)
    assert_parity(oracle.BF16, pattern, got, oracle_run(pattern, inp), "pipelined, pageable")


def test_host_buffer_pipelined_two_threads(ws):
    """Two host threads drive pipelined calls on one workspace, each on its
    own stream with its own staging and buffers: the workspace's shared copy
    streams and events must not mix one call's ordering with the other's."""
    import threading

    shapes = [(4, 1501, 7168, 0.7, 912), (2, 2400, 4096, 0.5, 913)]
    results, errors = {}, []

    def worker(k, W, M, H, sigma, cid):
        try:
            inp = inputs(W, M, H, sigma=sigma, cid=cid)
            P = [p.pin_memory() for p in inp.partials]
            R, G = inp.residual.pin_memory(), inp.gamma.pin_memory()
            out = torch.empty_like(R).pin_memory()
            ro = torch.empty_like(R).pin_memory()
            runner = arf.HostRunner(ws, RMS, W, M, H, torch.bfloat16)
            s = torch.cuda.Stream()
            got = []
            for _ in range(3):
                out.fill_(0)
                ro.fill_(0)
                runner(P, R, G, 1e-6, out, ro, stream=s)
                s.synchronize()
                got.append((wl.codes(out).copy(), wl.codes(ro).copy()))
            results[k] = (inp, got)
        except Exception as e:  # noqa: BLE001 - reported below
            errors.append(e)

    threads = [threading.Thread(target=worker, args=(k, *sh)) for k, sh in enumerate(shapes)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    for k, (inp, got) in results.items():
        ref = oracle_run(RMS, inp)
        for i, g in enumerate(got):
            assert_parity(oracle.BF16, RMS, g, ref, f"thread {k} call {i}")


def test_host_buffer_pipelined_graph(ws):
    """The pipelined form captured into a CUDA graph (its copy streams fork
    from and join back into the capturing stream) and replayed."""
    W, M, H = 4, 1501, 7168
    inp = inputs(W, M, H, sigma=0.7, cid=911)
    P = [p.pin_memory() for p in inp.partials]
    R, G = inp.residual.pin_memory(), inp.gamma.pin_memory()
    out = torch.empty_like(R).pin_memory()
    ro = torch.empty_like(R).pin_memory()
    runner = arf.HostRunner(ws, RMS, W, M, H, torch.bfloat16)
    runner(P, R, G, 1e-6, out, ro)  # plans the block shapes outside the capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            runner(P, R, G, 1e-6, out, ro, stream=s)
    torch.cuda.synchronize()
    ref = oracle_run(RMS, inp)
    for k in range(2):
        out.fill_(0)
        ro.fill_(0)
        g.replay()
        torch.cuda.synchronize()
        assert_parity(oracle.BF16, RMS, (wl.codes(out), wl.codes(ro)), ref, f"graph replay {k}")


@pytest.mark.parametrize("by_value,pdl", [(True, False), (False, True), (True, True)])
@pytest.mark.parametrize("W,M,H", [(8, 1, 7168), (2, 128, 4096), (8, 300, 7168), (17, 5, 264)])
@pytest.mark.parametrize("pattern", [AR, RMS])
def test_run_ex_options(ws, pattern, W, M, H, by_value, pdl):
    """Partials passed by value and/or a programmatic dependent launch give
    exactly the results of arf_run (same plan), and match the oracle."""
    inp = inputs(W, M, H)
    P, R, G = to_device(inp)
    base = gpu_run(ws, pattern, P, R, G, 1e-6)
    out, ro = arf.run(ws, pattern, P, R, G, 1e-6, by_value=by_value, pdl=pdl)
    torch.cuda.synchronize()
    got = (wl.codes(out.cpu()), wl.codes(ro.cpu()) if pattern == RMS else None)
    assert np.array_equal(got[0], base[0])
    if pattern == RMS:
        assert np.array_equal(got[1], base[1])
    assert_parity(oracle.BF16, pattern, got, oracle_run(pattern, inp))


def test_pdl_dependent_chain(ws):
    """A chain where every call reads the previous call's output: with
    programmatic dependent launches each kernel still waits for its
    predecessor's writes. Checked against the same chain without PDL."""
    M, H = 256, 4096
    a = torch.randn((M, H), device="cuda").to(torch.bfloat16)
    b = torch.randn((M, H), device="cuda").to(torch.bfloat16) * 0.01
    G = torch.ones((H,), device="cuda", dtype=torch.bfloat16)

    def chain(pdl, by_value):
        x = a.clone()
        outs = []
        for k in range(12):
            if k % 2 == 0:
                y, _ = arf.run(ws, AR, [x, b], pdl=pdl, by_value=by_value)
            else:
                y, _ = arf.run(ws, RMS, [x, b], b, G, 1e-6, pdl=pdl, by_value=by_value)
            outs.append(y)
            x = y
        torch.cuda.synchronize()
        return [wl.codes(o.cpu()) for o in outs]

    ref = chain(False, False)
    for pdl, by_value in ((True, False), (True, True)):
        for _ in range(3):
            got = chain(pdl, by_value)
            for k, (g_, r_) in enumerate(zip(got, ref)):
                assert np.array_equal(g_, r_), f"step {k} differs (pdl={pdl}, by_value={by_value})"


def test_pdl_by_value_graph_replay(ws):
    W, M, H = 4, 64, 4096
    inp = inputs(W, M, H, cid=930)
    P, R, G = to_device(inp)
    out, ro = torch.empty_like(R), torch.empty_like(R)
    arf.run(ws, RMS, P, R, G, 1e-6, out=out, residual_out=ro, pdl=True, by_value=True)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    with torch.cuda.graph(g, stream=s):
        for _ in range(3):
            arf.run(ws, RMS, P, R, G, 1e-6, out=out, residual_out=ro, pdl=True, by_value=True)
    for k in range(2):
        new = inputs(W, M, H, cid=940 + k)
        for dst, src in zip(P + [R, G], new.partials + [new.residual, new.gamma]):
            dst.copy_(src)
        g.replay()
        torch.cuda.synchronize()
        assert_parity(oracle.BF16, RMS, (wl.codes(out.cpu()), wl.codes(ro.cpu())), oracle_run(RMS, new))


def test_run_ex_rejects_null_by_value_pointer(ws):
    R = torch.zeros((2, 64), device="cuda", dtype=torch.bfloat16)
    opts = arf.RunOpts(plan=None, partials_by_value=1, pdl=0)
    st = arf.arf_run_ex(ws.handle, opts, AR, 2, [R.data_ptr(), 0], None, None, 0.0, R.data_ptr(), None, 2, 64,
                        arf.ARF_BF16, torch.cuda.current_stream().cuda_stream)
    assert st == arf.ARF_ERR_INVALID_ARG


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_every_code_sums_exactly(ws, dtype):
    """All 65 536 codes (zeros of both signs, subnormals, normals, the
    largest values, infinities, NaNs) pass through the rank sum and the
    residual add exactly as in the oracle: widened exactly, added with one
    binary32 round-to-nearest, rounded once to the I/O type."""
    d = DT[dtype]
    allc = np.arange(65536, dtype=np.uint16).reshape(2, 32768)
    rng = np.random.default_rng(11)
    partner = pins.nearest_codes(d, rng.standard_normal((2, 32768)) * 2.0 ** rng.integers(-30, 12, (2, 32768)))
    cases = [[allc], [allc, partner], [partner, allc, partner[::-1].copy()]]
    for P in cases:
        Pd = [wl.from_codes(p, dtype).cuda() for p in P]
        out, _ = arf.run(ws, AR, Pd)
        ref, _ = oracle.run(oracle.ALLREDUCE, P, dtype=d)
        torch.cuda.synchronize()
        assert bitwise_equal(d, wl.codes(out.cpu()), ref).all(), f"W={len(P)}"
    # every code as the residual
    G = np.full(32768, pins.exact_codes(d, "1")[0], np.uint16)
    Pd = [wl.from_codes(partner, dtype).cuda()]
    out, ro = arf.run(ws, RMS, Pd, wl.from_codes(allc, dtype).cuda(), wl.from_codes(G, dtype).cuda(), 1e-6)
    ref_out, ref_ro = oracle.run(oracle.AR_RESIDUAL_RMSNORM, [partner], allc, G, 1e-6, dtype=d)
    torch.cuda.synchronize()
    assert bitwise_equal(d, wl.codes(ro.cpu()), ref_ro).all()


@pytest.mark.parametrize("name,M", [("small", 8), ("llama_tp2", 128), ("k3_tp8", 64), ("tp16_8mib", 32)])
def test_zero_copy_host_buffers(ws, name, M):
    """arf_run directly on page-locked host buffers (kernels read and write
    host memory in place): same results as on device buffers, in place too."""
    w = wl.WORKLOADS[name].with_m(M)
    inp = wl.make_inputs(w)
    d = DT[w.dtype]
    P = [p.pin_memory() for p in inp.partials]
    R, G = inp.residual.pin_memory(), inp.gamma.pin_memory()
    for pat in (AR, RMS):
        out = torch.empty_like(R).pin_memory()
        ro = torch.empty_like(R).pin_memory()
        runner = arf.HostRunner(ws, pat, w.W, M, w.H, P[0].dtype, zero_copy=True)
        runner(P, R, G, w.eps, out, ro)
        torch.cuda.synchronize()
        got = (wl.codes(out), wl.codes(ro) if pat == RMS else None)
        assert_parity(d, pat, got, oracle_run(pat, inp), f"{name} zero-copy")
    # in place on host memory: residual_out is the residual buffer
    Rin = inp.residual.clone().pin_memory()
    out = torch.empty_like(R).pin_memory()
    HostRunner = arf.HostRunner(ws, RMS, w.W, M, w.H, P[0].dtype, zero_copy=True)
    HostRunner(P, Rin, G, w.eps, out, Rin)
    torch.cuda.synchronize()
    assert_parity(d, RMS, (wl.codes(out), wl.codes(Rin)), oracle_run(RMS, inp), f"{name} zero-copy in place")


@pytest.mark.parametrize("W,M,H,dtype", [(2, 128, 4096, "bf16"), (8, 1, 7168, "bf16"), (3, 37, 1000, "fp16"),
                                         (4, 300, 7168, "bf16"), (2, 5, 13, "bf16")])
@pytest.mark.parametrize("pattern", [AR, RMS])
def test_autotune_memoises_a_legal_plan(pattern, W, M, H, dtype):
    """arf_workspace_autotune picks one of the candidate plans, later calls of
    the shape use it, and results still match the oracle."""
    with arf.Workspace(0) as ws:
        inp = inputs(W, M, H, dtype)
        P, R, G = to_device(inp)
        plan, us = ws.autotune(pattern, P, R, G, inp.workload.eps, reps=5)
        assert us > 0
        caps = ws.caps
        assert arf.arf_plan_check(caps, plan, pattern, W, M, H, DT[dtype]) == arf.ARF_OK
        memo = ws.plan(pattern, W, M, H, wl.TORCH_DTYPE[dtype])
        assert memo.as_dict() == plan.as_dict()
        got = gpu_run(ws, pattern, P, R, G, inp.workload.eps)
        assert_parity(DT[dtype], pattern, got, oracle_run(pattern, inp), f"autotuned {plan}")


@pytest.mark.parametrize("W,M,H,vpt,cs", [(2, 40, 4096, 1, 1), (8, 33, 7168, 2, 1), (1, 9, 16384, 8, 1),
                                          (16, 7, 7168, 1, 2), (4, 12, 8192, 1, 4), (8, 5, 7168, 1, 8)])
def test_one_row_form_matches_the_row_loop(ws, W, M, H, vpt, cs):
    """A grid that gives every cluster one row launches the one-row form; a
    smaller grid of the same CTA shape runs the row loop. Both compute each
    row with the same threads and reduction tree: outputs bitwise equal,
    and both match the oracle."""
    inp = inputs(W, M, H, "bf16", 0.8, cid=990 + W)
    ref = oracle_run(RMS, inp)
    P, R, G = to_device(inp)
    C = H // 8
    threads = max(32, -(-(-(-C // cs) // vpt) // 32) * 32)
    path = arf.ARF_PATH_ROW if cs == 1 else arf.ARF_PATH_CLUSTER
    got = []
    for clusters in (M, max(1, M // 3)):  # one row per cluster; several rows per cluster
        plan = arf.Plan(path=path, threads=threads, vpt=vpt, cluster=cs, grid=clusters * cs, w_spec=W)
        assert arf.arf_plan_check(ws.caps, plan, RMS, W, M, H, arf.ARF_BF16) == arf.ARF_OK, plan
        got.append(gpu_run(ws, RMS, P, R, G, inp.workload.eps, plan=plan))
        assert_parity(oracle.BF16, RMS, got[-1], ref, f"{plan}")
    assert np.array_equal(got[0][0], got[1][0]) and np.array_equal(got[0][1], got[1][1])


def test_read_pass(ws):
    """The read-only measurement pass: reads, writes nothing it was given,
    and checks alignment and size."""
    buf = torch.arange(1 << 20, dtype=torch.int32, device="cuda")
    keep = buf.clone()
    s = torch.cuda.current_stream().cuda_stream
    assert arf.arf_read_pass(ws.handle, buf.data_ptr(), buf.numel() * 4, s) == arf.ARF_OK
    assert arf.arf_read_pass(ws.handle, buf.data_ptr(), 0, s) == arf.ARF_OK
    assert arf.arf_read_pass(ws.handle, buf.data_ptr() + 4, 1024, s) == arf.ARF_ERR_INVALID_ARG
    assert arf.arf_read_pass(ws.handle, buf.data_ptr(), 1000, s) == arf.ARF_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert torch.equal(buf, keep)


@pytest.mark.parametrize("code", [0, 1, 2])
def test_pdl_codes_in_graph(ws, code):
    """arf_run_opts_t.pdl: 0 (the library's choice: on for this decode-size
    call), 1 (always), 2 (never); each, replayed in a CUDA graph, matches the
    oracle; other values are refused."""
    inp = inputs(8, 4, 7168, "bf16")
    P, R, G = to_device(inp)
    ptrs = arf.pointer_array(P)
    out, ro = torch.empty_like(R), torch.empty_like(R)
    opts = arf.RunOpts(plan=None, partials_by_value=0, pdl=code)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())

    def call():
        st = arf.arf_run_ex(ws.handle, opts, RMS, 8, ptrs.data_ptr(), R.data_ptr(), G.data_ptr(), 1e-6,
                            out.data_ptr(), ro.data_ptr(), 4, 7168, arf.ARF_BF16, s.cuda_stream)
        assert st == arf.ARF_OK, arf.arf_status_string(st)

    with torch.cuda.stream(s):
        call()  # plan made outside the capture
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            for _ in range(3):
                call()
    out.zero_()
    ro.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert_parity(DT["bf16"], RMS, (wl.codes(out.cpu()), wl.codes(ro.cpu())), oracle_run(RMS, inp), f"pdl={code}")
    bad = arf.RunOpts(plan=None, partials_by_value=0, pdl=3)
    st = arf.arf_run_ex(ws.handle, bad, RMS, 8, ptrs.data_ptr(), R.data_ptr(), G.data_ptr(), 1e-6, out.data_ptr(),
                        ro.data_ptr(), 4, 7168, arf.ARF_BF16, torch.cuda.current_stream().cuda_stream)
    assert st == arf.ARF_ERR_INVALID_ARG
