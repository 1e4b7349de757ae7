"""The bulk-copy kARResidualRMSNorm kernel (ARF_PATH_BULK) against the oracle:
explicit plans over rank counts, ring depths, column-block widths (ragged last
blocks included), grids smaller and larger than the row count, in-place
residuals, row strides, and launch options; and its bounded waits: a ring
slot that is never filled makes every CTA give up, count itself, and leave
the context usable."""
import ctypes

import numpy as np
import pytest
import torch

import all_reduce_residual_gb300 as arf
import oracle
import pins
from all_reduce_residual_gb300 import workloads as wl
from gpu_util import DT, assert_parity, gpu_run, oracle_run, to_device

pytestmark = pytest.mark.gpu
RMS, AR = arf.ARF_AR_RESIDUAL_RMSNORM, arf.ARF_ALLREDUCE


@pytest.fixture(scope="module")
def ws():
    with arf.Workspace(0) as w:
        yield w


def bulk(threads, stages, grid, w_spec):
    return arf.Plan(path=arf.ARF_PATH_BULK, threads=threads, vpt=1, cluster=1, grid=grid, w_spec=w_spec,
                    stages=stages)


def legal(ws, plan, W, M, H, dtype="bf16"):
    return arf.arf_plan_check(ws.caps, plan, RMS, W, M, H, arf.dtype_code(wl.TORCH_DTYPE[dtype])) == arf.ARF_OK


def inputs(W, M, H, dtype, seed):
    return wl.make_inputs(wl.custom(W, M, H, dtype, 0.7, 1e-6, config_id=3000 + seed))


@pytest.mark.parametrize("W,M,H,dtype", [(1, 9, 8, "bf16"), (2, 37, 1000, "bf16"), (3, 5, 7168, "fp16"),
                                         (8, 41, 7176, "bf16"), (16, 23, 7168, "fp16"), (16, 3, 4096, "bf16"),
                                         (17, 6, 2056, "fp16"), (64, 2, 256, "bf16"), (4, 300, 264, "fp16"),
                                         (4, 2, 32768, "bf16"), (2, 5, 32776, "bf16"), (8, 3, 65536, "fp16"),
                                         (12, 11, 7168, "fp16")])
def test_bulk_plans(ws, W, M, H, dtype):
    inp = inputs(W, M, H, dtype, W * 131 + M)
    ref = oracle_run(RMS, inp)
    P, R, G = to_device(inp)
    w_specs = sorted({0, W if W in arf.COMPILED_W else 0})
    ran = 0
    for threads in (32, 128, 256, 512):
        for stages in (2, 3, 6, 16):
            for grid in sorted({1, 7, M, 2 * M + 1}):
                for w_spec in w_specs:
                    plan = bulk(threads, stages, grid, w_spec)
                    if not legal(ws, plan, W, M, H, dtype):
                        continue
                    got = gpu_run(ws, RMS, P, R, G, inp.workload.eps, plan=plan)
                    assert_parity(DT[dtype], RMS, got, ref, f"{plan}")
                    ran += 1
    assert ran > 0


def test_bulk_in_place_and_options(ws):
    W, M, H = 16, 40, 7168
    inp = inputs(W, M, H, "fp16", 7)
    ref = oracle_run(RMS, inp)
    P, R, G = to_device(inp)
    plan = bulk(128, 4, 19, 16)
    assert legal(ws, plan, W, M, H, "fp16")
    assert_parity(oracle.FP16, RMS, gpu_run(ws, RMS, P, R, G, inp.workload.eps, plan=plan, in_place=True), ref,
                  "in place")
    for by_value, pdl in ((True, False), (False, True), (True, True)):
        out, ro = arf.run(ws, RMS, P, R, G, inp.workload.eps, plan=plan, by_value=by_value, pdl=pdl)
        torch.cuda.synchronize()
        got = (wl.codes(out.cpu()), wl.codes(ro.cpu()))
        assert_parity(oracle.FP16, RMS, got, ref, f"by_value={by_value} pdl={pdl}")


@pytest.mark.parametrize("pads", [(8, 16, 24, 8), (0, 8, 0, 0), (64, 0, 8, 16)])
def test_bulk_row_strides(ws, pads):
    W, M, H = 4, 33, 4096
    rng = np.random.default_rng(sum(pads))
    d = oracle.BF16
    Pc = [pins.nearest_codes(d, rng.standard_normal((M, H)) * 1.5) for _ in range(W)]
    Rc = pins.nearest_codes(d, rng.standard_normal((M, H)))
    Gc = pins.nearest_codes(d, 0.5 + rng.random(H))

    def strided(codes, pad, fill=0x7FC1):
        big = np.full((M, H + pad), fill, np.uint16)
        big[:, :H] = codes
        t = wl.from_codes(big, "bf16").cuda()
        return t[:, :H], t

    Pd = [strided(p, pads[0])[0] for p in Pc]
    Rd = strided(Rc, pads[1])[0]
    Od, Ob = strided(np.zeros((M, H), np.uint16), pads[2], 0x1234)
    ROd, ROb = strided(np.zeros((M, H), np.uint16), pads[3], 0x1234)
    G = wl.from_codes(Gc, "bf16").cuda()
    arf.run(ws, RMS, Pd, Rd, G, 1e-6, out=Od, residual_out=ROd, plan=bulk(256, 3, 10, 4))
    torch.cuda.synchronize()
    ref = oracle.run(oracle.AR_RESIDUAL_RMSNORM, Pc, Rc, Gc, 1e-6, dtype=d)
    got = (wl.codes(Od.cpu().contiguous()), wl.codes(ROd.cpu().contiguous()))
    assert_parity(d, RMS, got, ref, f"pads={pads}")
    for big in (Ob, ROb):
        assert (wl.codes(big.cpu())[:, H:] == 0x1234).all(), "wrote outside the rows"


def test_bulk_refuses_binary32_partials(ws):
    M, H = 4, 64
    P = [torch.zeros((M, H), dtype=torch.float32, device="cuda") for _ in range(2)]
    R = torch.zeros((M, H), dtype=torch.bfloat16, device="cuda")
    G = torch.ones((H,), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(arf.ArfError) as e:
        arf.run(ws, RMS, P, R, G, 1e-6, plan=bulk(32, 2, 4, 0))
    assert e.value.status == arf.ARF_ERR_UNSUPPORTED


def run_opts_call(ws, P, R, G, out, ro, plan, **kw):
    ptrs = arf.pointer_array(P)
    M, H = R.shape
    o = arf.RunOpts(plan=ctypes.pointer(plan), **kw)
    st = arf.arf_run_ex(ws.handle, o, RMS, len(P), ptrs.data_ptr(), R.data_ptr(), G.data_ptr(), 1e-6,
                        out.data_ptr(), ro.data_ptr(), M, H, arf.ARF_BF16, torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    return st


def timeouts(ws):
    n = ctypes.c_uint(12345)
    assert arf.arf_workspace_wait_timeouts(ws.handle, n) == arf.ARF_OK
    return n.value


def test_bulk_wait_gives_up_and_context_survives(ws):
    """Every CTA leaves its first slot unfilled (hold_first_copy), so its first
    wait runs out after wait_limit_cycles (about a millisecond here): each CTA
    that owns rows counts itself once, and the next ordinary call is exact."""
    W, M, H = 8, 24, 7168
    inp = inputs(W, M, H, "bf16", 11)
    ref = oracle_run(RMS, inp)
    P, R, G = to_device(inp)
    out, ro = torch.empty_like(R), torch.empty_like(R)
    assert timeouts(ws) == 0
    grid = 40  # 24 CTAs own rows, 16 own none and never wait
    plan = bulk(128, 4, grid, 8)
    st = run_opts_call(ws, P, R, G, out, ro, plan, wait_limit_cycles=2_000_000, hold_first_copy=1)
    assert st == arf.ARF_OK
    assert timeouts(ws) == M
    assert timeouts(ws) == 0  # read-and-reset
    st = run_opts_call(ws, P, R, G, out, ro, plan, wait_limit_cycles=2_000_000)
    assert st == arf.ARF_OK
    assert timeouts(ws) == 0
    assert_parity(oracle.BF16, RMS, (wl.codes(out.cpu()), wl.codes(ro.cpu())), ref, "after the timeout")


@pytest.mark.parametrize("case", range(30))
def test_bulk_fuzz(ws, case):
    """Random rank counts, shapes, dtypes and legal bulk plans (any block width,
    ring depth and grid), half of them in place; no wait may give up."""
    rng = np.random.default_rng(5000 + case)
    W = int(rng.choice([1, 2, 3, 4, 6, 8, 12, 16, 24, 33, 64]))
    M = int(rng.choice([1, 3, 17, 150, 301]))
    H = 8 * int(rng.choice([1, 5, 64, 130, 513, 896, 2048]))
    dtype = str(rng.choice(["bf16", "fp16"]))
    inp = wl.make_inputs(wl.custom(W, M, H, dtype, float(rng.choice([0.01, 1.0, 30.0])), 1e-6, config_id=6000 + case))
    for _ in range(100):
        plan = bulk(int(rng.choice([32, 64, 96, 128, 256, 384, 512])), int(rng.integers(2, 17)),
                    int(rng.integers(1, 700)), int(rng.choice([0, W])) if W in arf.COMPILED_W else 0)
        if legal(ws, plan, W, M, H, dtype):
            break
    else:
        pytest.skip("no legal bulk plan drawn for this shape")
    P, R, G = to_device(inp)
    try:
        got = gpu_run(ws, RMS, P, R, G, inp.workload.eps, plan=plan, in_place=bool(case % 2))
    except arf.ArfError as e:  # legal by the rules, but more shared memory than this device lets it have
        assert e.status == arf.ARF_ERR_UNSUPPORTED
        return
    assert_parity(DT[dtype], RMS, got, oracle_run(RMS, inp), f"case {case}: W={W} M={M} H={H} {dtype} {plan}")
    assert timeouts(ws) == 0


@pytest.mark.parametrize("warm", [True, False])
def test_bulk_graph_replay(ws, warm):
    """A shape the planner sends to the bulk kernel (W = 3, no compiled rank
    count), captured in a CUDA graph and replayed with new values in the same
    buffers; warm=False makes the first call for the shape under capture."""
    W, M, H = (3, 300, 7168) if warm else (3, 301, 7168)
    P, R, G = to_device(inputs(W, M, H, "bf16", 40 + warm))
    assert ws.plan(RMS, W, M, H, torch.bfloat16).path == arf.ARF_PATH_BULK
    ptrs = arf.pointer_array(P)
    out, ro = torch.empty_like(R), torch.empty_like(R)
    if warm:
        arf.run(ws, RMS, P, R, G, 1e-6, out=out, residual_out=ro, ptrs=ptrs)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            arf.run(ws, RMS, P, R, G, 1e-6, out=out, residual_out=ro, ptrs=ptrs)
    for k in range(3):
        inp = inputs(W, M, H, "bf16", 50 + k)
        for dst, src in zip(P + [R, G], inp.partials + [inp.residual, inp.gamma]):
            dst.copy_(src)
        g.replay()
        torch.cuda.synchronize()
        ref = oracle.run(oracle.AR_RESIDUAL_RMSNORM, [wl.codes(p) for p in inp.partials], wl.codes(inp.residual),
                         wl.codes(inp.gamma), 1e-6, dtype=oracle.BF16)
        assert_parity(oracle.BF16, RMS, (wl.codes(out.cpu()), wl.codes(ro.cpu())), ref, f"replay {k}")
    assert timeouts(ws) == 0


def test_bulk_pdl_chain(ws):
    """Bulk-kernel calls chained through their outputs, with programmatic
    dependent launches: each waits for its predecessor's writes before its
    first copy. Bitwise equal to the same chain without PDL."""
    M, H = 200, 7168
    base = [torch.randn((M, H), device="cuda").to(torch.bfloat16) for _ in range(3)]
    G = torch.ones((H,), device="cuda", dtype=torch.bfloat16)
    R = torch.randn((M, H), device="cuda").to(torch.bfloat16)

    def chain(pdl):
        x = base[0].clone()
        outs = []
        for _ in range(8):
            y, _ = arf.run(ws, RMS, [x, base[1], base[2]], R, G, 1e-6, pdl=pdl)
            outs.append(y)
            x = y
        torch.cuda.synchronize()
        return [wl.codes(o.cpu()) for o in outs]

    assert ws.plan(RMS, 3, M, H, torch.bfloat16).path == arf.ARF_PATH_BULK
    ref = chain(False)
    for _ in range(3):
        for k, (a, b) in enumerate(zip(chain(True), ref)):
            assert np.array_equal(a, b), f"step {k} differs under PDL"


@pytest.mark.parametrize("W,M,H,dtype", [(1, 9, 8, "bf16"), (2, 37, 1000, "fp16"), (3, 5, 7168, "bf16"),
                                         (8, 41, 7176, "bf16"), (16, 23, 7168, "fp16"), (64, 2, 256, "bf16"),
                                         (4, 300, 264, "fp16"), (12, 7, 1000, "bf16")])
def test_bulk_allreduce_plans(ws, W, M, H, dtype):
    """The kAllReduce form of the bulk kernel: bitwise equal to the oracle for
    every block width, ring depth and grid drawn."""
    inp = inputs(W, M, H, dtype, 700 + W)
    ref = oracle_run(AR, inp)
    P, R, G = to_device(inp)
    ran = 0
    for threads in (32, 128, 512):
        for stages in (2, 5, 16):
            for grid in sorted({1, 7, M, 2 * M + 1}):
                for w_spec in sorted({0, W if W in arf.COMPILED_W else 0}):
                    plan = bulk(threads, stages, grid, w_spec)
                    if arf.arf_plan_check(ws.caps, plan, AR, W, M, H, arf.dtype_code(wl.TORCH_DTYPE[dtype])) != 0:
                        continue
                    assert_parity(DT[dtype], AR, gpu_run(ws, AR, P, R, G, 1e-6, plan=plan), ref, f"{plan}")
                    ran += 1
    assert ran > 0 and timeouts(ws) == 0
