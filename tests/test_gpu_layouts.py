"""General layouts on the GPU against the oracle's general entry point:
H not a multiple of 8 (elementwise kernels), row strides (16-byte kernels
when they are multiples of 8 elements, elementwise otherwise), tensors only
2-byte aligned, binary32 partials, and explicit elementwise plans."""
import ctypes

import numpy as np
import pytest
import torch

import all_reduce_residual_gb300 as arf
import oracle
import pins
from all_reduce_residual_gb300 import workloads as wl
from gpu_util import DT, assert_parity

pytestmark = pytest.mark.gpu
RMS, AR = arf.ARF_AR_RESIDUAL_RMSNORM, arf.ARF_ALLREDUCE
OPAT = {AR: oracle.ALLREDUCE, RMS: oracle.AR_RESIDUAL_RMSNORM}


@pytest.fixture(scope="module")
def ws():
    with arf.Workspace(0) as w:
        yield w


def codes_of(rng, d, shape, sigma):
    return pins.nearest_codes(d, rng.standard_normal(shape) * sigma)


def embed(a, pad, fill, dtype):
    """A CUDA [M,H] view with row stride H+pad of a wider buffer (padding = fill)."""
    M, H = a.shape
    big = np.full((M, H + pad), fill, dtype=a.dtype)
    big[:, :H] = a
    if a.dtype == np.float32:
        t = torch.from_numpy(big).cuda()
    else:
        t = wl.from_codes(big, dtype).cuda()
    return t[:, :H], t


def host_codes(t):
    return wl.codes(t.cpu().contiguous())


def run_case(ws, pattern, dtype, W, M, H, pads=(0, 0, 0, 0), f32p=False, plan=None, seed=0):
    d = DT[dtype]
    rng = np.random.default_rng(seed)
    if f32p:
        P = [(rng.standard_normal((M, H)) * 2.0 ** rng.uniform(-4, 6)).astype(np.float32) for _ in range(W)]
    else:
        P = [codes_of(rng, d, (M, H), 1.5) for _ in range(W)]
    R = codes_of(rng, d, (M, H), 1.0)
    G = pins.nearest_codes(d, 0.5 + rng.random(H))
    junk = np.float32(np.nan) if f32p else np.uint16(0x7FC1)
    Pd, Pbig = zip(*[embed(p, pads[0], junk, dtype) for p in P])
    # all partials share one row stride
    Rd, _ = embed(R, pads[1], np.uint16(0x7FC1), dtype)
    Od, Ob = embed(np.zeros((M, H), np.uint16), pads[2], np.uint16(0x1234), dtype)
    ROd, ROb = embed(np.zeros((M, H), np.uint16), pads[3], np.uint16(0x1234), dtype)
    Gd = wl.from_codes(G, dtype).cuda()
    rms = pattern == RMS
    arf.run(ws, pattern, list(Pd), Rd if rms else None, Gd if rms else None, 1e-6, out=Od,
            residual_out=ROd if rms else None, plan=plan)
    torch.cuda.synchronize()
    ref = oracle.run_general(OPAT[pattern], P, R if rms else None, G if rms else None, 1e-6, dtype=d)
    got = (host_codes(Od), host_codes(ROd) if rms else None)
    assert_parity(d, pattern, got, ref, f"{dtype} W={W} M={M} H={H} pads={pads} f32p={f32p} plan={plan}")
    # the outputs' row padding is untouched
    for big in (Ob,) + ((ROb,) if rms else ()):
        pad = host_codes(big)[:, H:]
        assert (pad == 0x1234).all(), "wrote outside the rows"


@pytest.mark.parametrize("H", [1, 3, 7, 13, 1001, 4099, 7170])
@pytest.mark.parametrize("W", [1, 2, 3, 8])
@pytest.mark.parametrize("pattern", [AR, RMS])
def test_h_not_multiple_of_8(ws, pattern, W, H):
    run_case(ws, pattern, "bf16" if H % 2 else "fp16", W, 5, H, seed=H + W)


@pytest.mark.parametrize("pads", [(8, 16, 24, 8), (3, 1, 5, 7), (0, 0, 8, 0), (8, 8, 8, 8), (0, 2, 0, 1)])
@pytest.mark.parametrize("H", [64, 4096, 7168])
@pytest.mark.parametrize("pattern", [AR, RMS])
def test_row_strides(ws, pattern, H, pads):
    run_case(ws, pattern, "bf16", 4, 37, H, pads=pads, seed=H)


@pytest.mark.parametrize("H,pads", [(4098, (6, 6, 6, 6)), (1001, (4, 4, 4, 4)), (7170, (6, 14, 22, 30)),
                                    (13, (8, 0, 0, 8)), (64, (3, 3, 3, 3)), (4096, (1, 9, 17, 1))])
@pytest.mark.parametrize("pattern", [AR, RMS])
def test_strided_rows_vector_form(ws, pattern, H, pads):
    """Row strides congruent modulo 8 (every tensor's row r starts at the same
    offset within a 16-byte vector) take the elementwise kernels' 16-byte
    form row by row, with heads that differ from row to row where the
    stride is not a multiple of 8; padding stays untouched. Planner plans and
    explicit ones with the narrowest and widest CTAs."""
    for i, W in enumerate((1, 2, 3, 4, 8)):
        dtype = "bf16" if i % 2 == 0 else "fp16"
        run_case(ws, pattern, dtype, W, 37, H, pads=pads, seed=H + W)
        for threads, grid in ((32, 5), (512, 64)):
            plan = arf.Plan(path=arf.ARF_PATH_ELEM, threads=threads, vpt=1, cluster=1, grid=grid, w_spec=0)
            run_case(ws, pattern, dtype, W, 37, H, pads=pads, plan=plan, seed=H + W + threads)


@pytest.mark.parametrize("case", range(45))
def test_fuzz_elementwise_layouts(ws, case):
    """Seeded random layouts against the oracle: contiguous tensors, row
    strides congruent modulo 8 (the vector forms) or arbitrary (one element
    per thread), any H, compiled and run-time rank counts, and the planner's
    plan or a random elementwise one."""
    rng = np.random.default_rng(7000 + case)
    W = int(rng.choice([1, 2, 3, 4, 5, 8, 16, 17]))
    M = int(rng.choice([1, 2, 7, 33, 150]))
    H = int(rng.integers(1, 9000))
    H = max(1, min(H, 3_000_000 // (M * W)))
    kind = case % 3
    if kind == 0:
        pads = (0, 0, 0, 0)
    elif kind == 1:
        base = int(rng.integers(0, 8))
        pads = tuple(base + 8 * int(rng.integers(0, 3)) for _ in range(4))
    else:
        pads = tuple(int(rng.integers(0, 20)) for _ in range(4))
    plan = None
    if rng.random() < 0.5:
        plan = arf.Plan(path=arf.ARF_PATH_ELEM, threads=32 * int(rng.integers(1, 17)), vpt=1, cluster=1,
                        grid=int(rng.integers(1, 2000)), w_spec=0)
    pattern = AR if rng.random() < 0.4 else RMS
    dtype = "bf16" if rng.random() < 0.5 else "fp16"
    run_case(ws, pattern, dtype, W, M, H, pads=pads, plan=plan, seed=7000 + case)


@pytest.mark.parametrize("W", [1, 2, 3, 8, 17])
@pytest.mark.parametrize("M,H", [(1, 8), (37, 4096), (300, 7168), (5, 13), (2, 65536)])
@pytest.mark.parametrize("pattern", [AR, RMS])
def test_f32_partials(ws, pattern, W, M, H):
    run_case(ws, pattern, "bf16" if W % 2 else "fp16", W, M, H, f32p=True, seed=W * 7 + M)


def test_f32_partials_strided(ws):
    for pattern in (AR, RMS):
        run_case(ws, pattern, "bf16", 3, 20, 1024, pads=(8, 8, 16, 8), f32p=True, seed=3)
        run_case(ws, pattern, "fp16", 3, 20, 1000, pads=(3, 5, 1, 2), f32p=True, seed=4)


@pytest.mark.parametrize("M,H", [(3, 8), (40, 7168), (2, 65536)])
@pytest.mark.parametrize("pattern", [AR, RMS])
def test_explicit_elementwise_plans(ws, pattern, M, H):
    for threads in (32, 256, 512):
        for grid in (1, 7, 300):
            plan = arf.Plan(path=arf.ARF_PATH_ELEM, threads=threads, vpt=1, cluster=1, grid=grid, w_spec=0)
            run_case(ws, pattern, "fp16", 3, M, H, plan=plan, seed=threads + grid)


@pytest.mark.parametrize("W", [1, 2, 4, 8, 5])
def test_odd_h_in_place(ws, W):
    """residual_out == residual on the elementwise kernels' vector form (each
    thread reads a chunk of the residual before it writes the same chunk,
    two chunks per trip for W <= 2), against the oracle."""
    from gpu_util import gpu_run, oracle_run, to_device
    inp = wl.make_inputs(wl.custom(W, 300, 4098, "bf16" if W % 2 == 0 else "fp16", 0.7, 1e-6, config_id=4100 + W))
    P, R, G = to_device(inp)
    got = gpu_run(ws, RMS, P, R, G, inp.workload.eps, in_place=True)
    assert_parity(DT[inp.workload.dtype], RMS, got, oracle_run(RMS, inp), f"W={W}")
    assert ws.plan(RMS, W, 300, 4098, P[0].dtype).path == arf.ARF_PATH_ELEM


@pytest.mark.parametrize("ld", [4098, 4104])
@pytest.mark.parametrize("g_off", [0, 1])
def test_vector_form_gamma_alignment(ws, ld, g_off):
    """kARResidualRMSNorm's vector form with H = 4098: rows whose chunks start
    on a 16-byte boundary (every row at ld = 4104, one in four contiguous)
    load gamma as 16-byte vectors when gamma is aligned, element by element
    when it sits at a 2-byte offset (g_off = 1); all match the oracle."""
    M, H, W = 41, 4098, 2
    rng = np.random.default_rng(ld + g_off)
    P = [codes_of(rng, oracle.BF16, (M, H), 1.0) for _ in range(W)]
    R = codes_of(rng, oracle.BF16, (M, H), 1.0)
    G = pins.nearest_codes(oracle.BF16, 0.5 + rng.random(H))
    pad = ld - H
    Pd = [embed(p, pad, np.uint16(0x7FC1), "bf16")[0] for p in P]
    Rd, _ = embed(R, pad, np.uint16(0x7FC1), "bf16")
    Od, _ = embed(np.zeros((M, H), np.uint16), pad, np.uint16(0x1234), "bf16")
    ROd, _ = embed(np.zeros((M, H), np.uint16), pad, np.uint16(0x1234), "bf16")
    gbuf = torch.zeros(H + 8, dtype=torch.int16, device="cuda")
    Gd = gbuf[g_off:g_off + H].view(torch.bfloat16)
    Gd.copy_(wl.from_codes(G, "bf16").cuda())
    arf.run(ws, RMS, Pd, Rd, Gd, 1e-6, out=Od, residual_out=ROd)
    torch.cuda.synchronize()
    ref = oracle.run_general(oracle.AR_RESIDUAL_RMSNORM, P, R, G, 1e-6, dtype=oracle.BF16)
    assert_parity(oracle.BF16, RMS, (host_codes(Od), host_codes(ROd)), ref, f"ld={ld} g_off={g_off}")


def test_two_byte_aligned_tensors(ws):
    """out / residual / gamma / residual_out at 2-byte (not 16-byte) offsets:
    the elementwise kernels; an odd address is refused."""
    M, H, W = 9, 256, 3
    rng = np.random.default_rng(9)
    P = [codes_of(rng, oracle.BF16, (M, H), 1.0) for _ in range(W)]
    R = codes_of(rng, oracle.BF16, (M, H), 1.0)
    G = pins.nearest_codes(oracle.BF16, 0.5 + rng.random(H))
    Pd = [wl.from_codes(p, "bf16").cuda() for p in P]
    buf = torch.zeros(4 * M * H + 64, dtype=torch.int16, device="cuda")
    Rd = buf[1:1 + M * H].view(torch.bfloat16).view(M, H)
    Rd.copy_(wl.from_codes(R, "bf16").cuda())
    Gd = buf[M * H + 3:M * H + 3 + H].view(torch.bfloat16)
    Gd.copy_(wl.from_codes(G, "bf16").cuda())
    Od = buf[2 * M * H + 5:3 * M * H + 5].view(torch.bfloat16).view(M, H)
    ROd = buf[3 * M * H + 7:4 * M * H + 7].view(torch.bfloat16).view(M, H)
    arf.run(ws, RMS, Pd, Rd, Gd, 1e-6, out=Od, residual_out=ROd)
    torch.cuda.synchronize()
    ref = oracle.run(oracle.AR_RESIDUAL_RMSNORM, P, R, G, 1e-6, dtype=oracle.BF16)
    assert_parity(oracle.BF16, RMS, (host_codes(Od), host_codes(ROd)), ref)
    ptrs = arf.pointer_array(Pd)
    st = arf.arf_run(ws.handle, RMS, W, ptrs.data_ptr(), Rd.data_ptr(), Gd.data_ptr(), 1e-6, Od.data_ptr() + 1,
                     ROd.data_ptr(), M, H, arf.ARF_BF16, torch.cuda.current_stream().cuda_stream)
    assert st == arf.ARF_ERR_UNSUPPORTED


def test_layout_argument_errors(ws):
    M, H = 4, 64
    P = [torch.zeros((M, H), dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    R = torch.zeros((M, H), dtype=torch.bfloat16, device="cuda")
    G = torch.ones((H,), dtype=torch.bfloat16, device="cuda")
    out = torch.empty_like(R)
    ptrs = arf.pointer_array(P)
    s = torch.cuda.current_stream().cuda_stream

    def call(**kw):
        o = arf.RunOpts(plan=None, partials_by_value=0, pdl=0, **kw)
        return arf.arf_run_ex(ws.handle, o, RMS, 2, ptrs.data_ptr(), R.data_ptr(), G.data_ptr(), 1e-6,
                              out.data_ptr(), R.data_ptr(), M, H, arf.ARF_BF16, s)

    assert call(ld_partials=32) == arf.ARF_ERR_INVALID_ARG          # stride below H
    assert call(ld_partials=(1 << 38) + 8) == arf.ARF_ERR_UNSUPPORTED  # M x stride above 2^40
    assert call(ld_out=1 << 62) == arf.ARF_ERR_UNSUPPORTED
    assert call(ld_residual=72, ld_residual_out=80) == arf.ARF_ERR_INVALID_ARG  # in place, strides differ
    assert call() == arf.ARF_OK                                      # in place, equal strides
    plan = arf.Plan(path=arf.ARF_PATH_ROW, threads=32, vpt=2, cluster=1, grid=4, w_spec=2)
    o = arf.RunOpts(plan=ctypes.pointer(plan), partials_by_value=0, pdl=0, partials_f32=1)
    # an explicit run-time-W plan is needed for binary32 partials
    assert arf.arf_run_ex(ws.handle, o, RMS, 2, ptrs.data_ptr(), R.data_ptr(), G.data_ptr(), 1e-6,
                          out.data_ptr(), R.data_ptr(), M, H, arf.ARF_BF16, s) == arf.ARF_ERR_UNSUPPORTED
    torch.cuda.synchronize()


@pytest.mark.parametrize("W", [2, 3, 4])
@pytest.mark.parametrize("M,H", [(5, 13), (64, 7170), (3, 1), (7, 1001), (2, 24579)])
@pytest.mark.parametrize("misaligned", [False, True])
@pytest.mark.parametrize("pattern", [AR, RMS])
def test_odd_h_flat_range(ws, pattern, M, H, misaligned, W):
    """Contiguous tensors with H % 8 != 0: the whole tensor is one flat range
    (kAllReduce: 16-byte body and elementwise tail; kARResidualRMSNorm: each
    row's aligned chunks with an elementwise head and tail) when every partial
    pointer is 16-byte aligned, and plain elementwise when one is only 2-byte
    aligned. Both match the oracle, with the rank count compiled in (W = 2, 4)
    or not (W = 3)."""
    rng = np.random.default_rng(M * 7 + H + W)
    P = [codes_of(rng, oracle.BF16, (M, H), 1.0) for _ in range(W)]
    R = codes_of(rng, oracle.BF16, (M, H), 1.0)
    G = pins.nearest_codes(oracle.BF16, 0.5 + rng.random(H))
    bufs = [torch.zeros(M * H + 8, dtype=torch.int16, device="cuda") for _ in range(W)]
    Pd = []
    for r, (b, p) in enumerate(zip(bufs, P)):
        off = 1 if (misaligned and r == 1) else 0
        v = b[off:off + M * H].view(torch.bfloat16).view(M, H)
        v.copy_(wl.from_codes(p, "bf16").cuda())
        Pd.append(v)
    Rd = wl.from_codes(R, "bf16").cuda()
    Gd = wl.from_codes(G, "bf16").cuda()
    rms = pattern == RMS
    out, ro = arf.run(ws, pattern, Pd, Rd if rms else None, Gd if rms else None, 1e-6)
    torch.cuda.synchronize()
    ref = oracle.run(OPAT[pattern], P, R if rms else None, G if rms else None, 1e-6, dtype=oracle.BF16)
    got = (host_codes(out), host_codes(ro) if rms else None)
    assert_parity(oracle.BF16, pattern, got, ref, f"M={M} H={H} misaligned={misaligned}")


@pytest.mark.parametrize("W,M,H", [(2, 4096, 4098), (2, 4, 4098), (4, 8, 7175), (1, 16, 1001), (3, 8, 7170),
                                   (16, 8, 13), (8, 24, 7171)])
def test_flat_range_for_h_not_multiple_of_8(ws, W, M, H):
    """kAllReduce with H % 8 != 0 on the 16-byte flat kernel: contiguous
    tensors whose M * H is a multiple of 8 run as one range of chunks."""
    assert (M * H) % 8 == 0
    wspec = W if W in arf.COMPILED_W else 0
    for t, u in ((128, 1), (256, 2), (512, 4)):
        if (u == 2 and wspec > 8) or (u == 4 and wspec > 4):
            continue
        grid = -(-(M * H // 8) // (t * u))
        plan = arf.Plan(path=arf.ARF_PATH_FLAT, threads=t, vpt=u, cluster=1, grid=grid, w_spec=wspec, stages=0)
        assert arf.arf_plan_check(ws.caps, plan, AR, W, M, H, arf.ARF_BF16) == arf.ARF_OK
        run_case(ws, AR, "bf16", W, M, H, plan=plan, seed=M + t)


def test_flat_range_needs_contiguous_rows_and_whole_chunks(ws):
    """The flat range is refused where M * H is not a multiple of 8, and on
    strided rows (an explicit plan is rejected; the planner's own plan falls
    back to the elementwise kernel)."""
    caps = ws.caps
    plan = arf.Plan(path=arf.ARF_PATH_FLAT, threads=128, vpt=1, cluster=1, grid=11, w_spec=2, stages=0)
    assert arf.arf_plan_check(caps, plan, AR, 2, 3, 4098, arf.ARF_BF16) == arf.ARF_ERR_UNSUPPORTED
    assert arf.arf_plan_check(caps, plan, AR, 2, 4, 4098, arf.ARF_BF16) == arf.ARF_OK
    with pytest.raises(arf.ArfError) as e:
        run_case(ws, AR, "bf16", 2, 4, 4098, pads=(8, 0, 8, 0), plan=plan)
    assert e.value.status == arf.ARF_ERR_UNSUPPORTED
    run_case(ws, AR, "bf16", 2, 4, 4098, pads=(8, 0, 8, 0))  # the planner's plan on the strided rows
