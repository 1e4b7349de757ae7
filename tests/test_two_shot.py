"""The row-sharded two-shot form on the host: two gloo ranks, each holding
its own partial, with the CPU oracle as the local step. Every rank must end
with exactly the oracle's one-call result on the whole problem (residual_out,
out and the all-reduce bitwise: the partition changes no row's arithmetic),
for ragged row counts, fewer rows than ranks, and both patterns."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

import oracle
from all_reduce_residual_gb300 import two_shot as ts
from all_reduce_residual_gb300 import workloads as wl

DT = {"bf16": oracle.BF16, "fp16": oracle.FP16}


def test_row_blocks_cover_in_order():
    for M in (0, 1, 2, 5, 7, 8, 585, 5851):
        for G in (1, 2, 3, 4, 8, 16):
            b = ts.row_blocks(M, G)
            assert len(b) == G
            assert b[0][0] == 0 and b[-1][1] == M
            for (a0, a1), (c0, c1) in zip(b, b[1:]):
                assert a1 == c0 and a0 <= a1
            sizes = [m1 - m0 for m0, m1 in b]
            assert max(sizes) == -(-M // G) if M else max(sizes) == 0
    with pytest.raises(ValueError):
        ts.row_blocks(4, 0)


def _oracle_epilogue(dtype):
    """The local step on host tensors, computed by the oracle."""
    def step(pattern, partials, residual, gamma, eps):
        P = [wl.codes(p) for p in partials]
        if pattern == 0:
            o, _ = oracle.run(oracle.ALLREDUCE, P, dtype=DT[dtype])
            return wl.from_codes(o, dtype), None
        o, ro = oracle.run(oracle.AR_RESIDUAL_RMSNORM, P, wl.codes(residual), wl.codes(gamma), eps, dtype=DT[dtype])
        return wl.from_codes(o, dtype), wl.from_codes(ro, dtype)
    return step


def _rank(rank, world, port, cases, q):
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        for W, M, H, dtype, pattern in cases:
            w = wl.custom(W, M, H, dtype, 1.0, 1e-6, config_id=970 + M)
            inp = wl.make_inputs(w)
            out, ro = ts.two_shot(pattern, inp.partials[rank], inp.residual, inp.gamma, w.eps,
                                  epilogue=_oracle_epilogue(dtype))
            q.put((rank, (W, M, H, dtype, pattern), wl.codes(out), None if ro is None else wl.codes(ro)))
    finally:
        dist.destroy_process_group()


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def test_two_ranks_reproduce_the_one_call_result():
    world = 2
    cases = [(2, 7, 64, "bf16", "rmsnorm"), (2, 7, 64, "bf16", "allreduce"), (2, 1, 40, "fp16", "rmsnorm"),
             (2, 8, 1024, "bf16", "rmsnorm"), (2, 5, 24, "fp16", "allreduce")]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, world, port, cases, q)) for r in range(world)]
    for p in procs:
        p.start()
    got = [q.get(timeout=240) for _ in range(world * len(cases))]
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    for rank, (W, M, H, dtype, pattern), out, ro in got:
        w = wl.custom(W, M, H, dtype, 1.0, 1e-6, config_id=970 + M)
        inp = wl.make_inputs(w)
        P = [wl.codes(p) for p in inp.partials]
        if pattern == "allreduce":
            ref_out, _ = oracle.run(oracle.ALLREDUCE, P, dtype=DT[dtype])
            assert np.array_equal(out, ref_out), (rank, W, M, H, dtype, pattern)
        else:
            ref_out, ref_ro = oracle.run(oracle.AR_RESIDUAL_RMSNORM, P, wl.codes(inp.residual),
                                         wl.codes(inp.gamma), w.eps, dtype=DT[dtype])
            assert np.array_equal(ro, ref_ro), (rank, W, M, H, dtype, pattern)
            assert np.array_equal(out, ref_out), (rank, W, M, H, dtype, pattern)


@pytest.mark.gpu
@pytest.mark.parametrize("pattern", ["allreduce", "rmsnorm"])
def test_one_rank_on_the_gpu_matches_the_oracle(pattern):
    """G = 1: the two-shot form is the library call on the whole problem."""
    import all_reduce_residual_gb300 as arf
    from gpu_util import DT as GDT, assert_parity, oracle_run

    w = wl.custom(1, 37, 7168, "bf16", 1.0, 1e-6, config_id=990)
    inp = wl.make_inputs(w)
    with arf.Workspace(0) as ws:
        out, ro = ts.two_shot(pattern, inp.partials[0].cuda(), inp.residual.cuda(), inp.gamma.cuda(), w.eps, ws=ws)
        torch.cuda.synchronize()
    pat = arf.pattern_code(pattern)
    got = (wl.codes(out.cpu()), wl.codes(ro.cpu()) if ro is not None else None)
    assert_parity(GDT["bf16"], pat, got, oracle_run(pat, inp), f"two_shot G=1 {pattern}")


def _gpu_rank(rank, world, port, cases, q):
    """One rank of the two-shot form whose local step is the library's kernels
    on cuda:0; the exchange is gloo on host tensors. The ranks' kernels never
    wait on one another: each runs its own block to completion."""
    import torch.distributed as dist

    import all_reduce_residual_gb300 as arf

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ws = arf.Workspace(0)

    def gpu_step(pattern, partials, residual, gamma, eps):
        out, ro = arf.run(ws, pattern, [p.cuda() for p in partials], None if residual is None else residual.cuda(),
                          None if gamma is None else gamma.cuda(), eps)
        torch.cuda.synchronize()
        return out.cpu(), None if ro is None else ro.cpu()

    try:
        for W, M, H, dtype, pattern in cases:
            w = wl.custom(W, M, H, dtype, 0.7, 1e-6, config_id=980 + M)
            inp = wl.make_inputs(w)
            out, ro = ts.two_shot(pattern, inp.partials[rank], inp.residual, inp.gamma, w.eps, epilogue=gpu_step)
            q.put((rank, (W, M, H, dtype, pattern), wl.codes(out), None if ro is None else wl.codes(ro)))
    finally:
        ws.close()
        dist.destroy_process_group()


@pytest.mark.gpu
def test_two_ranks_with_the_library_epilogue_on_one_gpu():
    """G = 2 through gloo, each rank's block on the library's kernels: every
    rank ends with the oracle's one-call result (bitwise residual_out and
    kAllReduce out, out within 1 ulp), ragged row counts included."""
    from gpu_util import DT as GDT, assert_parity, oracle_run

    world = 2
    cases = [(2, 37, 7168, "bf16", "rmsnorm"), (2, 37, 7168, "bf16", "allreduce"), (2, 3, 4096, "fp16", "rmsnorm"),
             (2, 1, 7168, "bf16", "rmsnorm")]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_gpu_rank, args=(r, world, port, cases, q)) for r in range(world)]
    for p in procs:
        p.start()
    got = [q.get(timeout=300) for _ in range(world * len(cases))]
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    import all_reduce_residual_gb300 as arf

    for rank, (W, M, H, dtype, pattern), out, ro in got:
        w = wl.custom(W, M, H, dtype, 0.7, 1e-6, config_id=980 + M)
        inp = wl.make_inputs(w)
        pat = arf.pattern_code(pattern)
        assert_parity(GDT[dtype], pat, (out, ro), oracle_run(pat, inp), f"rank {rank} {pattern} M={M}")
