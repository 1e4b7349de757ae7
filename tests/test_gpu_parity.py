"""Parity of the CUDA path with the CPU oracle on every workload (and the
extra shapes the benchmark's sweep measures), at full size, through the C
ABI with the planner's launch configuration (the one the benchmark times). residual_out and kAllReduce out must be bitwise equal;
kARResidualRMSNorm out within 1 ulp (see gpu_util)."""
import pytest
import torch

import all_reduce_residual_gb300 as arf
from all_reduce_residual_gb300 import workloads as wl
from gpu_util import DT, PAT, assert_parity, gpu_run, oracle_run, to_device

pytestmark = pytest.mark.gpu

ALL = {**wl.WORKLOADS, **wl.EXTRA_WORKLOADS}
CASES = []
for name, w in ALL.items():
    Ms = wl.K3_M_SWEEP if name == "k3_tp8" else (w.M,)
    for M in Ms:
        for pat in w.patterns:
            CASES.append((name, M, pat))


@pytest.fixture(scope="module")
def ws():
    with arf.Workspace(0) as w:
        yield w


@pytest.mark.parametrize("name,M,pattern", CASES, ids=[f"{n}-M{m}-{p}" for n, m, p in CASES])
def test_workload_parity(ws, name, M, pattern):
    inp = wl.make_inputs(ALL[name], M=M)
    P, R, G = to_device(inp)
    pat = PAT[pattern]
    if name in wl.EXTRA_WORKLOADS:  # these shapes exist to reach particular kernel paths
        plan = ws.plan(pattern, len(P), M, inp.workload.H, P[0].dtype)
        want = wl.extra_path(name, pattern)
        if want == "bulk":
            assert plan.path == arf.ARF_PATH_BULK, plan
        elif want == "elem":
            assert plan.path == arf.ARF_PATH_ELEM, plan
        elif want == "flat":
            assert plan.path == arf.ARF_PATH_FLAT, plan
        elif want == "cluster":
            assert plan.path == arf.ARF_PATH_CLUSTER, plan
        elif want == "row":
            assert plan.path == arf.ARF_PATH_ROW, plan
        else:
            assert plan.path == arf.ARF_PATH_ROW and plan.grid == M, plan
    got = gpu_run(ws, pat, P, R, G, inp.workload.eps)
    ref = oracle_run(pat, inp)
    n1 = assert_parity(DT[inp.workload.dtype], pat, got, ref, f"{name} M={M} {pattern}")
    # 1-ulp differences in out must stay rare (binary32 error << half an ulp)
    assert n1 <= max(8, got[0].size // 200), f"{n1} one-ulp differences in {got[0].size} elements"
    del P, R, G
    torch.cuda.empty_cache()
