"""Every plan of the measured plan table that applies to this GPU, run through
arf_run (the planner picks it) and compared with the CPU oracle: residual_out
and the all-reduce bitwise, the normalised out within 1 ulp. Shapes are taken
at the low end of each row's M range and at a ragged count inside it. Inputs
are drawn on the GPU with the seeded recipe and copied to the host for the
oracle; beyond a few million elements the oracle checks a sample of rows,
which it computes independently of the others."""
import numpy as np
import pytest
import torch

import all_reduce_residual_gb300 as arf
from all_reduce_residual_gb300 import plan_table as pt
from all_reduce_residual_gb300 import workloads as wl
from gpu_util import DT, assert_parity, oracle_run

pytestmark = pytest.mark.gpu

FULL_ROWS_ELEMS = 4 << 20  # W * M * H elements the oracle checks in full


def _cases():
    rows = pt.read_table()
    out = []
    for i, r in enumerate(rows):
        Ms = {r["m_lo"]}
        if r["m_hi"] - r["m_lo"] >= 2:
            Ms.add(min(r["m_hi"], r["m_lo"] + 1 + (r["m_lo"] % 7)))  # a ragged count inside the range
        for M in sorted(Ms):
            if (r["W"] + 3) * M * r["H"] * 2 <= (3 << 30):
                out.append(pytest.param(r, M, id=f"row{i}-M{M}"))
    return out


@pytest.fixture(scope="module")
def ws():
    with arf.Workspace(0) as w:
        yield w


@pytest.mark.parametrize("row,M", _cases())
def test_table_plan_matches_oracle(ws, row, M):
    caps = ws.caps
    if (caps.num_sms, caps.max_cluster, caps.max_threads_per_sm, caps.max_smem_per_block) != \
            (row["num_sms"], row["max_cluster"], row["max_threads_per_sm"], row["max_smem_per_block"]):
        pytest.skip("the table row was measured on a device with other capabilities")
    dts = "bf16" if row["dtype"] == arf.ARF_BF16 else "fp16"
    W, H, pattern = row["W"], row["H"], row["pattern"]
    plan = ws.plan(pattern, W, M, H, wl.TORCH_DTYPE[dts])
    row_plan = arf.Plan(*pt.row_plan_fields(row, M))
    if arf.arf_plan_check(caps, row_plan, pattern, W, M, H, row["dtype"]) == arf.ARF_OK:
        assert (plan.path, plan.threads, plan.vpt, plan.cluster, plan.grid, plan.w_spec, plan.stages) == \
            pt.row_plan_fields(row, M)
    w = wl.custom(W, M, H, dts, 0.5, 1e-6, config_id=960 + (M % 17))
    dev = wl.make_inputs(w, device="cuda")  # drawn on the GPU; the oracle gets the same bytes
    out, ro = arf.run(ws, pattern, dev.partials, dev.residual, dev.gamma, w.eps)
    torch.cuda.synchronize()
    rms = pattern == arf.ARF_AR_RESIDUAL_RMSNORM
    if W * M * H <= FULL_ROWS_ELEMS:
        pick = np.arange(M)
    else:
        pick = np.unique(np.concatenate([[0, M - 1], np.random.default_rng(M).integers(0, M, 24)]))
    idx = torch.as_tensor(pick, device="cuda")
    sub = wl.Inputs(w.with_m(len(pick)), [p[idx].cpu() for p in dev.partials], dev.residual[idx].cpu(),
                    dev.gamma.cpu())
    ref = oracle_run(pattern, sub)
    got = (wl.codes(out[idx].cpu()), wl.codes(ro[idx].cpu()) if rms else None)
    assert_parity(DT[dts], pattern, got, ref, f"table row {row} at M={M}")
