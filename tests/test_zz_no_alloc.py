"""arf_run_host_static: the host-buffer entry point that allocates nothing.

It serves callers that may not allocate device memory themselves, such as a
plugin running inside a framework or serving engine whose allocator already
owns the GPU's memory, or a latency-critical host thread that cannot take
cudaMalloc's implicit synchronisation. Instead of a caller-provided staging
buffer it uses a device array built into the library, whose address each
workspace looks up when it is created.

The tests call it through the C ABI on two calls in a row with different
shapes and inputs, so stale contents of the shared array would show, and
check each result against the CPU oracle and against the allocating entry
point (arf_run_host with a staging buffer allocated here). Tolerances are the
suite's: residual_out and the all-reduce bitwise, the normalised out within
1 ulp. A last test runs in a fresh process under lazy module loading and
checks that the array is taken when the workspace is created, not inside a
call. This file is collected last and needs nothing from the other tests.
"""
import json
import os
import subprocess
import sys

import pytest
import torch

import all_reduce_residual_gb300 as arf
from all_reduce_residual_gb300 import workloads as wl
from gpu_util import DT, assert_parity, oracle_run

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _host_inputs(name, M, cid_shift=0):
    w = wl.WORKLOADS[name]
    w = wl.custom(w.W, M, w.H, w.dtype, w.partial_sigma, w.eps, config_id=w.config_id + cid_shift)
    inp = wl.make_inputs(w)
    P = [p.pin_memory() for p in inp.partials]
    return w, inp, P, inp.residual.pin_memory(), inp.gamma.pin_memory()


def _outputs(w):
    dt = wl.TORCH_DTYPE[w.dtype]
    return (torch.empty((w.M, w.H), dtype=dt).pin_memory(), torch.empty((w.M, w.H), dtype=dt).pin_memory())


@pytest.mark.parametrize("pattern", [arf.ARF_ALLREDUCE, arf.ARF_AR_RESIDUAL_RMSNORM])
def test_static_staging_matches_oracle_and_allocating_entry_point(pattern):
    rms = pattern == arf.ARF_AR_RESIDUAL_RMSNORM
    cap = arf.arf_static_staging_bytes()
    with arf.Workspace(0) as ws:
        stream = torch.cuda.current_stream()
        for name, M, shift in (("llama_tp2", 128, 0), ("k3_tp8", 32, 7)):  # two calls in a row
            w, inp, P, R, G = _host_inputs(name, M, shift)
            dcode = arf.dtype_code(wl.TORCH_DTYPE[w.dtype])
            assert arf.arf_host_staging_bytes(pattern, w.W, M, w.H, dcode) <= cap
            ref_out, ref_ro = _outputs(w)
            arf.HostRunner(ws, pattern, w.W, M, w.H, wl.TORCH_DTYPE[w.dtype])(P, R, G, w.eps, ref_out, ref_ro)
            out, ro = _outputs(w)
            st = arf.arf_run_host_static(ws.handle, pattern, w.W, [p.data_ptr() for p in P],
                                         R.data_ptr() if rms else None, G.data_ptr() if rms else None, w.eps,
                                         out.data_ptr(), ro.data_ptr() if rms else None, M, w.H, dcode,
                                         stream.cuda_stream)
            assert st == arf.ARF_OK, arf.arf_status_string(st)
            torch.cuda.synchronize()
            got = (wl.codes(out), wl.codes(ro) if rms else None)
            assert_parity(DT[w.dtype], pattern, got, oracle_run(pattern, inp), f"{name} M={M} vs oracle")
            ref = (wl.codes(ref_out), wl.codes(ref_ro) if rms else None)
            assert_parity(DT[w.dtype], pattern, got, ref, f"{name} M={M} vs arf_run_host")


def test_static_staging_rejects_sizes_beyond_its_capacity():
    w, _, P, R, G = _host_inputs("k3_tp8", 2048)
    dcode = arf.dtype_code(wl.TORCH_DTYPE[w.dtype])
    pattern = arf.ARF_AR_RESIDUAL_RMSNORM
    assert arf.arf_host_staging_bytes(pattern, w.W, w.M, w.H, dcode) > arf.arf_static_staging_bytes()
    out, ro = _outputs(w)
    out.fill_(3.0)
    with arf.Workspace(0) as ws:
        st = arf.arf_run_host_static(ws.handle, pattern, w.W, [p.data_ptr() for p in P], R.data_ptr(),
                                     G.data_ptr(), w.eps, out.data_ptr(), ro.data_ptr(), w.M, w.H, dcode,
                                     torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert st == arf.ARF_ERR_UNSUPPORTED
    assert bool((out.float() == 3.0).all()), "a rejected call wrote its output"


# Run in a fresh process: device memory free before and after the workspace
# is created, and after two calls; the results checked against the oracle.
_LAZY_CHILD = r"""
import json, sys
sys.path.insert(0, sys.argv[1]); sys.path.insert(0, sys.argv[1] + "/tests")
import torch
import all_reduce_residual_gb300 as arf
from all_reduce_residual_gb300 import workloads as wl
from gpu_util import DT, assert_parity, oracle_run
torch.zeros(1, device="cuda")
torch.cuda.synchronize()
arf.load()
free0 = torch.cuda.mem_get_info()[0]
ws = arf.Workspace(0)
free1 = torch.cuda.mem_get_info()[0]
for M, cid in ((8, 31), (16, 32)):
    w = wl.custom(2, M, 1024, "bf16", 1.0, 1e-6, config_id=cid)
    inp = wl.make_inputs(w)
    P = [p.pin_memory() for p in inp.partials]
    R, G = inp.residual.pin_memory(), inp.gamma.pin_memory()
    out = torch.empty((M, 1024), dtype=torch.bfloat16).pin_memory()
    ro = torch.empty((M, 1024), dtype=torch.bfloat16).pin_memory()
    st = arf.arf_run_host_static(ws.handle, arf.ARF_AR_RESIDUAL_RMSNORM, 2, [p.data_ptr() for p in P],
                                 R.data_ptr(), G.data_ptr(), w.eps, out.data_ptr(), ro.data_ptr(), M, 1024,
                                 arf.ARF_BF16, torch.cuda.current_stream().cuda_stream)
    assert st == arf.ARF_OK, arf.arf_status_string(st)
    torch.cuda.synchronize()
    assert_parity(DT["bf16"], arf.ARF_AR_RESIDUAL_RMSNORM, (wl.codes(out), wl.codes(ro)),
                  oracle_run(arf.ARF_AR_RESIDUAL_RMSNORM, inp), f"M={M}")
free2 = torch.cuda.mem_get_info()[0]
ws.close()
print(json.dumps({"at_create": free0 - free1, "in_calls": free1 - free2}))
"""


def test_static_staging_is_taken_at_workspace_creation_under_lazy_loading():
    env = dict(os.environ, CUDA_MODULE_LOADING="LAZY")
    r = subprocess.run([sys.executable, "-c", _LAZY_CHILD, ROOT], capture_output=True, text=True, env=env,
                       timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    got = json.loads(r.stdout.strip().splitlines()[-1])
    cap = arf.arf_static_staging_bytes()
    assert got["at_create"] >= cap, f"the staging array was not loaded at workspace creation: {got}"
    assert got["in_calls"] < cap, f"the calls took device memory the size of the staging array: {got}"
