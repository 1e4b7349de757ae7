"""arf_run_host_static: the host-buffer entry point that allocates nothing.

It serves callers that may not allocate device memory themselves, such as a
plugin running inside a framework or serving engine whose allocator already
owns the GPU's memory, or a latency-critical host thread that cannot take
cudaMalloc's implicit synchronisation. Instead of a caller-provided staging
buffer it uses a device array built into the library.

The test calls it through the C ABI and checks it against the allocating
entry point (arf_run_host with a staging buffer allocated here) on two calls
in a row with different shapes and inputs, so stale contents of the shared
array would show. Tolerances are the suite's: residual_out and the
all-reduce bitwise, the normalised out within 1 ulp. This file is collected
last and needs nothing from the other tests.
"""
import pytest
import torch

import all_reduce_residual_gb300 as arf
from all_reduce_residual_gb300 import workloads as wl
from gpu_util import DT, assert_parity

pytestmark = pytest.mark.gpu


def _host_inputs(name, M, cid_shift=0):
    w = wl.WORKLOADS[name]
    w = wl.custom(w.W, M, w.H, w.dtype, w.partial_sigma, w.eps, config_id=w.config_id + cid_shift)
    inp = wl.make_inputs(w)
    P = [p.pin_memory() for p in inp.partials]
    return w, P, inp.residual.pin_memory(), inp.gamma.pin_memory()


def _outputs(w):
    dt = wl.TORCH_DTYPE[w.dtype]
    return (torch.empty((w.M, w.H), dtype=dt).pin_memory(), torch.empty((w.M, w.H), dtype=dt).pin_memory())


@pytest.mark.parametrize("pattern", [arf.ARF_ALLREDUCE, arf.ARF_AR_RESIDUAL_RMSNORM])
def test_static_staging_matches_allocating_entry_point(pattern):
    rms = pattern == arf.ARF_AR_RESIDUAL_RMSNORM
    with arf.Workspace(0) as ws:
        stream = torch.cuda.current_stream()
        for name, M, shift in (("llama_tp2", 128, 0), ("k3_tp8", 32, 7)):  # two calls in a row
            w, P, R, G = _host_inputs(name, M, shift)
            dcode = arf.dtype_code(wl.TORCH_DTYPE[w.dtype])
            assert arf.arf_host_staging_bytes(pattern, w.W, M, w.H, dcode) <= arf.ARF_STATIC_STAGING_BYTES
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
            ref = (wl.codes(ref_out), wl.codes(ref_ro) if rms else None)
            assert_parity(DT[w.dtype], pattern, got, ref, f"{name} M={M}")


def test_static_staging_rejects_sizes_beyond_its_capacity():
    w, P, R, G = _host_inputs("k3_tp8", 2048)
    dcode = arf.dtype_code(wl.TORCH_DTYPE[w.dtype])
    pattern = arf.ARF_AR_RESIDUAL_RMSNORM
    assert arf.arf_host_staging_bytes(pattern, w.W, w.M, w.H, dcode) > arf.ARF_STATIC_STAGING_BYTES
    out, ro = _outputs(w)
    out.fill_(3.0)
    with arf.Workspace(0) as ws:
        st = arf.arf_run_host_static(ws.handle, pattern, w.W, [p.data_ptr() for p in P], R.data_ptr(),
                                     G.data_ptr(), w.eps, out.data_ptr(), ro.data_ptr(), w.M, w.H, dcode,
                                     torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert st == arf.ARF_ERR_UNSUPPORTED
    assert bool((out.float() == 3.0).all()), "a rejected call wrote its output"
