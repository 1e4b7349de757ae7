"""Helpers for the GPU tests: run the CUDA path through the C ABI and compare
it with the CPU oracle element by element.

Tolerances (the library's numeric contract):
* kAllReduce ``out`` and ``residual_out``: bitwise equal (one correct value);
* kARResidualRMSNorm ``out``: within 1 ulp of the output dtype, measured at the
  larger magnitude: |gpu - oracle| <= ulp(max(|gpu|, |oracle|)); equal
  infinities and zeros of either sign pass, NaN must meet NaN.
"""
from __future__ import annotations

import numpy as np
import torch

import all_reduce_residual_gb300 as arf
import oracle
from all_reduce_residual_gb300 import workloads as wl

DT = {"bf16": oracle.BF16, "fp16": oracle.FP16}
PAT = {"allreduce": arf.ARF_ALLREDUCE, "rmsnorm": arf.ARF_AR_RESIDUAL_RMSNORM}


def decode(dtype: int, codes) -> np.ndarray:
    c = np.ascontiguousarray(codes, dtype=np.uint16)
    if dtype == oracle.BF16:
        return torch.from_numpy(c.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
    return c.view(np.float16).astype(np.float64)


def ulp_of(dtype: int, a: np.ndarray) -> np.ndarray:
    """Spacing of the format at |a| (its binade; the subnormal spacing below)."""
    p, emin = (8, -126) if dtype == oracle.BF16 else (11, -14)
    a = np.abs(a)
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.maximum(e, emin)
    return np.ldexp(1.0, (e - (p - 1)).astype(np.int64))


def within_one_ulp(dtype: int, got, want) -> np.ndarray:
    g, w = decode(dtype, got), decode(dtype, want)
    both_nan = np.isnan(g) & np.isnan(w)
    with np.errstate(invalid="ignore"):
        same = (g == w)  # equal values, +-0, equal infinities
        diff = np.abs(g - w)
        ok = diff <= ulp_of(dtype, np.maximum(np.abs(g), np.abs(w)))
    return both_nan | same | (np.isfinite(g) & np.isfinite(w) & ok)


def bitwise_equal(dtype: int, got, want) -> np.ndarray:
    got = np.asarray(got, np.uint16)
    want = np.asarray(want, np.uint16)
    nan = lambda c: (c & np.uint16(0x7FFF)) > (0x7F80 if dtype == oracle.BF16 else 0x7C00)  # noqa: E731
    return (got == want) | (nan(got) & nan(want))


def assert_parity(dtype, pattern, gpu, ref, what=""):
    """gpu / ref: (out_codes, residual_out_codes or None). Returns the number
    of 1-ulp differences in the normalised output."""
    g_out, g_ro = gpu
    r_out, r_ro = ref
    if pattern == arf.ARF_ALLREDUCE:
        eq = bitwise_equal(dtype, g_out, r_out)
        assert eq.all(), f"{what}: kAllReduce out differs bitwise at {np.argwhere(~eq)[:5].tolist()}"
        return 0
    eq = bitwise_equal(dtype, g_ro, r_ro)
    assert eq.all(), f"{what}: residual_out differs bitwise at {np.argwhere(~eq)[:5].tolist()} " \
                     f"({(~eq).sum()} elements)"
    ok = within_one_ulp(dtype, g_out, r_out)
    assert ok.all(), f"{what}: out beyond 1 ulp at {np.argwhere(~ok)[:5].tolist()} ({(~ok).sum()} elements)"
    return int((~bitwise_equal(dtype, g_out, r_out)).sum())


def to_device(inp: wl.Inputs, device="cuda"):
    return ([p.to(device) for p in inp.partials], inp.residual.to(device), inp.gamma.to(device))


def gpu_run(ws, pattern, P, R, G, eps, plan=None, in_place=False):
    """Run through the C ABI; returns host codes (out, residual_out or None).
    in_place: residual_out is the residual buffer itself (a copy of R)."""
    rms = pattern == arf.ARF_AR_RESIDUAL_RMSNORM
    if rms and in_place:
        buf = R.clone()
        out, ro = arf.run(ws, pattern, P, buf, G, eps, residual_out=buf, plan=plan)
    else:
        out, ro = arf.run(ws, pattern, P, R, G, eps, plan=plan)
    torch.cuda.synchronize()
    return wl.codes(out.cpu()), (wl.codes(ro.cpu()) if rms else None)


def oracle_run(pattern, inp: wl.Inputs, eps=None, order=None):
    P = [wl.codes(p) for p in inp.partials]
    if order is not None:
        P = [P[i] for i in order]
    dtype = DT[inp.workload.dtype]
    e = inp.workload.eps if eps is None else eps
    if pattern == arf.ARF_ALLREDUCE:
        return oracle.run(oracle.ALLREDUCE, P, dtype=dtype)
    return oracle.run(oracle.AR_RESIDUAL_RMSNORM, P, wl.codes(inp.residual), wl.codes(inp.gamma), e, dtype=dtype)
