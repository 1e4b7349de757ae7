"""arf: the all-reduce fusion epilogue (kAllReduce, kARResidualRMSNorm) on one GB300.

``_binding`` exposes every C entry point of include/arf.h under its own name.
The helpers below only marshal torch tensors into those calls: they check
shapes, dtypes and devices, build the device pointer array, and pass torch's
current stream. All arithmetic runs in libarf.so's CUDA kernels.
"""
from __future__ import annotations

import ctypes

from ._binding import (  # noqa: F401  (re-exported C-ABI names)
    ARF_AR_RESIDUAL_RMSNORM, ARF_ALLREDUCE, ARF_BF16, ARF_ERR_CUDA, ARF_ERR_DEVICE_MISMATCH,
    ARF_ERR_INVALID_ARG, ARF_ERR_UNSUPPORTED, ARF_FP16, ARF_MAX_H, ARF_MAX_H_PER_CTA, ARF_MAX_W, ARF_OK,
    ARF_PATH_ASYNC, ARF_PATH_BULK, ARF_PATH_CLUSTER, ARF_PATH_ELEM, ARF_PATH_FLAT, ARF_PATH_ROW,
    ARF_STATIC_STAGING_BYTES, COMPILED_W, ArfError, DeviceCaps, Plan, RunOpts,
    arf_host_staging_bytes, arf_last_cuda_error, arf_plan_check, arf_plan_for_caps, arf_plan_rules, arf_read_pass,
    arf_run,
    arf_run_ex,
    arf_run_host, arf_run_host_static, arf_run_planned, arf_static_staging_bytes, arf_status_string, arf_supports,
    arf_workspace_autotune, arf_workspace_caps, arf_workspace_create, arf_workspace_destroy, arf_workspace_plan,
    arf_workspace_wait_timeouts, load,
)

PATTERNS = {"allreduce": ARF_ALLREDUCE, "rmsnorm": ARF_AR_RESIDUAL_RMSNORM}


def _torch():
    import torch
    return torch


def dtype_code(dt) -> int:
    torch = _torch()
    if dt == torch.bfloat16:
        return ARF_BF16
    if dt == torch.float16:
        return ARF_FP16
    raise ValueError(f"unsupported dtype {dt}: bf16 or fp16")


def pattern_code(pattern) -> int:
    return PATTERNS[pattern] if isinstance(pattern, str) else int(pattern)


class Workspace:
    """Owns one arf_workspace_t (host state for one device)."""

    def __init__(self, device: int = 0):
        self.handle = ctypes.c_void_p()
        st = arf_workspace_create(device, self.handle)
        if st != ARF_OK:
            raise ArfError(st, f"arf_workspace_create({device})")
        self.device = device

    @property
    def caps(self) -> DeviceCaps:
        c = DeviceCaps()
        st = arf_workspace_caps(self.handle, c)
        if st != ARF_OK:
            raise ArfError(st, "arf_workspace_caps")
        return c

    def plan(self, pattern, W: int, M: int, H: int, dtype) -> Plan:
        p = Plan()
        dt = dtype if isinstance(dtype, int) else dtype_code(dtype)
        st = arf_workspace_plan(self.handle, pattern_code(pattern), W, M, H, dt, p)
        if st != ARF_OK:
            raise ArfError(st, "arf_workspace_plan")
        return p

    def autotune(self, pattern, partials, residual=None, gamma=None, eps: float = 0.0, out=None,
                 residual_out=None, reps: int = 20, ptrs=None):
        """arf_workspace_autotune on CUDA tensors (contiguous 16-bit layout);
        returns (plan, microseconds per call). Later calls of the shape use it."""
        torch = _torch()
        pat = pattern_code(pattern)
        P = list(partials)
        M, H = P[0].shape
        dev, dt = P[0].device, P[0].dtype
        rms = pat == ARF_AR_RESIDUAL_RMSNORM
        out = out if out is not None else torch.empty((M, H), dtype=dt, device=dev)
        ro = residual_out if residual_out is not None else (torch.empty((M, H), dtype=dt, device=dev) if rms else None)
        ptrs = ptrs if ptrs is not None else pointer_array(P, dev)
        plan, us = Plan(), ctypes.c_float()
        st = arf_workspace_autotune(self.handle, pat, len(P), ptrs.data_ptr(), residual.data_ptr() if rms else None,
                                    gamma.data_ptr() if rms else None, float(eps), out.data_ptr(),
                                    ro.data_ptr() if rms else None, M, H, dtype_code(dt), reps,
                                    torch.cuda.current_stream(dev).cuda_stream, plan, us)
        if st != ARF_OK:
            raise ArfError(st, "arf_workspace_autotune", arf_last_cuda_error(self.handle) if st == ARF_ERR_CUDA else 0)
        return plan, us.value

    def close(self):
        if self.handle:
            arf_workspace_destroy(self.handle)
            self.handle = ctypes.c_void_p()

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def pointer_array(tensors, device=None):
    """A device int64 tensor holding the data pointers of `tensors`, in order
    (the DEVICE array of W pointers that arf_run reads)."""
    torch = _torch()
    dev = device if device is not None else tensors[0].device
    host = torch.tensor([t.data_ptr() for t in tensors], dtype=torch.int64)
    return host.to(dev)


def _check_operand(t, name, shape, dtype, device):
    """Returns the row stride in elements ([M,H] tensors may be row-strided
    views whose elements are contiguous within a row)."""
    if t.dtype != dtype:
        raise ValueError(f"{name}: dtype {t.dtype} != {dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: shape {tuple(t.shape)} != {tuple(shape)}")
    if t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if len(shape) == 1 or shape[0] <= 1:
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
        return shape[-1]
    if t.stride(1) != 1 or t.stride(0) < shape[1]:
        raise ValueError(f"{name}: rows must be contiguous with a row stride >= H")
    return t.stride(0)


def run(ws: Workspace, pattern, partials, residual=None, gamma=None, eps: float = 0.0, out=None,
        residual_out=None, stream=None, plan: Plan | None = None, ptrs=None, by_value: bool = False,
        pdl=None):
    """Run one pattern on CUDA tensors.

    partials: list of W [M,H] tensors (rank order). ``ptrs`` may be passed
    instead of building the pointer array here (for CUDA-graph capture, keep
    it alive and stable). out / residual_out are allocated when None.
    by_value / pdl / plan: the options of arf_run_ex (partials passed in the
    launch, programmatic dependent launch, an explicit launch plan). pdl:
    None = the library's choice (on for latency-bound launches), True =
    always, False = never.
    Returns (out, residual_out); residual_out is None for kAllReduce.
    """
    torch = _torch()
    pat = pattern_code(pattern)
    P = list(partials)
    W = len(P)
    if W == 0:
        raise ValueError("at least one partial is required")
    M, H = P[0].shape
    dev, pdt = P[0].device, P[0].dtype
    f32p = pdt == torch.float32
    rms = pat == ARF_AR_RESIDUAL_RMSNORM
    # the I/O dtype: the partials' own, or (binary32 partials) that of the other tensors
    dt = pdt if not f32p else (residual.dtype if rms and residual is not None else
                               (out.dtype if out is not None else torch.bfloat16))
    ldp = None
    for i, p in enumerate(P):
        ld = _check_operand(p, f"partials[{i}]", (M, H), pdt, dev)
        if ldp is not None and ld != ldp:
            raise ValueError("all partials must have the same row stride")
        ldp = ld
    if out is None:
        out = torch.empty((M, H), dtype=dt, device=dev)
    ldo = _check_operand(out, "out", (M, H), dt, dev)
    r_ptr = g_ptr = ro_ptr = None
    ldr = ldro = H
    if rms:
        if residual is None or gamma is None:
            raise ValueError("kARResidualRMSNorm needs residual and gamma")
        ldr = _check_operand(residual, "residual", (M, H), dt, dev)
        _check_operand(gamma, "gamma", (H,), dt, dev)
        if residual_out is None:
            residual_out = torch.empty((M, H), dtype=dt, device=dev)
        ldro = _check_operand(residual_out, "residual_out", (M, H), dt, dev)
        r_ptr, g_ptr, ro_ptr = residual.data_ptr(), gamma.data_ptr(), residual_out.data_ptr()
    s = stream if stream is not None else torch.cuda.current_stream(dev)
    tail = (r_ptr, g_ptr, float(eps), out.data_ptr(), ro_ptr, M, H, dtype_code(dt), s.cuda_stream)
    general = f32p or (ldp, ldr, ldo, ldro) != (H, H, H, H)
    pdl_code = 0 if pdl is None else (1 if pdl else 2)  # arf_run_opts_t.pdl: 0 auto, 1 always, 2 never
    if by_value or pdl is not None or general:
        opts = RunOpts(plan=ctypes.pointer(plan) if plan is not None else None, partials_by_value=int(by_value),
                       pdl=pdl_code, ld_partials=ldp, ld_residual=ldr, ld_out=ldo, ld_residual_out=ldro,
                       partials_f32=int(f32p))
        if by_value:
            parts = [p.data_ptr() for p in P]
        else:
            if ptrs is None:
                ptrs = pointer_array(P, dev)
                if stream is not None and M > 0:
                    ptrs.record_stream(s)
            parts = ptrs.data_ptr()
        st = arf_run_ex(ws.handle, opts, pat, W, parts, *tail)
    else:
        if ptrs is None:
            ptrs = pointer_array(P, dev)
            if stream is not None and M > 0:
                ptrs.record_stream(s)  # the temporary array must outlive the kernel
        args = (pat, W, ptrs.data_ptr(), *tail)
        st = arf_run_planned(ws.handle, plan, *args) if plan is not None else arf_run(ws.handle, *args)
    if st != ARF_OK:
        raise ArfError(st, "arf_run", arf_last_cuda_error(ws.handle) if st == ARF_ERR_CUDA else 0)
    return out, (residual_out if rms else None)


class HostRunner:
    """Calls on host (page-locked) buffers for one shape.

    zero_copy=False: arf_run_host, with a device staging buffer allocated
    once by torch and reused by every call (copies in, kernel, copies out).
    zero_copy=True: arf_run on the host buffers themselves, which the kernels
    read and write over the host link; the pointer array is a page-locked
    host array kept per set of partials for the runner's lifetime."""

    def __init__(self, ws: Workspace, pattern, W: int, M: int, H: int, dtype, zero_copy: bool = False):
        torch = _torch()
        self.ws, self.pat, self.W, self.M, self.H = ws, pattern_code(pattern), W, M, H
        self.dt = dtype
        self.zero_copy = zero_copy
        self._ptr_arrays = {}
        if zero_copy:
            return
        self.nbytes = arf_host_staging_bytes(self.pat, W, M, H, dtype_code(dtype))
        if self.nbytes == 0 and M > 0:
            raise ArfError(ARF_ERR_UNSUPPORTED, "arf_host_staging_bytes")
        self.staging = torch.empty(max(self.nbytes, 256) + 256, dtype=torch.uint8, device=f"cuda:{ws.device}")
        base = self.staging.data_ptr()
        self.staging_ptr = (base + 255) & ~255

    def __call__(self, partials, residual=None, gamma=None, eps=0.0, out=None, residual_out=None, stream=None):
        """partials / residual / gamma / out / residual_out: CPU tensors
        (page-locked for asynchronous copies). Enqueues on `stream` and returns;
        synchronise the stream before reading the outputs."""
        torch = _torch()
        s = stream if stream is not None else torch.cuda.current_stream(self.ws.device)
        rms = self.pat == ARF_AR_RESIDUAL_RMSNORM
        if self.zero_copy:
            key = tuple(p.data_ptr() for p in partials)
            ptrs = self._ptr_arrays.get(key)
            if ptrs is None:
                ptrs = torch.tensor(list(key), dtype=torch.int64).pin_memory()
                self._ptr_arrays[key] = ptrs
            st = arf_run(self.ws.handle, self.pat, self.W, ptrs.data_ptr(), residual.data_ptr() if rms else None,
                         gamma.data_ptr() if rms else None, float(eps), out.data_ptr(),
                         residual_out.data_ptr() if rms else None, self.M, self.H, dtype_code(self.dt),
                         s.cuda_stream)
            if st != ARF_OK:
                raise ArfError(st, "arf_run (host buffers)",
                               arf_last_cuda_error(self.ws.handle) if st == ARF_ERR_CUDA else 0)
            return
        st = arf_run_host(self.ws.handle, self.pat, self.W, [p.data_ptr() for p in partials],
                          residual.data_ptr() if rms else None, gamma.data_ptr() if rms else None, float(eps),
                          out.data_ptr(), residual_out.data_ptr() if rms else None, self.M, self.H,
                          dtype_code(self.dt), self.staging_ptr, self.nbytes, s.cuda_stream)
        if st != ARF_OK:
            raise ArfError(st, "arf_run_host", arf_last_cuda_error(self.ws.handle) if st == ARF_ERR_CUDA else 0)
