"""ctypes binding of include/arf.h: one Python function per C entry point,
same names, same arguments (pointers as ints, streams as ints). Argument
marshalling only: every step of the epilogue runs in the CUDA library.

The library is loaded on first use. If libarf.so has not been built the call
raises at once; there is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os
import threading

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libarf.so")

# arf_status_t
ARF_OK = 0
ARF_ERR_INVALID_ARG = 1
ARF_ERR_UNSUPPORTED = 2
ARF_ERR_CUDA = 3
ARF_ERR_DEVICE_MISMATCH = 4
# arf_pattern_t
ARF_ALLREDUCE = 0
ARF_AR_RESIDUAL_RMSNORM = 1
# arf_dtype_t
ARF_BF16 = 0
ARF_FP16 = 1
# arf_path_t
ARF_PATH_FLAT = 0
ARF_PATH_ROW = 1
ARF_PATH_CLUSTER = 2
ARF_PATH_ASYNC = 3
ARF_PATH_ELEM = 4
ARF_PATH_BULK = 5
ARF_MAX_W = 64
ARF_MAX_H = 524288
ARF_MAX_H_PER_CTA = 32768
ARF_STATIC_STAGING_BYTES = 16 << 20
# Rank counts with kernels specialised at compile time (w_spec values other than 0).
COMPILED_W = (1, 2, 4, 8, 12, 16)

STATUS_NAMES = {0: "ARF_OK", 1: "ARF_ERR_INVALID_ARG", 2: "ARF_ERR_UNSUPPORTED", 3: "ARF_ERR_CUDA",
                4: "ARF_ERR_DEVICE_MISMATCH"}


class DeviceCaps(ctypes.Structure):
    _fields_ = [("num_sms", ctypes.c_int), ("max_cluster", ctypes.c_int), ("max_threads_per_sm", ctypes.c_int),
                ("max_smem_per_block", ctypes.c_int)]

    def __repr__(self):
        return f"DeviceCaps(num_sms={self.num_sms}, max_cluster={self.max_cluster}, " \
               f"max_threads_per_sm={self.max_threads_per_sm}, max_smem_per_block={self.max_smem_per_block})"


class Plan(ctypes.Structure):
    _fields_ = [("path", ctypes.c_int), ("threads", ctypes.c_int), ("vpt", ctypes.c_int),
                ("cluster", ctypes.c_int), ("grid", ctypes.c_int), ("w_spec", ctypes.c_int),
                ("stages", ctypes.c_int)]

    def as_dict(self):
        return {k: getattr(self, k) for k, _ in self._fields_}

    def __repr__(self):
        return "Plan(" + ", ".join(f"{k}={v}" for k, v in self.as_dict().items()) + ")"


class RunOpts(ctypes.Structure):
    _fields_ = [("plan", ctypes.POINTER(Plan)), ("partials_by_value", ctypes.c_int), ("pdl", ctypes.c_int),
                ("ld_partials", ctypes.c_int64), ("ld_residual", ctypes.c_int64), ("ld_out", ctypes.c_int64),
                ("ld_residual_out", ctypes.c_int64), ("partials_f32", ctypes.c_int),
                ("wait_limit_cycles", ctypes.c_int64), ("hold_first_copy", ctypes.c_int)]


_c = ctypes
_vp = _c.c_void_p
_i64 = _c.c_int64
_SIGNATURES = {
    "arf_status_string": (_c.c_char_p, [_c.c_int]),
    "arf_workspace_create": (_c.c_int, [_c.c_int, _c.POINTER(_vp)]),
    "arf_workspace_destroy": (_c.c_int, [_vp]),
    "arf_workspace_caps": (_c.c_int, [_vp, _c.POINTER(DeviceCaps)]),
    "arf_last_cuda_error": (_c.c_int, [_vp]),
    "arf_workspace_wait_timeouts": (_c.c_int, [_vp, _c.POINTER(_c.c_uint)]),
    "arf_supports": (_c.c_int, [_vp, _c.c_int, _c.c_int, _i64, _i64, _c.c_int]),
    "arf_plan_for_caps": (_c.c_int, [_c.POINTER(DeviceCaps), _c.c_int, _c.c_int, _i64, _i64, _c.c_int,
                                     _c.POINTER(Plan)]),
    "arf_plan_rules": (_c.c_int, [_c.POINTER(DeviceCaps), _c.c_int, _c.c_int, _i64, _i64, _c.c_int,
                                  _c.POINTER(Plan)]),
    "arf_workspace_plan": (_c.c_int, [_vp, _c.c_int, _c.c_int, _i64, _i64, _c.c_int, _c.POINTER(Plan)]),
    "arf_plan_check": (_c.c_int, [_c.POINTER(DeviceCaps), _c.POINTER(Plan), _c.c_int, _c.c_int, _i64, _i64,
                                  _c.c_int]),
    "arf_run": (_c.c_int, [_vp, _c.c_int, _c.c_int, _vp, _vp, _vp, _c.c_float, _vp, _vp, _i64, _i64, _c.c_int,
                           _vp]),
    "arf_run_planned": (_c.c_int, [_vp, _c.POINTER(Plan), _c.c_int, _c.c_int, _vp, _vp, _vp, _c.c_float, _vp,
                                   _vp, _i64, _i64, _c.c_int, _vp]),
    "arf_run_ex": (_c.c_int, [_vp, _c.POINTER(RunOpts), _c.c_int, _c.c_int, _vp, _vp, _vp, _c.c_float, _vp, _vp,
                              _i64, _i64, _c.c_int, _vp]),
    "arf_workspace_autotune": (_c.c_int, [_vp, _c.c_int, _c.c_int, _vp, _vp, _vp, _c.c_float, _vp, _vp, _i64, _i64,
                                          _c.c_int, _c.c_int, _vp, _c.POINTER(Plan), _c.POINTER(_c.c_float)]),
    "arf_host_staging_bytes": (_c.c_size_t, [_c.c_int, _c.c_int, _i64, _i64, _c.c_int]),
    "arf_run_host": (_c.c_int, [_vp, _c.c_int, _c.c_int, _c.POINTER(_vp), _vp, _vp, _c.c_float, _vp, _vp, _i64,
                                _i64, _c.c_int, _vp, _c.c_size_t, _vp]),
    "arf_read_pass": (_c.c_int, [_vp, _vp, _i64, _vp]),
    "arf_run_host_static": (_c.c_int, [_vp, _c.c_int, _c.c_int, _c.POINTER(_vp), _vp, _vp, _c.c_float, _vp, _vp,
                                       _i64, _i64, _c.c_int, _vp]),
    "arf_static_staging_bytes": (_c.c_size_t, []),
}

_lib = None
_lock = threading.Lock()


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libarf.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(path):
                raise RuntimeError(
                    f"{path} is not built: run `python -m all_reduce_residual_gb300.build` "
                    "(or __graft_entry__.build()); there is no non-CUDA fallback")
            lib = ctypes.CDLL(path)
            for name, (res, args) in _SIGNATURES.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib


def exported_names():
    return list(_SIGNATURES)


class ArfError(RuntimeError):
    def __init__(self, status: int, what: str = "", cuda_error: int = 0):
        self.status = status
        self.cuda_error = cuda_error
        msg = f"{what}: {STATUS_NAMES.get(status, status)} ({arf_status_string(status)})"
        if cuda_error:
            msg += f", cudaError {cuda_error}"
        super().__init__(msg)


# --- one function per C entry point -------------------------------------------------


def arf_status_string(status: int) -> str:
    return load().arf_status_string(status).decode()


def arf_workspace_create(device: int, ws_out) -> int:
    """ws_out: a ctypes.c_void_p receiving the handle."""
    return load().arf_workspace_create(device, ctypes.byref(ws_out))


def arf_workspace_destroy(ws) -> int:
    return load().arf_workspace_destroy(ws)


def arf_workspace_caps(ws, caps_out: DeviceCaps) -> int:
    return load().arf_workspace_caps(ws, ctypes.byref(caps_out))


def arf_last_cuda_error(ws) -> int:
    return load().arf_last_cuda_error(ws)


def arf_workspace_wait_timeouts(ws, count_out) -> int:
    """count_out: a ctypes.c_uint."""
    return load().arf_workspace_wait_timeouts(ws, ctypes.byref(count_out))


def arf_supports(ws, pattern: int, W: int, M: int, H: int, dtype: int) -> int:
    return load().arf_supports(ws, pattern, W, M, H, dtype)


def arf_plan_for_caps(caps: DeviceCaps, pattern: int, W: int, M: int, H: int, dtype: int, plan_out: Plan) -> int:
    return load().arf_plan_for_caps(ctypes.byref(caps), pattern, W, M, H, dtype, ctypes.byref(plan_out))


def arf_plan_rules(caps: DeviceCaps, pattern: int, W: int, M: int, H: int, dtype: int, plan_out: Plan) -> int:
    return load().arf_plan_rules(ctypes.byref(caps), pattern, W, M, H, dtype, ctypes.byref(plan_out))


def arf_workspace_plan(ws, pattern: int, W: int, M: int, H: int, dtype: int, plan_out: Plan) -> int:
    return load().arf_workspace_plan(ws, pattern, W, M, H, dtype, ctypes.byref(plan_out))


def arf_plan_check(caps: DeviceCaps, plan: Plan, pattern: int, W: int, M: int, H: int, dtype: int) -> int:
    return load().arf_plan_check(ctypes.byref(caps), ctypes.byref(plan), pattern, W, M, H, dtype)


def arf_run(ws, pattern, W, partials_dev, residual, gamma, eps, out, residual_out, M, H, dtype, stream) -> int:
    return load().arf_run(ws, pattern, W, partials_dev, residual, gamma, eps, out, residual_out, M, H, dtype,
                          stream)


def arf_run_planned(ws, plan: Plan, pattern, W, partials_dev, residual, gamma, eps, out, residual_out, M, H,
                    dtype, stream) -> int:
    return load().arf_run_planned(ws, ctypes.byref(plan), pattern, W, partials_dev, residual, gamma, eps, out,
                                  residual_out, M, H, dtype, stream)


def arf_run_ex(ws, opts, pattern, W, partials, residual, gamma, eps, out, residual_out, M, H, dtype,
               stream) -> int:
    """opts: a RunOpts or None. With opts.partials_by_value, `partials` is a
    sequence of W device addresses (a host array is built here); else the
    address of a device array of W pointers."""
    if opts is not None and opts.partials_by_value:
        partials = ctypes.cast((ctypes.c_void_p * W)(*partials), ctypes.c_void_p)
    return load().arf_run_ex(ws, ctypes.byref(opts) if opts is not None else None, pattern, W, partials, residual,
                             gamma, eps, out, residual_out, M, H, dtype, stream)


def arf_workspace_autotune(ws, pattern, W, partials_dev, residual, gamma, eps, out, residual_out, M, H, dtype, reps,
                           stream, plan_out=None, us_out=None) -> int:
    """plan_out: a Plan or None; us_out: a ctypes.c_float or None."""
    return load().arf_workspace_autotune(ws, pattern, W, partials_dev, residual, gamma, eps, out, residual_out, M, H,
                                         dtype, reps, stream, ctypes.byref(plan_out) if plan_out is not None else None,
                                         ctypes.byref(us_out) if us_out is not None else None)


def arf_host_staging_bytes(pattern, W, M, H, dtype) -> int:
    return load().arf_host_staging_bytes(pattern, W, M, H, dtype)


def arf_run_host(ws, pattern, W, partials_host, residual_host, gamma_host, eps, out_host, residual_out_host, M, H,
                 dtype, staging_dev, staging_bytes, stream) -> int:
    """partials_host: a sequence of W host addresses (ints)."""
    arr = (ctypes.c_void_p * W)(*partials_host)
    return load().arf_run_host(ws, pattern, W, arr, residual_host, gamma_host, eps, out_host, residual_out_host,
                               M, H, dtype, staging_dev, staging_bytes, stream)


def arf_read_pass(ws, buf, nbytes, stream) -> int:
    return load().arf_read_pass(ws, buf, nbytes, stream)


def arf_run_host_static(ws, pattern, W, partials_host, residual_host, gamma_host, eps, out_host,
                        residual_out_host, M, H, dtype, stream) -> int:
    """arf_run_host with the library's built-in staging array (allocates
    nothing). partials_host: a sequence of W host addresses (ints)."""
    arr = (ctypes.c_void_p * W)(*partials_host)
    return load().arf_run_host_static(ws, pattern, W, arr, residual_host, gamma_host, eps, out_host,
                                      residual_out_host, M, H, dtype, stream)


def arf_static_staging_bytes() -> int:
    return load().arf_static_staging_bytes()
