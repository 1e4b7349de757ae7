"""CPU oracle for the all-reduce fusion epilogue (ctypes wrapper).

TEST INFRASTRUCTURE, not part of the library. Only ``tests/``, the package's
``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg import this
module. It builds and loads ``liboracle.so`` from ``arf_oracle.c`` (plain C,
single-threaded) and shares nothing with the CUDA library.

Buffers are numpy ``uint16`` arrays holding bf16 / fp16 codes. Enum values:
pattern 0 = kAllReduce, 1 = kARResidualRMSNorm; dtype 0 = bf16, 1 = fp16.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import tempfile

import numpy as np

ALLREDUCE = 0
AR_RESIDUAL_RMSNORM = 1
BF16 = 0
FP16 = 1

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "arf_oracle.c")
HDR = os.path.join(HERE, "arf_oracle.h")
LIB = os.path.join(HERE, "liboracle.so")

# Strict IEEE binary32: no FMA contraction, no fast-math reassociation.
CFLAGS = ["-std=c99", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]


def compile_oracle(src: str, out: str) -> str:
    """Compile one oracle source file to a shared library (atomic rename)."""
    d = os.path.dirname(os.path.abspath(out))
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=d)
    os.close(fd)
    try:
        subprocess.run(["gcc", *CFLAGS, "-I", HERE, "-o", tmp, src, "-lm"], check=True)
        os.replace(tmp, out)
    finally:
        if os.path.exists(tmp):
            os.unlink(tmp)
    return out


def _stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(p) > t for p in (SRC, HDR))


def build(force: bool = False) -> str:
    """Build oracle/liboracle.so with gcc if it is missing or out of date."""
    if force or _stale():
        compile_oracle(SRC, LIB)
    return LIB


def _u16(a):
    return np.ascontiguousarray(a, dtype=np.uint16)


class Oracle:
    """One loaded copy of the oracle library."""

    def __init__(self, path: str):
        L = ctypes.CDLL(path)
        u16p = ctypes.POINTER(ctypes.c_uint16)
        f32p = ctypes.POINTER(ctypes.c_float)
        f64p = ctypes.POINTER(ctypes.c_double)
        L.arf_oracle_widen.argtypes = [ctypes.c_int, ctypes.c_uint16]
        L.arf_oracle_widen.restype = ctypes.c_float
        L.arf_oracle_narrow_f32.argtypes = [ctypes.c_int, ctypes.c_float]
        L.arf_oracle_narrow_f32.restype = ctypes.c_uint16
        L.arf_oracle_narrow_f64.argtypes = [ctypes.c_int, ctypes.c_double]
        L.arf_oracle_narrow_f64.restype = ctypes.c_uint16
        L.arf_oracle_widen_n.argtypes = [ctypes.c_int, u16p, f32p, ctypes.c_int64]
        L.arf_oracle_widen_n.restype = None
        L.arf_oracle_narrow_f32_n.argtypes = [ctypes.c_int, f32p, u16p, ctypes.c_int64]
        L.arf_oracle_narrow_f32_n.restype = None
        L.arf_oracle_narrow_f64_n.argtypes = [ctypes.c_int, f64p, u16p, ctypes.c_int64]
        L.arf_oracle_narrow_f64_n.restype = None
        L.arf_oracle_inv_rms.argtypes = [ctypes.c_int, u16p, ctypes.c_int64, ctypes.c_float, f64p]
        L.arf_oracle_inv_rms.restype = ctypes.c_double
        L.arf_oracle_run.argtypes = [
            ctypes.c_int, ctypes.c_int, ctypes.POINTER(ctypes.c_void_p),
            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_float,
            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int,
        ]
        L.arf_oracle_run.restype = ctypes.c_int
        L.arf_oracle_run_general.argtypes = [
            ctypes.c_int, ctypes.c_int, ctypes.POINTER(ctypes.c_void_p), ctypes.c_int, ctypes.c_int64,
            ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_float,
            ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
            ctypes.c_int,
        ]
        L.arf_oracle_run_general.restype = ctypes.c_int
        self.lib = L
        self.path = path

    def widen(self, dtype: int, bits) -> np.ndarray:
        """16-bit codes -> exact float32 values."""
        b = _u16(bits)
        out = np.empty(b.shape, np.float32)
        self.lib.arf_oracle_widen_n(dtype, b.ctypes.data_as(ctypes.POINTER(ctypes.c_uint16)),
                                    out.ctypes.data_as(ctypes.POINTER(ctypes.c_float)), b.size)
        return out

    def narrow_f32(self, dtype: int, v) -> np.ndarray:
        """float32 values -> nearest 16-bit codes (ties to even)."""
        a = np.ascontiguousarray(v, dtype=np.float32)
        out = np.empty(a.shape, np.uint16)
        self.lib.arf_oracle_narrow_f32_n(dtype, a.ctypes.data_as(ctypes.POINTER(ctypes.c_float)),
                                         out.ctypes.data_as(ctypes.POINTER(ctypes.c_uint16)), a.size)
        return out

    def narrow_f64(self, dtype: int, v) -> np.ndarray:
        """float64 values -> nearest 16-bit codes (ties to even, one rounding)."""
        a = np.ascontiguousarray(v, dtype=np.float64)
        out = np.empty(a.shape, np.uint16)
        self.lib.arf_oracle_narrow_f64_n(dtype, a.ctypes.data_as(ctypes.POINTER(ctypes.c_double)),
                                         out.ctypes.data_as(ctypes.POINTER(ctypes.c_uint16)), a.size)
        return out

    def inv_rms(self, dtype: int, x_row, eps: float):
        """(1/sqrt(sum x^2 / H + eps), sum x^2) of one row of codes, in float64."""
        x = _u16(x_row)
        ss = ctypes.c_double()
        inv = self.lib.arf_oracle_inv_rms(dtype, x.ctypes.data_as(ctypes.POINTER(ctypes.c_uint16)),
                                          x.size, eps, ctypes.byref(ss))
        return inv, ss.value

    def run(self, pattern: int, partials, residual=None, gamma=None, eps: float = 0.0,
            dtype: int = BF16, residual_out=None):
        """Run the epilogue on host arrays of codes.

        partials: sequence of W uint16 arrays of shape [M, H], rank order as
        given. Returns (out, residual_out); residual_out is None for
        kAllReduce. ``residual_out`` may be passed in (for example the
        residual array itself, to run in place).
        """
        P = [_u16(p) for p in partials]
        if not P:
            raise ValueError("W must be >= 1")
        M, H = P[0].shape
        for p in P:
            if p.shape != (M, H):
                raise ValueError("all partials must have the same [M, H] shape")
        ptrs = (ctypes.c_void_p * len(P))(*[p.ctypes.data for p in P])
        out = np.empty((M, H), np.uint16)
        r_ptr = g_ptr = ro_ptr = None
        R = G = None
        if pattern == AR_RESIDUAL_RMSNORM:
            if residual is None or gamma is None:
                raise ValueError("kARResidualRMSNorm needs residual and gamma")
            R = residual if (isinstance(residual, np.ndarray) and residual.dtype == np.uint16
                             and residual.flags.c_contiguous) else _u16(residual)
            R = R.reshape(M, H)
            G = _u16(gamma).reshape(H)
            if residual_out is None:
                residual_out = np.empty((M, H), np.uint16)
            r_ptr, g_ptr, ro_ptr = R.ctypes.data, G.ctypes.data, residual_out.ctypes.data
        rc = self.lib.arf_oracle_run(pattern, len(P), ptrs, r_ptr, g_ptr, float(eps),
                                     out.ctypes.data, ro_ptr, M, H, dtype)
        if rc != 0:
            raise ValueError(f"arf_oracle_run rejected its arguments (rc={rc})")
        return out, residual_out


F32 = 2  # partial dtype code for binary32 partials


def _rows(a, name, H=None):
    """(row stride in elements, array) of a 2-D array whose rows may be wider
    than H (a column slice of a wider array); elements must be contiguous."""
    if a.ndim != 2 or a.strides[1] != a.itemsize or a.strides[0] % a.itemsize:
        raise ValueError(f"{name}: rows must be contiguous")
    return a.strides[0] // a.itemsize


def run_general_with(o, pattern, partials, residual=None, gamma=None, eps=0.0, dtype=BF16, out=None,
                     residual_out=None):
    """The general entry point: partials are uint16 codes or float32 arrays
    of shape [M, H], possibly column slices of wider arrays (row strides are
    read from the arrays); out / residual_out likewise (allocated contiguous
    when None). Returns (out, residual_out)."""
    P = list(partials)
    M, H = P[0].shape
    pdtype = F32 if P[0].dtype == np.float32 else dtype
    ldp = _rows(P[0], "partials")
    for p in P:
        if p.shape != (M, H) or p.dtype != P[0].dtype or _rows(p, "partials") != ldp:
            raise ValueError("partials must share shape, dtype and row stride")
    ptrs = (ctypes.c_void_p * len(P))(*[p.ctypes.data for p in P])
    if out is None:
        out = np.empty((M, H), np.uint16)
    r_ptr = g_ptr = ro_ptr = None
    ldr = ldro = H
    if pattern == AR_RESIDUAL_RMSNORM:
        if residual_out is None:
            residual_out = np.empty((M, H), np.uint16)
        ldr, ldro = _rows(residual, "residual"), _rows(residual_out, "residual_out")
        G = _u16(gamma).reshape(H)
        r_ptr, g_ptr, ro_ptr = residual.ctypes.data, G.ctypes.data, residual_out.ctypes.data
    rc = o.lib.arf_oracle_run_general(pattern, len(P), ptrs, pdtype, ldp, r_ptr, ldr, g_ptr, float(eps),
                                      out.ctypes.data, _rows(out, "out"), ro_ptr, ldro, M, H, dtype)
    if rc != 0:
        raise ValueError(f"arf_oracle_run_general rejected its arguments (rc={rc})")
    return out, residual_out


Oracle.run_general = run_general_with

_default = None


def default() -> Oracle:
    """The oracle built from this directory's source (built on first use)."""
    global _default
    if _default is None:
        _default = Oracle(build())
    return _default


def widen(dtype, bits):
    return default().widen(dtype, bits)


def narrow_f32(dtype, v):
    return default().narrow_f32(dtype, v)


def narrow_f64(dtype, v):
    return default().narrow_f64(dtype, v)


def inv_rms(dtype, x_row, eps):
    return default().inv_rms(dtype, x_row, eps)


def run(pattern, partials, residual=None, gamma=None, eps=0.0, dtype=BF16, residual_out=None):
    return default().run(pattern, partials, residual, gamma, eps, dtype, residual_out)


def run_general(pattern, partials, residual=None, gamma=None, eps=0.0, dtype=BF16, out=None, residual_out=None):
    return default().run_general(pattern, partials, residual, gamma, eps, dtype, out, residual_out)
