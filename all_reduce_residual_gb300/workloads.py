"""Seeded synthetic inputs for the all-reduce fusion epilogue.

This module holds no arithmetic of the method itself: it only draws the
inputs. Both the CUDA path and the CPU oracle consume the exact bytes it
returns, so the two sides are compared on identical data.

Workloads (shapes and value distributions of the decode settings on the pages):

* ``small``    - W=2, M=8, H=1024, bf16, partials N(0,1); RMS only.
* ``llama_tp2``- Llama-3-8B-like TP2 decode (flashinfer PR #1507 "update
  allreduce to match trtllm", Description: llama3, tp2, gen-only):
  W=2, M=128, H=4096, bf16, partials N(0,0.5), eps=1e-5; both patterns.
* ``k3_tp8``   - K3-like TP8 decode sweep at hidden 7168 (tokenspeed PR #1075
  "route generic MNNVL AR patterns to upstream flashinfer", Summary):
  W=8, M in {1,...,2048}, bf16, partials N(0,0.25), eps=1e-6; both patterns.
* ``tp4_80mib``- the 79.994 MiB per-rank edge payload of single-node TP4
  (vLLM PR #53318 "Tune FlashInfer all-reduce selection on SM103",
  Performance table): W=4, M=5851, H=7168, bf16, N(0,1); both patterns.
* ``tp16_8mib``- the 7.998 MiB edge payload of four-node TP16 (same table):
  W=16, M=585, H=7168, fp16, partials N(0,0.1) with 1% of elements replaced
  by N(0,8) outliers; RMS only.

Recipe, every workload: seed = 1000 * config_id + tensor_id, tensor ids
0..W-1 for the partials, 100 for the residual, 101 for gamma. Values are drawn
in float32 (``sigma * randn``; residual N(0,1); gamma U(0.5,1.5)) and rounded
to the I/O dtype by torch's own conversion. N(0, s) means standard deviation s.
Outliers (tp16_8mib): an independent U(0,1) draw < 0.01 per element and per
partial selects an N(0,8) value instead of the N(0,0.1) one.
"""
from __future__ import annotations

from dataclasses import dataclass, replace
from typing import Optional

import numpy as np
import torch

K3_M_SWEEP = (1, 2, 4, 8, 16, 32, 64, 128, 256, 512, 1024, 2048)

TORCH_DTYPE = {"bf16": torch.bfloat16, "fp16": torch.float16}
ELEM_BYTES = 2


@dataclass(frozen=True)
class Workload:
    name: str
    config_id: int
    W: int
    M: int
    H: int
    dtype: str
    partial_sigma: float
    eps: float
    patterns: tuple
    outlier_frac: float = 0.0
    outlier_sigma: float = 0.0

    def with_m(self, M: int) -> "Workload":
        return replace(self, M=M)

    def read_bytes_per_call(self, pattern: str) -> int:
        """The reads among bytes_per_call: the partials, and for the RMS
        pattern the residual and gamma."""
        s, n = ELEM_BYTES, self.M * self.H
        if pattern == "allreduce":
            return self.W * n * s
        return (self.W + 1) * n * s + self.H * s

    def bytes_per_call(self, pattern: str) -> int:
        """Algorithmic HBM bytes of one call: every partial element read once,
        the residual read once, gamma once, each output written once."""
        s, n = ELEM_BYTES, self.M * self.H
        if pattern == "allreduce":
            return (self.W + 1) * n * s
        return (self.W + 3) * n * s + self.H * s


WORKLOADS = {
    "small": Workload("small", 1, 2, 8, 1024, "bf16", 1.0, 1e-6, ("rmsnorm",)),
    "llama_tp2": Workload("llama_tp2", 2, 2, 128, 4096, "bf16", 0.5, 1e-5, ("allreduce", "rmsnorm")),
    "k3_tp8": Workload("k3_tp8", 3, 8, 2048, 7168, "bf16", 0.25, 1e-6, ("allreduce", "rmsnorm")),
    "tp4_80mib": Workload("tp4_80mib", 4, 4, 5851, 7168, "bf16", 1.0, 1e-6, ("allreduce", "rmsnorm")),
    "tp16_8mib": Workload("tp16_8mib", 5, 16, 585, 7168, "fp16", 0.1, 1e-6, ("rmsnorm",),
                          outlier_frac=0.01, outlier_sigma=8.0),
}


# Shapes beyond the five above, measured in the benchmark's sweep because the
# planner sends them to kernels the five do not reach: the bulk-copy kernel
# for a rank count without a compiled kernel (W = 3 and W = 12), for fp16
# rows of two chunks per thread with one rank and many rows, and for rows of
# 32768 elements and of 32776 (more than one CTA's row, many rows); the row
# kernel's one-CTA-per-row grid for the 80 MiB shape in fp16; and the
# elementwise kernels' 16-byte form for H not a multiple of 8. Same input
# recipe.
EXTRA_WORKLOADS = {
    "w3_generic": Workload("w3_generic", 6, 3, 2000, 7168, "bf16", 0.5, 1e-6, ("rmsnorm",)),
    "w12_generic": Workload("w12_generic", 7, 12, 585, 7168, "fp16", 0.1, 1e-6, ("rmsnorm",)),
    "tp4_80mib_fp16": Workload("tp4_80mib_fp16", 8, 4, 5851, 7168, "fp16", 1.0, 1e-6, ("rmsnorm",)),
    "h32768": Workload("h32768", 9, 4, 512, 32768, "bf16", 1.0, 1e-6, ("rmsnorm",)),
    "w1_fp16": Workload("w1_fp16", 10, 1, 4972, 7168, "fp16", 1.0, 1e-6, ("rmsnorm",)),
    "h32776": Workload("h32776", 11, 2, 1024, 32776, "bf16", 1.0, 1e-6, ("rmsnorm",)),
    "odd_h4098": Workload("odd_h4098", 12, 2, 4096, 4098, "bf16", 0.5, 1e-5, ("allreduce", "rmsnorm")),
}
# The kernel path the planner takes for each extra shape on GB300, from its
# measured plan table (the closed-form rules send w12_generic, h32768 and
# w1_fp16 to the bulk kernel, and odd_h4098's kAllReduce to the elementwise
# kernel). A dict gives the path per pattern.
EXTRA_PATHS = {"w3_generic": "bulk", "w12_generic": "cluster", "tp4_80mib_fp16": "row, one CTA per row",
               "h32768": "row", "w1_fp16": "row, one CTA per row", "h32776": "bulk",
               "odd_h4098": {"allreduce": "flat", "rmsnorm": "elem"}}


def extra_path(name: str, pattern: str) -> str:
    """The kernel path EXTRA_PATHS names for one pattern of an extra shape."""
    v = EXTRA_PATHS[name]
    return v[pattern] if isinstance(v, dict) else v


def custom(W: int, M: int, H: int, dtype: str = "bf16", sigma: float = 1.0,
           eps: float = 1e-6, config_id: int = 900) -> Workload:
    """An ad-hoc shape (edge cases in the tests) with the same recipe."""
    return Workload(f"custom_W{W}_M{M}_H{H}_{dtype}", config_id, W, M, H, dtype, sigma, eps,
                    ("allreduce", "rmsnorm"))


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _normal(shape, sigma: float, seed: int, device) -> torch.Tensor:
    return torch.randn(shape, generator=_gen(seed, device), dtype=torch.float32, device=device) * sigma


@dataclass
class Inputs:
    workload: Workload
    partials: list          # W tensors [M, H] of the I/O dtype
    residual: torch.Tensor  # [M, H]
    gamma: torch.Tensor     # [H]


def make_inputs(wl: Workload, device="cpu", M: Optional[int] = None) -> Inputs:
    """Draw the seeded inputs of workload ``wl`` (optionally at another M)."""
    if M is not None:
        wl = wl.with_m(M)
    dt = TORCH_DTYPE[wl.dtype]
    shape = (wl.M, wl.H)
    base = 1000 * wl.config_id
    partials = []
    for r in range(wl.W):
        g = _gen(base + r, device)
        v = torch.randn(shape, generator=g, dtype=torch.float32, device=device) * wl.partial_sigma
        if wl.outlier_frac > 0.0:
            pick = torch.rand(shape, generator=g, dtype=torch.float32, device=device) < wl.outlier_frac
            out = torch.randn(shape, generator=g, dtype=torch.float32, device=device) * wl.outlier_sigma
            v = torch.where(pick, out, v)
        partials.append(v.to(dt))
    residual = _normal(shape, 1.0, base + 100, device).to(dt)
    gamma = (0.5 + torch.rand((wl.H,), generator=_gen(base + 101, device),
                              dtype=torch.float32, device=device)).to(dt)
    return Inputs(wl, partials, residual, gamma)


def codes(t: torch.Tensor) -> np.ndarray:
    """The raw 16-bit codes of a CPU bf16/fp16 tensor as a numpy uint16 array."""
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def from_codes(a: np.ndarray, dtype: str) -> torch.Tensor:
    """A CPU tensor of the I/O dtype holding the given uint16 codes."""
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint16).view(np.int16)).view(TORCH_DTYPE[dtype])
