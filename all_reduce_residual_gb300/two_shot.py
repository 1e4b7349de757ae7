"""Row-sharded two-shot form of the epilogue over G ranks, one GPU each.

In tensor-parallel decode every rank holds its own partial [M,H] and the same
residual and gamma. The one-GPU library sums W partials that sit in one GPU's
memory; across G GPUs the same sum splits by rows, in two shots (the "two-shot"
all-reduce the source pages set beside the one-shot kernels: tokenspeed PR #1075
"route generic MNNVL AR patterns to upstream flashinfer", Summary, and vLLM
PR #53318 "Tune FlashInfer all-reduce selection on SM103", Tests):

1. Reduce-scatter by rows. The rows are cut into G contiguous blocks of
   ceil(M / G) rows (the last ones shorter or empty). One all-to-all sends
   block j of every rank's partial to rank j, so rank g holds block g of all G
   partials, stacked in source-rank order.
2. Rank g runs the epilogue on its block with W = G partials in rank order,
   through this library's kernels (arf_run), so every row is computed exactly
   as the one-GPU call computes it: the same binary32 sum in the same order,
   the same residual add and statistic.
3. All-gather. Every rank receives every block of out (and residual_out).

The exchange runs on torch.distributed (NCCL between GPUs; gloo for the host
tests), on byte views of the 16-bit tensors. No kernel of this library waits
on another GPU. The local step is a parameter, so the partition, the exchange
and the rank order can be checked on the host with a reference epilogue.
"""
from __future__ import annotations

from typing import Callable, Optional


def row_blocks(M: int, G: int) -> list:
    """[(m0, m1)] for g = 0..G-1: contiguous blocks of ceil(M / G) rows; the
    last blocks are shorter or empty. Their union is [0, M) in order."""
    if G < 1 or M < 0:
        raise ValueError("G must be >= 1 and M >= 0")
    mb = -(-M // G) if M > 0 else 0
    return [(min(g * mb, M), min((g + 1) * mb, M)) for g in range(G)]


def _world(group):
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()):
        return 1, 0
    return dist.get_world_size(group), dist.get_rank(group)


def _bytes(t):
    import torch

    return t.contiguous().view(torch.uint8)


def library_epilogue(ws) -> Callable:
    """The local step on CUDA tensors: arf_run on W = G stacked partials."""
    import all_reduce_residual_gb300 as arf

    def step(pattern, partials, residual, gamma, eps):
        return arf.run(ws, pattern, partials, residual, gamma, eps)

    return step


def two_shot(pattern, partial, residual=None, gamma=None, eps: float = 0.0, *, ws=None, group=None,
             epilogue: Optional[Callable] = None):
    """The epilogue over the G ranks of `group` (the default group, or one rank
    when torch.distributed is not initialised).

    partial: this rank's [M,H] partial (bf16/fp16, contiguous); residual
    [M,H] and gamma [H]: the same on every rank (kARResidualRMSNorm only).
    Every rank returns the full (out, residual_out); residual_out is None for
    kAllReduce. epilogue(pattern, partials, residual_block, gamma, eps) ->
    (out_block, residual_out_block) is the local step, by default arf_run
    through workspace `ws`.
    """
    import torch
    import torch.distributed as dist

    import all_reduce_residual_gb300 as arf

    pat = arf.pattern_code(pattern)
    rms = pat == arf.ARF_AR_RESIDUAL_RMSNORM
    if epilogue is None:
        if ws is None:
            raise ValueError("two_shot needs a workspace (ws) or an epilogue")
        epilogue = library_epilogue(ws)
    G, g = _world(group)
    M, H = partial.shape
    blocks = row_blocks(M, G)
    mb = blocks[0][1] - blocks[0][0]
    m0, m1 = blocks[g]
    n = m1 - m0
    dev, dt = partial.device, partial.dtype

    # 1. reduce-scatter by rows: block j of every rank's partial to rank j
    if G == 1:
        recv = partial.contiguous().view(1, M, H)
    else:
        send = torch.zeros((G * mb, H), dtype=dt, device=dev)
        send[:M].copy_(partial)
        recv = torch.empty((G, mb, H), dtype=dt, device=dev)
        dist.all_to_all_single(_bytes(recv).view(G * mb, -1), _bytes(send), group=group)

    # 2. the epilogue on this rank's rows, partials in source-rank order
    out_b = torch.zeros((mb, H), dtype=dt, device=dev)
    ro_b = torch.zeros((mb, H), dtype=dt, device=dev) if rms else None
    if n > 0:
        parts = [recv[r, :n] for r in range(G)]
        o, ro = epilogue(pat, parts, residual[m0:m1] if rms else None, gamma if rms else None, eps)
        out_b[:n].copy_(o)
        if rms:
            ro_b[:n].copy_(ro)
    if G == 1:
        return out_b[:M], (ro_b[:M] if rms else None)

    # 3. all-gather every rank's block
    def gather(block):
        parts = [torch.empty((mb, H), dtype=dt, device=dev) for _ in range(G)]
        dist.all_gather([_bytes(p) for p in parts], _bytes(block), group=group)
        return torch.cat(parts, 0)[:M]

    out = gather(out_b)
    return out, (gather(ro_b) if rms else None)
