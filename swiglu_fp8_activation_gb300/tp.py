"""Host side of the tensor-parallel all-reduce folded into the fused norm.

`allreduce_rmsnorm_add_quant` (the C entry point) sums the ranks' partial
rows and normalises them in one launch; this module holds the row partition
of the "two shot" form and its gather, for a process group of `world` ranks
(one per GPU). The pages' fused all-reduce + norm runs one stage for small
batches (every rank reads every partial and computes all rows) and two
stages beyond (each rank computes a slice of the rows, then the slices are
gathered): "[ROCm] Fuse per-token activation quant into RMSNorm for
per-channel quantized attention" (sglang PR 34502), review of the fused
collective (1-stage up to 128 KiB, 2-stage beyond); "[ROCm][MiniMax-M3.1]
Fuse MXFP8 quant into the add+RMSNorm and SwiGLU epilogues" (vllm PR 65478),
"Purpose" commit 1.

Peer access to the other ranks' partials (mapping their memory into this
process) and the barrier that makes them complete before the launch are the
caller's: `partials` is a list of tensors this rank can read.
"""
from __future__ import annotations

ONE_SHOT_MAX_BYTES = 128 * 1024   # the one-stage form up to this many bytes of one partial


def rank_rows(M: int, world: int, rank: int) -> tuple:
    """Rows [start, stop) of `rank` in the two-shot split of M rows over
    `world` ranks: contiguous blocks, the first M % world ranks one row more."""
    if world < 1 or not 0 <= rank < world or M < 0:
        raise ValueError(f"bad partition: M={M}, world={world}, rank={rank}")
    base, extra = divmod(M, world)
    start = rank * base + min(rank, extra)
    return start, start + base + (1 if rank < extra else 0)


def one_shot(M: int, H: int, elem_bytes: int = 2) -> bool:
    """Whether a partial of M rows of H elements is small enough for the
    one-stage form."""
    return M * H * elem_bytes <= ONE_SHOT_MAX_BYTES


def _gather_rows(t, world: int, rows: list, group=None):
    """All ranks' row slices of one output, in rank order (torch.distributed
    all_gather of slices padded to the largest), concatenated."""
    import torch
    import torch.distributed as dist
    most = max(b - a for a, b in rows)
    pad = torch.zeros((most,) + tuple(t.shape[1:]), dtype=t.dtype, device=t.device)
    pad[: t.shape[0]] = t
    wire = pad.view(torch.uint8)          # the bytes, whatever the type (every backend carries uint8)
    bufs = [torch.empty_like(wire) for _ in range(world)]
    dist.all_gather(bufs, wire, group=group)
    out = [b.view(t.dtype)[: rows[k][1] - rows[k][0]] for k, b in enumerate(bufs)]
    return torch.cat(out, dim=0)


def two_shot(compute, partials: list, residual, *, rank: int, world: int, group=None):
    """The two-shot form for this rank: `compute(partial_slices, residual_slice)`
    (the fused kernel on this rank's rows, returning (q, scale, normed or
    None, residual_out or None) with row-major scales) runs on rows
    rank_rows(M, world, rank) of every partial and of the residual; then every
    output's slices are gathered from all ranks into the full [M, ...]
    tensors, which are returned in the same order."""
    M = partials[0].shape[0]
    rows = [rank_rows(M, world, k) for k in range(world)]
    a, b = rows[rank]
    outs = compute([p[a:b] for p in partials], None if residual is None else residual[a:b])
    return tuple(None if o is None else _gather_rows(o, world, rows, group) for o in outs)
