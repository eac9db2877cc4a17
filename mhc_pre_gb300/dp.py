"""Data parallelism for the mHC layer: split the tokens, sum the parameter
gradients.

Every token is independent in all four ops (openPangu 2.0 notes, section 5.3:
the norm, the projection, the gates, Sinkhorn and both mixes act on one
token's n streams).  A batch is therefore split by tokens across ranks, and
the forward needs no exchange.  The parameters phi, b and alpha are shared by
all tokens, so the backward's one exchange is the sum over ranks of the
dphi, db and dalpha that ``mhc_pre_bwd`` returns for each rank's tokens.
"""

from __future__ import annotations


def shard_range(T: int, rank: int, world: int) -> tuple[int, int]:
    """Token range [start, stop) of ``rank`` when T tokens are split over
    ``world`` ranks in contiguous blocks whose sizes differ by at most one
    (the first T % world ranks take one more).  A rank may get no token."""
    if world < 1 or not 0 <= rank < world or T < 0:
        raise ValueError("need world >= 1, 0 <= rank < world and T >= 0")
    base, extra = divmod(T, world)
    start = rank * base + min(rank, extra)
    return start, start + base + (1 if rank < extra else 0)


def allreduce_param_grads(dphi, db, dalpha, group=None) -> None:
    """Sum dphi [K, G], db [G] and dalpha [3] over the ranks of ``group``,
    in place, with one all-reduce of a packed buffer.

    The tensors must share a device and dtype (fp32 from ``mhc_pre_bwd``).
    The sum is the full-batch gradient, since each rank's values are sums over
    its own tokens."""
    import torch
    import torch.distributed as dist

    parts = (dphi, db, dalpha)
    flat = torch.cat([p.reshape(-1) for p in parts])
    dist.all_reduce(flat, op=dist.ReduceOp.SUM, group=group)
    off = 0
    for p in parts:
        p.copy_(flat[off:off + p.numel()].view_as(p))
        off += p.numel()
