"""Row-sharded RMSNorm over several processes (one GPU each).

Rows are independent units, so M rows split into contiguous blocks, one per
rank: the forward and dx need no exchange.  dgamma is a sum over every row
("Hướng dẫn Triton RMSNorm: kernel, backward…", section "Tổng không phải
trung bình"), so each rank's backward yields the dgamma of its own rows and
one exchange step finishes it: every rank all-gathers the per-rank float32
vectors, in rank order, and adds them in that order with the library's
rms_dgamma_combine kernel.  The total is bit for bit the same on every rank
and independent of the collective's own reduction order (an all-reduce would
add in whatever order its ring or tree takes).

This module only partitions rows and moves the per-rank vectors with
torch.distributed (NCCL between GPUs); every arithmetic step runs in the
library's kernels, through the same binding as the single-GPU calls.
"""
from __future__ import annotations

from . import ln_bwd, rms_bwd, rms_dgamma_combine


def row_block(M: int, world: int, rank: int):
    """[start, stop) of rank's contiguous rows: the first M % world ranks
    take one row more than the others."""
    if world < 1 or not 0 <= rank < world or M < 0:
        raise ValueError(f"bad partition: M={M}, world={world}, rank={rank}")
    base, extra = divmod(M, world)
    start = rank * base + min(rank, extra)
    return start, start + base + (1 if rank < extra else 0)


def gather_rank_ordered(local, group=None):
    """(world, N) tensor whose row r is rank r's ``local`` (N,) vector, on
    every rank.  NCCL gathers into one buffer; other backends (gloo) gather
    a list of rows that is stacked in rank order."""
    import torch
    import torch.distributed as dist

    world = dist.get_world_size(group)
    if dist.get_backend(group) == "nccl":
        out = torch.empty((world,) + tuple(local.shape), dtype=local.dtype, device=local.device)
        dist.all_gather_into_tensor(out, local.contiguous(), group=group)
        return out
    rows = [torch.empty_like(local) for _ in range(world)]
    dist.all_gather(rows, local.contiguous(), group=group)
    return torch.stack(rows)


def exchange_dgamma(local, dgamma, group=None, stream=None, combine=None):
    """dgamma = sum over ranks of every rank's ``local`` vector, added in rank
    order (``combine(stacked, dgamma)``, default the library kernel on the
    GPU).  With one rank (or no process group) dgamma is ``local``."""
    import torch.distributed as dist

    if not dist.is_available() or not dist.is_initialized() or dist.get_world_size(group) == 1:
        if dgamma.data_ptr() != local.data_ptr():
            dgamma.copy_(local)
        return dgamma
    stacked = gather_rank_ordered(local, group)
    if combine is None:
        rms_dgamma_combine(stacked, dgamma, stream=stream)
    else:
        combine(stacked, dgamma)
    return dgamma


def rms_bwd_sharded(dy, x, gamma, rstd, dx, dgamma, dgamma_local, workspace, gemma: int = 0,
                    inplace_dx: int = 0, group=None, stream=None):
    """rms_bwd over this rank's rows (dy, x, rstd, dx hold only them), then
    the dgamma exchange: dgamma_local (N,) float32 receives this rank's sum,
    dgamma (N,) the total over all ranks' rows."""
    rms_bwd(dy, x, gamma, rstd, dx, dgamma_local, workspace, gemma, inplace_dx, stream=stream)
    return exchange_dgamma(dgamma_local, dgamma, group, stream)


def ln_bwd_sharded(dy, x, w, mean, rstd, dx, dwdb, dwdb_local, workspace, inplace_dx: int = 0,
                   group=None, stream=None):
    """ln_bwd over this rank's rows with dw and db exchanged together:
    dwdb_local and dwdb are (2, N) float32, row 0 dw and row 1 db."""
    ln_bwd(dy, x, w, mean, rstd, dx, dwdb_local[0], dwdb_local[1], workspace, inplace_dx,
           stream=stream)
    exchange_dgamma(dwdb_local.view(-1), dwdb.view(-1), group, stream)
    return dwdb
