"""Synchronized BatchNorm over a batch split across processes.

Each process runs the local halves in libnrm (per-channel partial statistics,
then the normalization with the combined ones); this module only moves the
small binary64 arrays between processes with torch.distributed (an
all-gather in rank order, so every process combines the same parts in the
same order and gets the same statistics).  With no process group, or a
group of one, it is bn_fwd_train / bn_bwd computed through the same pieces.
"""
from __future__ import annotations

import torch

from . import _binding as B


def _world(group):
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return None, 1
    return dist, dist.get_world_size(group)


def exchange_parts(local: torch.Tensor, group=None) -> torch.Tensor:
    """All-gather this process's [C, k] array: returns [world, C, k] in rank
    order (a view of `local` itself when there is a single process)."""
    dist, world = _world(group)
    if world == 1:
        return local.unsqueeze(0)
    parts = [torch.empty_like(local) for _ in range(world)]
    dist.all_gather(parts, local.contiguous(), group=group)
    return torch.stack(parts)


def global_count(local_count: int, device, group=None) -> int:
    """Sum over processes of the local batch * HW."""
    dist, world = _world(group)
    if world == 1:
        return int(local_count)
    t = torch.tensor([local_count], dtype=torch.int64, device=device)
    dist.all_reduce(t, group=group)
    return int(t.item())


def sync_bn_fwd_train(x, gamma=None, beta=None, running_mean=None, running_var=None, eps=1e-5,
                      momentum=0.1, group=None):
    """BatchNorm2d training forward with statistics over the whole distributed
    batch.  Returns (y, save_mean, save_rstd) for the local batch."""
    parts = exchange_parts(B.bn_fwd_partial_stats(x), group)
    return B.bn_fwd_apply_stats(x, parts, gamma, beta, running_mean, running_var, eps, momentum)


def sync_bn_bwd(dy, x, save_mean, save_rstd, gamma=None, group=None):
    """BatchNorm2d training backward with the sums over the whole distributed
    batch.  Returns (dx, dgamma, dbeta) for the local batch."""
    batch, c = x.shape[0], x.shape[1]
    hw = x.numel() // (batch * c) if batch * c else 0
    parts = exchange_parts(B.bn_bwd_partial_sums(dy, x, save_mean, save_rstd), group)
    count = global_count(batch * hw, x.device, group)
    return B.bn_bwd_apply_sums(dy, x, save_mean, save_rstd, parts, count, gamma)
