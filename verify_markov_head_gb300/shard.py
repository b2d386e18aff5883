"""Data parallelism over requests: the host-side logic of a multi-rank step.

Requests are independent through drafting, confidence and verification
("DSpark：半自回归生成与置信度调度的投机解码", sections 整体架构 and 形式化定义):
each rank owns a contiguous block of the global batch and runs those steps on
its block alone.  Its random streams stay those of the unsharded batch
because every Philox counter carries the request's global index
(req_base + local index).

The one exchange is the prefix scheduler (same page, section 硬件感知前缀调度器;
"DeepSeek-AI与北京大学联手破局" sections 四, 五 on its asynchronous form): it ranks all
requests' draft positions together against one throughput curve, so the
survival lists are gathered from every rank, every rank runs the same
deterministic scheduler on the whole list, and each keeps the verify lengths
of its own block.  Nothing else crosses ranks.

This module holds only that logic and imports no compiled code: the
scheduler is passed in (the device scheduler on GPUs).
"""
from __future__ import annotations

from typing import Callable, Optional, Tuple


def shard_of(rank: int, world: int, B_total: int) -> Tuple[int, int]:
    """(first request, count) of `rank`'s contiguous block.  Blocks are
    equal: the batch must divide evenly, since the gathered lists are
    concatenated in rank order."""
    if world < 1 or not (0 <= rank < world):
        raise ValueError("rank out of range")
    if B_total % world:
        raise ValueError(f"global batch {B_total} does not split evenly over {world} ranks")
    n = B_total // world
    return rank * n, n


def gather_rows(x, group=None, out=None):
    """All ranks' equal-shaped blocks concatenated along dim 0, in rank order,
    into `out` ([world * rows, ...], contiguous) when given."""
    import torch
    import torch.distributed as dist

    world = dist.get_world_size(group)
    if out is None:
        out = torch.empty((world * x.shape[0],) + tuple(x.shape[1:]), dtype=x.dtype, device=x.device)
    if tuple(out.shape) != (world * x.shape[0],) + tuple(x.shape[1:]) or not out.is_contiguous():
        raise ValueError("gather target has the wrong shape")
    dist.all_gather(list(out.chunk(world, dim=0)), x.contiguous(), group=group)
    return out


def global_schedule(log_surv, log_surv_hist, schedule_fn: Callable, group=None, surv_out=None, hist_out=None):
    """Verify lengths of this rank's requests under the scheduler over all
    ranks' requests.

    log_surv [B_local, gamma] (and log_surv_hist, or None) are this rank's
    lists; schedule_fn(all_surv, all_hist) -> (K_all, n_total, theta) runs
    the scheduler on the gathered [world * B_local, gamma] lists (gathered
    into surv_out / hist_out when given).  Returns (K_local, n_total, theta,
    K_all), K_local a view of K_all's rows of this rank."""
    import torch.distributed as dist

    rank = dist.get_rank(group)
    world = dist.get_world_size(group)
    B_local = log_surv.shape[0]
    all_surv = gather_rows(log_surv, group, surv_out)
    all_hist: Optional[object] = None if log_surv_hist is None else gather_rows(log_surv_hist, group, hist_out)
    K_all, n_total, theta = schedule_fn(all_surv, all_hist)
    start, n = shard_of(rank, world, B_local * world)
    return K_all[start:start + n], n_total, theta, K_all
