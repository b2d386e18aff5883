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


# --------------------------------------------------------------------------- #
# Vocabulary split for one request or a few (the latency case)                 #
# --------------------------------------------------------------------------- #
# The Markov bias of a position spans the whole vocabulary ("DSpark：半自回归
# 生成与置信度调度的投机解码", section Markov Head：一阶转移偏置), so with V split
# over ranks every rank holds columns [v0, v1) of W2, U and the target logits
# and W1 whole.  Per draft position each rank forms its slice's partial state
# -- the Gumbel-max winner (score, global index, its logit) and the slice's
# log-sum-exp -- and one all-gather of these few numbers per request gives
# every rank the same draw, which the next position needs.  Verification
# gathers per walked row the slices' log-sum-exps and the target logit of the
# drafted token (from the rank that holds it), walks the accept test on every
# rank alike, and gathers the residual (or bonus) draw's partial winners.
# The merge rules are those of the device kernels across CTAs: larger score,
# then lower index; log-sum-exps add.  The partial states are computed by the
# callables passed in.  Host logic only: not measured on GPUs.

def _gather_parts(x, group=None):
    """[world, ...] stack of every rank's float64 tensor x."""
    import torch
    import torch.distributed as dist

    world = dist.get_world_size(group)
    out = [torch.empty_like(x) for _ in range(world)]
    dist.all_gather(out, x.contiguous(), group=group)
    return torch.stack(out)


def merge_draws(best, idx):
    """Per request, the rank whose draw wins: larger score, then lower index
    (best, idx [world, B]); returns (rank index [B], best [B], idx [B])."""
    import torch

    world = best.shape[0]
    win = torch.zeros(best.shape[1], dtype=torch.long)
    for r in range(1, world):
        better = (best[r] > best[win, torch.arange(best.shape[1])]) | (
            (best[r] == best[win, torch.arange(best.shape[1])]) & (idx[r] < idx[win, torch.arange(best.shape[1])]))
        win = torch.where(better, torch.full_like(win, r), win)
    ar = torch.arange(best.shape[1])
    return win, best[win, ar], idx[win, ar]


def merge_lse(lse):
    """log sum exp over ranks of per-rank log-sum-exps lse [world, ...]."""
    import torch

    m = lse.max(dim=0).values
    finite = torch.isfinite(m)
    safe = torch.where(finite, m, torch.zeros_like(m))
    return torch.where(finite, safe + torch.log(torch.exp(lse - safe).sum(dim=0)), m)


def split_v_draft(slice_draft: Callable, anchor, gamma: int, group=None):
    """The draft loop with V split over the ranks of `group`.

    slice_draft(k, prev) -> float64 [B, 4] of (best, idx, z_best, lse) on this
    rank's slice for position k (1-based), prev [B] the tokens of position
    k - 1 (the anchors at k = 1).  Returns (tok [B, gamma] int64, lse_q, z_tok)
    identical on every rank."""
    import torch

    prev = torch.as_tensor(anchor, dtype=torch.long).clone()
    B = prev.shape[0]
    tok = torch.zeros((B, gamma), dtype=torch.long)
    lse_q = torch.zeros((B, gamma), dtype=torch.float64)
    z_tok = torch.zeros((B, gamma), dtype=torch.float64)
    for k in range(1, gamma + 1):
        parts = _gather_parts(torch.as_tensor(slice_draft(k, prev), dtype=torch.float64), group)
        win, _, idx = merge_draws(parts[..., 0], parts[..., 1])
        ar = torch.arange(B)
        tok[:, k - 1] = idx.long()
        z_tok[:, k - 1] = parts[win, ar, 2]
        lse_q[:, k - 1] = merge_lse(parts[..., 3])
        prev = tok[:, k - 1].clone()
    return tok, lse_q, z_tok


def split_v_verify(row_lse: Callable, token_logit: Callable, uniform: Callable, residual: Callable,
                   bonus: Callable, tok, lse_q, z_tok, K, group=None):
    """Verification with V split over the ranks of `group`.

    row_lse() -> float64 [B, gamma] log sum exp(t / tau) of target rows
      0..gamma-1 on this rank's slice;
    token_logit() -> float64 [B, gamma] t / tau at the drafted token of row
      k-1 where this rank holds it, -inf elsewhere;
    uniform(b, k) -> the acceptance uniform of request b, position k;
    residual(b, j, lse_p, lse_q) -> (best_r, idx_r, best_p, idx_p) on this
      rank's slice of row j (0-based) of request b;
    bonus(b, k) -> (best, idx) of the bonus draw on row k of request b.
    Returns (accepted [B], final_tok [B]) identical on every rank."""
    import math

    import torch

    B, gamma = tok.shape
    lse_p = merge_lse(_gather_parts(torch.as_tensor(row_lse(), dtype=torch.float64), group))
    t_x = _gather_parts(torch.as_tensor(token_logit(), dtype=torch.float64), group).max(dim=0).values
    accepted = torch.zeros(B, dtype=torch.long)
    final = torch.zeros(B, dtype=torch.long)
    for b in range(B):
        Kb = int(K[b])
        rej = -1
        for k in range(1, Kb + 1):
            p = math.exp(float(t_x[b, k - 1]) - float(lse_p[b, k - 1]))
            q = math.exp(float(z_tok[b, k - 1]) - float(lse_q[b, k - 1]))
            if not (uniform(b, k) < min(1.0, p / q)):
                rej = k - 1
                break
        accepted[b] = Kb if rej < 0 else rej
        if rej >= 0:
            part = torch.as_tensor(residual(b, rej, float(lse_p[b, rej]), float(lse_q[b, rej])),
                                   dtype=torch.float64).reshape(1, 4)
            parts = _gather_parts(part, group)                      # [world, 1, 4]
            if bool(torch.isfinite(parts[:, 0, 0]).any()):
                _, _, idx = merge_draws(parts[..., 0], parts[..., 1])
            else:                                                    # no residual mass: the draw from p
                _, _, idx = merge_draws(parts[..., 2], parts[..., 3])
        else:
            part = torch.as_tensor(bonus(b, Kb), dtype=torch.float64).reshape(1, 2)
            parts = _gather_parts(part, group)
            _, _, idx = merge_draws(parts[..., 0], parts[..., 1])
        final[b] = int(idx[0])
    return accepted, final
