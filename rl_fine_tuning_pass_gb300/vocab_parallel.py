"""Vocabulary-parallel GRPO loss over ranks that each hold a column shard of the logits.

Each rank holds the columns [vocab_start, vocab_start + V_k) of every row (a
vocabulary-split LM head).  The row pass needs one exchange per step: an all-gather of a
4-float statistic per row.  After it, every rank holds the full rows' lse, logp, entropy
and GRPO terms (the same values on every rank), and each rank's backward writes its own
columns of dlogits with no further exchange.

This module orchestrates only: the statistics, the merge and the backward run in the
CUDA kernels (``grpo_vocab_shard_stats``, ``grpo_vocab_combine`` and
``grpo_loss_bwd_vocab_shard``); ``torch.distributed`` carries the all-gathers (NCCL on
GPUs).  The entry points are looked up on ``kernels`` (the binding module) at call time.
"""

from __future__ import annotations

import torch
import torch.distributed as dist

from . import binding as kernels


def gather_vocab_starts(vocab_local: int, group=None, device="cpu"):
    """Shard boundaries [0, V_0, V_0 + V_1, ..., V] from every rank's shard width, in rank
    order.  One small all-gather; call it once per model, not per step."""
    world = dist.get_world_size(group)
    mine = torch.tensor([int(vocab_local)], dtype=torch.int64, device=device)
    widths = [torch.empty_like(mine) for _ in range(world)]
    dist.all_gather(widths, mine, group=group)
    starts = [0]
    for w in widths:
        starts.append(starts[-1] + int(w.item()))
    return starts


def gather_stats(stats: torch.Tensor, group=None) -> torch.Tensor:
    """All-gather of every rank's [B*L, 4] shard statistic into [world, B*L, 4] (rank order)."""
    world = dist.get_world_size(group)
    parts = [torch.empty_like(stats) for _ in range(world)]
    dist.all_gather(parts, stats.contiguous(), group=group)
    return torch.stack(parts)


def grpo_loss_fwd_vocab_parallel(logits_shard, vocab_starts, idx, adv, *, T, beta, eps_low, eps_high,
                                 old_logp=None, ref_logp=None, mask=None, with_entropy=True, group=None,
                                 dev_err=None):
    """Forward of the GRPO loss on this rank's shard.  Returns the full rows' outputs (loss,
    logp, lse, kl, is_clipped, entropy, p_rest), the same on every rank of the group."""
    rank = dist.get_rank(group)
    B, L = (logits_shard.shape[0], logits_shard.shape[1]) if logits_shard.dim() == 3 else (1, logits_shard.shape[0])
    if vocab_starts[rank + 1] - vocab_starts[rank] != logits_shard.shape[-1]:
        raise ValueError("this rank's shard width does not match vocab_starts")
    stats = kernels.grpo_vocab_shard_stats(logits_shard, vocab_starts[rank], T=T, idx=idx, mask=mask)
    stats_all = gather_stats(stats, group)
    return kernels.grpo_vocab_combine(stats_all, vocab_starts, B, L, T=T, idx=idx, adv=adv, grpo=True, beta=beta,
                                      eps_low=eps_low, eps_high=eps_high, old_logp=old_logp, ref_logp=ref_logp,
                                      mask=mask, with_entropy=with_entropy, dev_err=dev_err)


def grpo_loss_bwd_vocab_parallel(logits_shard, vocab_starts, idx, adv, dloss, fwd, *, T, beta, eps_low, eps_high,
                                 old_logp=None, ref_logp=None, mask=None, dlogits=None, group=None, dev_err=None):
    """This rank's columns of dlogits, from the forward's outputs ``fwd`` (no exchange)."""
    rank = dist.get_rank(group)
    return kernels.grpo_loss_bwd_vocab_shard(
        logits_shard, vocab_starts[rank], vocab_starts[-1], idx, adv, dloss, fwd["logp"], fwd["lse"],
        fwd["p_rest"], T=T, beta=beta, eps_low=eps_low, eps_high=eps_high, old_logp=old_logp,
        ref_logp=ref_logp, mask=mask, dlogits=dlogits, dev_err=dev_err)
