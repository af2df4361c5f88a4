"""torch.autograd.Function wrappers over the C-ABI row pass.

The axolotl write-up ("2. benchmarks/bench_selective_logsoftmax.py") wraps its forward and
backward kernels in a custom autograd Function; these are the same idea over this
library's entry points.  Marshalling only: every step runs in the CUDA kernels.

* ``grpo_loss(logits, idx, adv, ...)``        -> per-token loss [B*L] (+ aux dict)
* ``selective_log_softmax(logits, idx, T)``  -> logp [B*L]
* ``entropy(logits, T)``                     -> H [B*L]

Gradients flow to ``logits`` only (the other inputs are treated as constants, as in GRPO).
The backward of ``grpo_loss`` receives d(objective)/d(loss_r) per token from autograd, which
is exactly the per-token ``dloss`` of grpo_loss_bwd.
"""

from __future__ import annotations

import torch

from . import binding as rp


class GRPOLossFunction(torch.autograd.Function):
    @staticmethod
    def forward(ctx, logits, idx, adv, old_logp, ref_logp, mask, T, beta, eps_low, eps_high):
        out = rp.grpo_loss_fwd(logits, idx, adv, T=T, beta=beta, eps_low=eps_low, eps_high=eps_high,
                               old_logp=old_logp, ref_logp=ref_logp, mask=mask, with_entropy=True)
        empty = torch.empty(0)
        ctx.save_for_backward(logits, idx, adv, old_logp if old_logp is not None else empty,
                              ref_logp if ref_logp is not None else empty, mask if mask is not None else empty,
                              out["logp"], out["lse"])
        ctx.has = (old_logp is not None, ref_logp is not None, mask is not None)
        ctx.scalars = (T, beta, eps_low, eps_high)
        ctx.mark_non_differentiable(out["logp"], out["kl"], out["is_clipped"], out["entropy"])
        return out["loss"], out["logp"], out["kl"], out["is_clipped"], out["entropy"]

    @staticmethod
    def backward(ctx, dloss, *unused):
        logits, idx, adv, old, ref, mask, logp, lse = ctx.saved_tensors
        has_old, has_ref, has_mask = ctx.has
        T, beta, el, eh = ctx.scalars
        # autograd may hand over an expanded (stride-0) tensor, e.g. from loss.sum()
        dl = rp.grpo_loss_bwd(logits, idx, adv, dloss.float().contiguous(), logp, lse, T=T, beta=beta,
                              eps_low=el, eps_high=eh, old_logp=old if has_old else None,
                              ref_logp=ref if has_ref else None, mask=mask if has_mask else None)
        return dl, None, None, None, None, None, None, None, None, None


def grpo_loss(logits, idx, adv, *, T=1.0, beta=0.0, eps_low=0.2, eps_high=0.2, old_logp=None, ref_logp=None,
              mask=None):
    """Per-token GRPO loss [B*L] and a dict of the forward's other outputs (logp, kl,
    is_clipped, entropy).  ``loss`` is differentiable with respect to ``logits``."""
    loss, logp, kl, clipped, ent = GRPOLossFunction.apply(logits, idx, adv, old_logp, ref_logp, mask, T, beta,
                                                          eps_low, eps_high)
    return loss, {"logp": logp, "kl": kl, "is_clipped": clipped, "entropy": ent}


class SelectiveLogSoftmaxFunction(torch.autograd.Function):
    @staticmethod
    def forward(ctx, logits, idx, T):
        logp, lse = rp.selective_log_softmax_fwd(logits, idx, T=T)
        ctx.save_for_backward(logits, idx, lse)
        ctx.T = T
        return logp

    @staticmethod
    def backward(ctx, dlogp):
        logits, idx, lse = ctx.saved_tensors
        return rp.selective_log_softmax_bwd(logits, idx, dlogp.float().contiguous(), lse, T=ctx.T), None, None


def selective_log_softmax(logits, idx, T=1.0):
    """log_softmax(logits / T)[idx] per row, differentiable with respect to ``logits``."""
    return SelectiveLogSoftmaxFunction.apply(logits, idx, T)


class EntropyFunction(torch.autograd.Function):
    @staticmethod
    def forward(ctx, logits, T):
        H, lse = rp.entropy_from_logits(logits, T=T, return_lse=True)
        ctx.save_for_backward(logits, lse, H)
        ctx.T = T
        return H

    @staticmethod
    def backward(ctx, dH):
        logits, lse, H = ctx.saved_tensors
        return rp.entropy_from_logits_bwd(logits, dH.float().contiguous(), lse, H, T=ctx.T), None


def entropy(logits, T=1.0):
    """Per-row entropy of softmax(logits / T), differentiable with respect to ``logits``."""
    return EntropyFunction.apply(logits, T)
