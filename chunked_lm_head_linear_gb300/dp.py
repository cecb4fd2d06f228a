"""Data-parallel (over tokens) use of the fused LM-head cross-entropy.

Each rank holds a shard of the tokens and the full W. Everything per token
(lse, loss_i, dH) is local; the only exchange is
  1. the global count of valid labels, which must be known before the
     gradient tile is scaled by g/n (the first page's multi-rank ``loss_1d``
     anomaly, "XTuner on Ascend 910C: Qwen3.5-2B training optimisation",
     section 3.1.4, is a normalisation problem of exactly this kind), and
  2. a sum of dW (and of the per-rank partial losses) after the backward.
With the global count as denominator, the sum over ranks of the shards'
losses and dW equals the unsharded result.
"""
from __future__ import annotations


def global_valid_count(y, ignore_index: int = -100, group=None, *, V: int) -> int:
    """All-reduce (sum) of the number of labels the library counts: those that
    are not ignore_index and lie in [0, V). A label outside the vocabulary is
    an error the library reports (a device status bit) while it treats that
    row as ignored, so counting it here would give the ranks a denominator the
    one-rank call does not use."""
    import torch
    import torch.distributed as dist
    n = ((y != ignore_index) & (y >= 0) & (y < V)).sum().to(torch.int64).reshape(1)
    dist.all_reduce(n, group=group)
    return int(n.item())


def dp_fwd_bwd(H, W, y, grad_loss=None, *, n_global: int | None = None, group=None, compute=None,
               ignore_index: int = -100, **opt_kw):
    """One rank's fused forward + backward with the global denominator, then
    the sum of dW and of the loss over the group. Returns (loss, lse, dH, dW),
    where loss and dW are the global ones and lse, dH belong to this shard.

    ``compute`` defaults to the CUDA entry point ``lce.lce_fwd_bwd``.
    """
    import torch.distributed as dist
    if compute is None:
        from . import lce
        compute = lce.lce_fwd_bwd
    if n_global is None:
        n_global = global_valid_count(y, ignore_index, group, V=W.shape[0])
    loss, lse, dH, dW = compute(H, W, y, grad_loss, n_valid_override=n_global, ignore_index=ignore_index,
                                **opt_kw)
    dist.all_reduce(dW, group=group)
    dist.all_reduce(loss, group=group)
    return loss, lse, dH, dW
