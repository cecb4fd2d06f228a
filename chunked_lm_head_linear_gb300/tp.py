"""Vocabulary-parallel (tensor-parallel) use of the fused LM-head cross-entropy.

Each rank holds the rows [vocab_offset, vocab_offset + V_shard) of W, all of H
and the global labels. Per token the ranks exchange 16 bytes of statistics
(max, sum-exp, label logit, has-label) -- an all-gather -- and merge them in
rank order, which gives every rank the same lse and loss; the backward's
partial dH is summed with an all-reduce, and each rank's dW rows are local.
The merge is the streaming max / sum-exp rule of "MindSpeed fusion
optimisation: principles and practice" (section 3.2), applied across
vocabulary shards instead of key blocks.
"""
from __future__ import annotations


def vocab_parallel_fwd_bwd(H, W_shard, y, vocab_offset: int, V_total: int, grad_loss=None, *, group=None,
                           backend=None, **opt_kw):
    """Returns (loss, lse, dH, dW_shard): loss, lse and dH are the full-vocabulary
    ones (identical on all ranks of the group), dW_shard this rank's rows.

    ``backend`` is an object with the three shard calls (forward_stats,
    combine, backward); by default the CUDA library's ``lce`` functions.
    """
    import torch
    import torch.distributed as dist
    if backend is None:
        from . import lce

        class _Cuda:
            forward_stats = staticmethod(lce.lce_vshard_forward_stats)
            combine = staticmethod(lce.lce_vshard_combine)
            backward = staticmethod(lce.lce_vshard_backward)
        backend = _Cuda
    world = dist.get_world_size(group)
    stats = backend.forward_stats(H, W_shard, y, vocab_offset, V_total, **opt_kw)
    gathered = [torch.empty_like(stats) for _ in range(world)]
    dist.all_gather(gathered, stats.contiguous(), group=group)
    stats_all = torch.stack(gathered).contiguous()          # [R, N, 4] in rank order
    loss, lse = backend.combine(stats_all, y, V_total, **opt_kw)
    dH, dW_shard = backend.backward(H, W_shard, y, vocab_offset, V_total, lse, grad_loss, **opt_kw)
    dist.all_reduce(dH, group=group)
    return loss, lse, dH, dW_shard
