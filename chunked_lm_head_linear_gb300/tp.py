"""Vocabulary-parallel (tensor-parallel) use of the fused LM-head cross-entropy.

Each rank holds the rows [vocab_offset, vocab_offset + V_shard) of W, all of H
and the global labels. Per token the ranks exchange 16 bytes of statistics
(max, sum-exp, label logit, has-label) -- an all-gather -- and merge them in
rank order, which gives every rank the same lse and loss; the backward's
partial dH is summed with an all-reduce, and each rank's dW rows are local.
The merge is the streaming max / sum-exp rule of "MindSpeed fusion
optimisation: principles and practice" (section 3.2), applied across
vocabulary shards instead of key blocks.

Two schedules:
  "stored" (default)  per chunk of tokens: statistics and the shard's exp tile,
                      the all-gather of the chunk's statistics, then the
                      chunk's backward from the kept tile (6 N V_shard d flops
                      per rank; memory of one chunk's tile);
  "recompute"         one all-gather for all tokens, the backward recomputing
                      the logits (8 N V_shard d flops; nothing kept between
                      the calls).
"""
from __future__ import annotations


def _chunk_size(N: int, chunk_tokens) -> int:
    """The chunk the library uses for these options (0: 4096), capped at N."""
    c = int(chunk_tokens or 0) or 4096
    return max(1, min(c, N))


def vocab_parallel_fwd_bwd(H, W_shard, y, vocab_offset: int, V_total: int, grad_loss=None, *, group=None,
                           backend=None, method: str = "stored", **opt_kw):
    """Returns (loss, lse, dH, dW_shard): loss, lse and dH are the full-vocabulary
    ones (identical on all ranks of the group), dW_shard this rank's rows.

    ``backend`` is an object with the shard calls (forward_stats, combine,
    backward for "recompute"; chunk_workspace, chunk_stats, chunk_backward,
    combine for "stored"); by default the CUDA library's ``lce`` functions.
    """
    import torch
    import torch.distributed as dist
    if method not in ("stored", "recompute"):
        raise ValueError('method must be "stored" or "recompute"')
    if backend is None:
        from . import lce

        class _Cuda:
            forward_stats = staticmethod(lce.lce_vshard_forward_stats)
            combine = staticmethod(lce.lce_vshard_combine)
            backward = staticmethod(lce.lce_vshard_backward)
            chunk_workspace = staticmethod(lce.vshard_chunk_workspace)
            chunk_stats = staticmethod(lce.lce_vshard_chunk_stats)
            chunk_backward = staticmethod(lce.lce_vshard_chunk_backward)
        backend = _Cuda
    world = dist.get_world_size(group)

    if method == "recompute":
        stats = backend.forward_stats(H, W_shard, y, vocab_offset, V_total, **opt_kw)
        gathered = [torch.empty_like(stats) for _ in range(world)]
        dist.all_gather(gathered, stats.contiguous(), group=group)
        stats_all = torch.stack(gathered).contiguous()          # [R, N, 4] in rank order
        loss, lse = backend.combine(stats_all, y, V_total, **opt_kw)
        dH, dW_shard = backend.backward(H, W_shard, y, vocab_offset, V_total, lse, grad_loss, **opt_kw)
        dist.all_reduce(dH, group=group)
        return loss, lse, dH, dW_shard

    if opt_kw.get("accumulate_dW"):
        raise ValueError("the stored schedule returns a new dW_shard; add it to an accumulator yourself")
    N, d = H.shape
    Vs = W_shard.shape[0]
    ftype = torch.float64 if H.dtype == torch.float64 else torch.float32
    chunk = opt_kw.get("chunk_tokens", 0)
    if chunk == "auto":
        from . import lce
        chunk = lce.auto_chunk(N, d, Vs, torch.cuda.mem_get_info(H.device)[0] // 2) if N > 0 else 0
    C = _chunk_size(N, chunk)
    opt_kw = dict(opt_kw, chunk_tokens=C)
    ws = backend.chunk_workspace(H, W_shard, y, **opt_kw)
    lse = torch.empty(N, dtype=ftype, device=H.device)
    dH = torch.empty((N, d), dtype=ftype, device=H.device)
    dW_shard = torch.zeros((Vs, d), dtype=ftype, device=H.device)
    per_chunk = []
    for c0 in range(0, N, C):
        rows = min(C, N - c0)
        stats = backend.chunk_stats(H, W_shard, y, vocab_offset, V_total, c0, rows, workspace=ws, **opt_kw)
        gathered = [torch.empty_like(stats) for _ in range(world)]
        dist.all_gather(gathered, stats.contiguous(), group=group)
        stats_all = torch.stack(gathered).contiguous()      # [R, rows, 4] in rank order
        backend.chunk_backward(H, W_shard, y, vocab_offset, V_total, c0, rows, stats_all, workspace=ws, lse=lse,
                               dH_partial=dH, dW_shard=dW_shard, grad_loss=grad_loss, **opt_kw)
        per_chunk.append(stats_all)
    stats_all = (torch.cat(per_chunk, dim=1) if per_chunk
                 else torch.empty((world, 0, 4), dtype=ftype, device=H.device))
    loss, _ = backend.combine(stats_all.contiguous(), y, V_total, **opt_kw)   # the loss over all chunks
    dist.all_reduce(dH, group=group)
    return loss, lse, dH, dW_shard
