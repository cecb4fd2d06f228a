"""FSDP-style use of the fused LM-head cross-entropy: W stored sharded by
vocabulary rows, dW reduced back to the owners slice by slice while the
backward is still running.

FSDP shards every parameter evenly over the data-parallel ranks, gathers a
layer's parameters before it computes and shards them again afterwards; its
communication is hidden when the computation around it takes longer ("XTuner
V1 introduction", communication masking section). The first page's section
3.2.1 ("XTuner on Ascend 910C: Qwen3.5-2B training optimisation") adds that
the gather should be ordered on the compute stream rather than left on a side
stream whose memory the compute stream cannot reuse. For the LM head the
mirror step of the backward is the reduction of dW [V, d] fp32, the largest
gradient of the model: each rank needs only the sum over ranks of its own
rows.

Here:
  * ``owner_bounds`` cuts the vocabulary into per-rank row ranges whose
    interior bounds are multiples of the dW tile height (256), so that a
    slice of dW never straddles a tile;
  * ``gather_weight`` is the unshard (an all-gather on the caller's stream);
  * ``fsdp_fwd_bwd`` runs ``lce_fwd_bwd_sliced`` with the global count of
    valid labels, and for every vocabulary slice issues, on a communication
    stream that waits only for that slice's event, a reduce of the slice's
    rows to the rank that owns them. With the default slicing (one slice per
    owner) these are R reduces with different roots, i.e. a reduce-scatter
    cut into pieces that each start as soon as their rows are final.
"""
from __future__ import annotations

SLICE_ALIGN = 256  # dW tile height of the CUDA path (LCE_SLICE_ALIGN)


def owner_bounds(V: int, world: int, align: int = SLICE_ALIGN) -> list:
    """Row ranges [b_r, b_{r+1}) of the vocabulary owned by each rank: nearly
    equal numbers of ``align``-row blocks, the last range ending at V."""
    if world < 1:
        raise ValueError("world must be >= 1")
    blocks = (V + align - 1) // align
    b = [min(V, align * ((r * blocks) // world)) for r in range(world + 1)]
    b[-1] = V
    return b


def slice_pieces(slices: list, owners: list) -> list:
    """For each slice s: the (owner, row_begin, row_end) pieces that the
    slice's rows split into along the owners' ranges (empty pieces dropped)."""
    out = []
    for s in range(len(slices) - 1):
        a, b = slices[s], slices[s + 1]
        pieces = []
        for r in range(len(owners) - 1):
            lo, hi = max(a, owners[r]), min(b, owners[r + 1])
            if lo < hi:
                pieces.append((r, lo, hi))
        out.append(pieces)
    return out


def gather_weight(W_shard, owners: list, group=None):
    """All-gather of the vocabulary shards of W into the full [V, d] matrix,
    on the current stream. Shards may differ in size (padded to the largest)."""
    import torch
    import torch.distributed as dist
    world = dist.get_world_size(group)
    rows = [owners[r + 1] - owners[r] for r in range(world)]
    width = max(rows)
    pad = W_shard.new_zeros((width,) + tuple(W_shard.shape[1:]))
    pad[: W_shard.shape[0]] = W_shard
    out = W_shard.new_empty((world * width,) + tuple(W_shard.shape[1:]))
    dist.all_gather_into_tensor(out, pad.contiguous(), group=group)
    return torch.cat([out[r * width: r * width + rows[r]] for r in range(world)])


def _global_rank(group, r: int) -> int:
    import torch.distributed as dist
    return r if group is None else dist.get_global_rank(group, r)


def fsdp_fwd_bwd(H, W, y, grad_loss=None, *, owners: list, slices: list | None = None, group=None,
                 backend=None, comm_stream=None, sm_limit: int = 0, ignore_index: int = -100, **opt_kw):
    """One rank's step: fused forward + backward on its tokens with the full W
    (already gathered) and the global denominator; dW reduced to its owners.

    Returns (loss, lse, dH, dW_own): loss summed over ranks (the global mean),
    lse and dH of this rank's tokens, dW_own = rows [owners[rank],
    owners[rank+1]) of the global dW. ``slices`` defaults to ``owners``.

    ``backend`` computes the local step: ``backend(H, W, y, grad_loss, bounds,
    n_valid_override, **opt_kw) -> (loss, lse, dH, dW, events)`` where
    ``events[s]`` (or None) marks slice s final on the compute stream. By
    default it is the CUDA entry point ``lce.lce_fwd_bwd_sliced``; the reduces
    then run on ``comm_stream`` (a new side stream if None), each waiting only
    for its slice's event, and the caller's stream waits for all of them
    before this function returns.
    """
    import torch
    import torch.distributed as dist
    from . import dp
    world = dist.get_world_size(group)
    rank = dist.get_rank(group)
    if len(owners) != world + 1 or owners[0] != 0 or owners[-1] != W.shape[0]:
        raise ValueError("owners must hold world + 1 bounds from 0 to V")
    slices = owners if slices is None else slices
    n_global = dp.global_valid_count(y, ignore_index, group, V=W.shape[0])
    cuda = backend is None
    if cuda:
        from . import lce

        def backend(H, W, y, grad_loss, bounds, n_valid_override, **kw):
            ev = [torch.cuda.Event() for _ in range(len(bounds) - 1)]
            out = lce.lce_fwd_bwd_sliced(H, W, y, grad_loss, bounds=bounds, events=ev, sm_limit=sm_limit,
                                         n_valid_override=n_valid_override, **kw)
            return out + (ev,)
    loss, lse, dH, dW, events = backend(H, W, y, grad_loss, slices, n_global, ignore_index=ignore_index, **opt_kw)
    pieces = slice_pieces(slices, owners)
    works = []
    if cuda:
        main = torch.cuda.current_stream(H.device)
        comm = comm_stream if comm_stream is not None else torch.cuda.Stream(H.device)
        with torch.cuda.stream(comm):
            for s, ps in enumerate(pieces):
                comm.wait_event(events[s])
                for r, a, b in ps:
                    works.append(dist.reduce(dW[a:b], dst=_global_rank(group, r), group=group, async_op=True))
        for w in works:
            w.wait()          # orders the caller's stream after the reduces
        main.wait_stream(comm)
    else:
        for ps in pieces:
            for r, a, b in ps:
                works.append(dist.reduce(dW[a:b], dst=_global_rank(group, r), group=group, async_op=True))
        for w in works:
            w.wait()
    dist.all_reduce(loss, group=group)
    return loss, lse, dH, dW[owners[rank]:owners[rank + 1]]
