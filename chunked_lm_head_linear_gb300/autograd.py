"""PyTorch autograd wrapper of the fused LM-head linear + cross-entropy.

    loss_fn = FusedLinearCrossEntropy(ignore_index=-100)
    loss = loss_fn(H, W, y)      # H [N, d] bf16, W [V, d] bf16, y [N] int64, all on the GPU
    loss.backward()              # H.grad, W.grad (in W's dtype: autograd casts the fp32 dW to it)

The forward pass runs the whole fused forward + backward (lce_fwd_bwd with an
upstream gradient of 1) and keeps dH and dW; the backward pass scales them by
the actual upstream gradient with lce_scale_grads (a device-side no-op when it
is 1). This is the arrangement of the fused loss on "XTuner on Ascend 910C:
Qwen3.5-2B training optimisation" (section 3.1.4: one fused kernel produces
d_input and d_weight, no d_logits is kept), and it costs 6 N V d flops.
``recompute=True`` instead saves only lse in the forward and recomputes the
logits in the backward (lce_backward, 8 N V d flops) -- for when the
gradients should not be held between the passes.

The library's dW is fp32; autograd hands a leaf its gradient in the leaf's own
dtype, so a bf16 W receives bf16 gradients. Callers that keep fp32 weight
gradients (gradient accumulation over micro-batches, fp32 reduction across
ranks) call ``lce.lce_fwd_bwd`` with their fp32 buffer as ``dW`` and
``accumulate_dW=True`` instead.
"""
from __future__ import annotations

import torch

from . import lce


class _FusedLCE(torch.autograd.Function):
    @staticmethod
    def forward(ctx, H, W, y, opts):
        loss, _, dH, dW = lce.lce_fwd_bwd(H, W, y, **opts)
        ctx.save_for_backward(dH, dW)
        return loss.reshape(())

    @staticmethod
    def backward(ctx, g):
        dH, dW = ctx.saved_tensors
        g = g.reshape(1).to(torch.float32).contiguous()
        lce.lce_scale_grads(dH, dW, g)
        return dH, dW, None, None


class _RecomputeLCE(torch.autograd.Function):
    @staticmethod
    def forward(ctx, H, W, y, opts):
        loss, lse = lce.lce_forward(H, W, y, **opts)
        ctx.save_for_backward(H, W, y, lse)
        ctx.opts = opts
        return loss.reshape(())

    @staticmethod
    def backward(ctx, g):
        H, W, y, lse = ctx.saved_tensors
        g = g.reshape(1).to(torch.float32).contiguous()
        dH, dW = lce.lce_backward(H, W, y, lse, g, **ctx.opts)
        return dH, dW, None, None


class FusedLinearCrossEntropy(torch.nn.Module):
    """Token-level cross-entropy of the LM-head logits H W^T (mean over tokens
    whose label is not ignore_index), fused and chunked on the GPU."""

    def __init__(self, ignore_index: int = -100, reduction: str = "mean", chunk_tokens=0, recompute: bool = False):
        super().__init__()
        self.opts = dict(ignore_index=ignore_index, reduction=reduction, chunk_tokens=chunk_tokens)
        self.recompute = recompute

    def forward(self, H, W, y):
        fn = _RecomputeLCE if self.recompute else _FusedLCE
        return fn.apply(H, W, y, self.opts)
