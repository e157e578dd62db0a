"""``FusedChunkedKLLoss``: the training-loop entry point over the C-ABI.

The pages tell the user to route the loss through a FusedChunkedKLLoss module
in place of a standard PyTorch loss (getaibook.com, "Configuring Fused Chunked
KL Loss").  This module takes the student's final hidden states and its
lm_head weight (the projection is folded into the loss) plus the cached
teacher top-K ids and logits; the forward saves only the per-row logsumexp,
and the backward recomputes the logit tiles chunk by chunk.
"""

from __future__ import annotations

import torch

from . import api


class _Workspace:
    """One workspace kept for the calls of one module instance (re-made when the sizes
    change).  The library carries nothing in it from a forward to its backward, so calls
    that share it only need to be ordered on one stream."""

    def __init__(self):
        self.key = None
        self.ws = None

    def get(self, T, d, V, K, chunk, dtype, device):
        key = (T, d, V, K, chunk, dtype, device)
        if key != self.key:
            self.ws = None
            self.ws = api.workspace(T, d, V, K, chunk, dtype, device)
            self.key = key
        return self.ws


class _FusedChunkedKL(torch.autograd.Function):
    @staticmethod
    def forward(ctx, H, W, topk_idx, topk_logits, valid, tau, chunk, holder):
        T, d = H.shape
        V = W.shape[0]
        K = topk_idx.shape[1]
        if holder is not None:
            ws = holder.get(T, d, V, K, chunk, H.dtype, H.device)
        else:
            ws = api.workspace(T, d, V, K, chunk, H.dtype, H.device)
        loss, lse = api.forward(H, W, topk_idx, topk_logits, valid, tau, chunk, ws=ws)
        ctx.save_for_backward(H, W, topk_idx, topk_logits, valid, lse)
        ctx.ws, ctx.tau, ctx.chunk = ws, tau, chunk
        return loss

    @staticmethod
    def backward(ctx, grad):
        H, W, topk_idx, topk_logits, valid, lse = ctx.saved_tensors
        g = grad.detach().to(torch.float32).contiguous()
        dH, dW = api.backward(H, W, topk_idx, topk_logits, valid, lse, ctx.tau, ctx.chunk, grad_loss=1.0,
                              ws=ctx.ws, grad_scale=g)
        # dW accumulates in float32 across chunks; the gradient takes W's dtype
        return dH, api.to_dtype(dW, W.dtype), None, None, None, None, None, None


def fused_chunked_kl_loss(hidden, lm_head_weight, topk_idx, topk_logits, valid=None, tau=1.0, chunk=4096,
                          _holder=None):
    """Mean forward KL(teacher top-K || student) over valid rows; differentiable in
    `hidden` [T, d] and `lm_head_weight` [V, d].  Each call makes its own workspace (the
    module keeps one instead)."""
    if valid is None:
        valid = torch.ones(hidden.shape[0], dtype=torch.uint8, device=hidden.device)
    return _FusedChunkedKL.apply(hidden.contiguous(), lm_head_weight.contiguous(),
                                 topk_idx.to(torch.int32).contiguous(),
                                 topk_logits.to(torch.float32).contiguous(), valid.to(torch.uint8).contiguous(),
                                 float(tau), int(chunk), _holder)


class FusedChunkedKLLoss(torch.nn.Module):
    """The loss as a module (getaibook.com, "Configuring Fused Chunked KL Loss"): call it
    with the student's final hidden states [T, d], its lm_head weight [V, d], the cached
    teacher ids and logits [T, K] and an optional valid mask [T].  One workspace (its size
    grows with `chunk`, never with T x V) is kept for the instance's calls, which must be
    ordered on one stream."""

    def __init__(self, tau: float = 1.0, chunk: int = 4096):
        super().__init__()
        self.tau = float(tau)
        self.chunk = int(chunk)
        self._ws = _Workspace()

    def forward(self, hidden, lm_head_weight, topk_idx, topk_logits, valid=None):
        return fused_chunked_kl_loss(hidden, lm_head_weight, topk_idx, topk_logits, valid, self.tau, self.chunk,
                                     _holder=self._ws)
