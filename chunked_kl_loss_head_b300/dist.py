"""Token-sharded data parallelism of the fused chunked KL loss over a process group.

The pages place the method in distillation runs that are otherwise spread over many
GPUs and nodes (getaibook.com, "Hardware and Performance Tradeoffs"; axbrief.com,
"Quantifying the Efficiency Gain: 15.6x VRAM Reduction").  The loss shards over
tokens: each rank holds its own rows of the student's hidden states H, of the teacher
cache (topk_idx, topk_logits) and of the valid mask, and the whole lm_head weight W.
Everything per row stays on its rank; three things cross ranks:

* before the backward, the loss sum and the valid-row count N (fp64 [2]): the mean
  divides by the N of all ranks, and so does the gradient scale g / (tau N);
* after the backward, dW (fp32 [V, d]), which sums over ranks.

dH stays with its rank.  The per-rank work runs in libfckl.so (fckl_forward,
fckl_backward, and fckl_loss_partials / fckl_loss_finish around the partials'
sum); this module only orders those calls and the collectives, which are
torch.distributed all-reduces (NCCL between GPUs).

``ShardedKL`` exposes the phases (``forward_local`` -> sum the partials over ranks ->
``finish`` -> ``backward_local`` -> sum dW over ranks) and composes them over a
process group in ``forward`` / ``backward``.
"""

from __future__ import annotations

import torch

from . import api


def _all_reduce_sum(group):
    import torch.distributed as dist

    def reduce(t):
        dist.all_reduce(t, op=dist.ReduceOp.SUM, group=group)

    return reduce


class LibraryOps:
    """The per-rank steps, all in libfckl.so: the forward with its partials, the finish
    of the partials summed over ranks, and the backward scaled to the total N."""

    def __init__(self, tau, chunk):
        self.tau = float(tau)
        self.chunk = int(chunk)
        self.ws = None
        self._ws_key = None

    def _workspace(self, H, W, topk_idx):
        T, d = H.shape
        key = (T, d, W.shape[0], topk_idx.shape[1], self.chunk, H.dtype, H.device)
        if key != self._ws_key:
            self.ws = api.workspace(T, d, W.shape[0], topk_idx.shape[1], self.chunk, H.dtype, H.device)
            self._ws_key = key
        return self.ws

    def forward_local(self, H, W, topk_idx, topk_logits, valid):
        """(lse [T], partials float64 [2] = (loss sum, N) of this rank's rows)."""
        ws = self._workspace(H, W, topk_idx)
        _, lse = api.forward(H, W, topk_idx, topk_logits, valid, self.tau, self.chunk, ws=ws)
        partials = torch.empty(2, dtype=torch.float64, device=H.device)
        api.fckl_loss_partials(ws, partials)
        return lse, partials

    def finish(self, total, local):
        """(loss = total sum / total N, grad_scale = local N / total N), float32 scalars."""
        loss = torch.empty((), dtype=torch.float32, device=total.device)
        scale = torch.empty((), dtype=torch.float32, device=total.device)
        api.fckl_loss_finish(total, local, loss, scale)
        return loss, scale

    def backward_local(self, H, W, topk_idx, topk_logits, valid, lse, grad_loss, grad_scale):
        """(dH [T, d] in H's dtype, dW [V, d] float32) of this rank's rows, scaled by
        grad_loss * grad_scale / (tau N_local)."""
        ws = self._workspace(H, W, topk_idx)
        return api.backward(H, W, topk_idx, topk_logits, valid, lse, self.tau, self.chunk, grad_loss=grad_loss,
                            ws=ws, grad_scale=grad_scale)


class ShardedKL:
    """One rank's share of the loss over a token-sharded batch.

    reduce: a callable summing a tensor over ranks in place; by default an all-reduce
    (sum) over `group` (None: the default process group).  reduce_dW: sum dW over ranks
    (turn it off when something else, e.g. a data-parallel wrapper of the model, already
    reduces the lm_head's gradient).  ops: the per-rank steps (LibraryOps by default).
    """

    def __init__(self, tau=1.0, chunk=4096, group=None, reduce=None, reduce_dW=True, ops=None):
        self.ops = ops if ops is not None else LibraryOps(tau, chunk)
        self.reduce = reduce if reduce is not None else _all_reduce_sum(group)
        self.reduce_dW = reduce_dW
        self._saved = None

    # ---- phases
    def forward_local(self, H, W, topk_idx, topk_logits, valid):
        """This rank's forward; returns its partials (loss sum, N) for the sum over ranks."""
        lse, local = self.ops.forward_local(H, W, topk_idx, topk_logits, valid)
        self._saved = dict(H=H, W=W, topk_idx=topk_idx, topk_logits=topk_logits, valid=valid, lse=lse, local=local)
        return local

    def state(self):
        """What the backward of the last forward needs (its inputs, lse and scales), to be
        handed back with restore() when another forward has run through this object since."""
        return dict(self._state())

    def restore(self, state):
        self._saved = dict(state)

    def _state(self, need_scale=False):
        if self._saved is None or (need_scale and "grad_scale" not in self._saved):
            raise RuntimeError("ShardedKL: run forward_local and finish (or forward) before this step")
        return self._saved

    def finish(self, total):
        """From the partials summed over ranks: the mean loss over every rank's valid rows."""
        loss, scale = self.ops.finish(total, self._state()["local"])
        self._saved["grad_scale"] = scale
        return loss

    def backward_local(self, grad_loss=1.0, grad_scale=None):
        """(dH, dW) of this rank's rows for the loss over all ranks; dW before the sum over
        ranks.  grad_scale (device float32 scalar, optional) multiplies grad_loss."""
        s = self._state(need_scale=True)
        scale = s["grad_scale"] if grad_scale is None else grad_scale * s["grad_scale"]
        return self.ops.backward_local(s["H"], s["W"], s["topk_idx"], s["topk_logits"], s["valid"], s["lse"],
                                       grad_loss, scale)

    # ---- composed over the process group
    def forward(self, H, W, topk_idx, topk_logits, valid):
        """The mean loss over every rank's valid rows (the same value on every rank)."""
        local = self.forward_local(H, W, topk_idx, topk_logits, valid)
        total = local.clone()
        self.reduce(total)
        return self.finish(total)

    def backward(self, grad_loss=1.0, grad_scale=None):
        """(dH of this rank's rows, dW summed over ranks when reduce_dW)."""
        dH, dW = self.backward_local(grad_loss, grad_scale)
        if self.reduce_dW:
            self.reduce(dW)
        return dH, dW


class _ShardedFn(torch.autograd.Function):
    @staticmethod
    def forward(ctx, H, W, topk_idx, topk_logits, valid, sharded):
        ctx.sharded = sharded
        ctx.w_dtype = W.dtype
        loss = sharded.forward(H, W, topk_idx, topk_logits, valid)
        # this call's own state: another forward through the same object (a second
        # micro-batch) may come before this call's backward
        ctx.state = sharded.state()
        return loss

    @staticmethod
    def backward(ctx, grad):
        g = grad.detach().to(torch.float32).reshape(())
        ctx.sharded.restore(ctx.state)
        dH, dW = ctx.sharded.backward(1.0, g)
        # dW is summed over ranks in float32; the gradient takes W's dtype
        return dH, api.to_dtype(dW, ctx.w_dtype), None, None, None, None


class ShardedFusedChunkedKLLoss(torch.nn.Module):
    """FusedChunkedKLLoss over a token-sharded batch: each rank passes its own rows and the
    whole lm_head weight; the loss is the mean over every rank's valid rows, dH is this
    rank's, and dW is summed over ranks (unless reduce_dW is off)."""

    def __init__(self, tau=1.0, chunk=4096, group=None, reduce_dW=True, reduce=None):
        super().__init__()
        self.sharded = ShardedKL(tau, chunk, group=group, reduce=reduce, reduce_dW=reduce_dW)

    def forward(self, hidden, lm_head_weight, topk_idx, topk_logits, valid=None):
        if valid is None:
            valid = torch.ones(hidden.shape[0], dtype=torch.uint8, device=hidden.device)
        return _ShardedFn.apply(hidden.contiguous(), lm_head_weight.contiguous(),
                                topk_idx.to(torch.int32).contiguous(), topk_logits.to(torch.float32).contiguous(),
                                valid.to(torch.uint8).contiguous(), self.sharded)
