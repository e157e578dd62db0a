"""fp64 CPU oracle for the fused chunked KL distillation loss.

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import or run this module.  It
shares no code with the CUDA library and never calls it.

What it computes
----------------
The pages describe the method but print no formula:

* the teacher is kept only as its top-K (id, logit) pairs per position,
  cached offline (axbrief.com, "Breaking the Bottleneck with Offline Caching
  and Chunked Loss"; calcaas.com, "What actually changed?": top-100);
* the loss is the KL divergence between teacher and student distributions
  (getaibook.com, "Configuring Fused Chunked KL Loss");
* the student's output projection is folded into the loss, so the loss is
  a function of the hidden states H and the lm_head weight W
  (calcaas.com, "What actually changed?").

The plain definition used here, on every row t with the tempered logits
s_t = (H_t . W^T) / tau over the full vocabulary:

    teacher   log p_tk = a_tk - logsumexp_k(a_t),  a_tk = topk_logits_tk / tau
              (p is zero outside the K cached ids)
    student   lse_t    = logsumexp_v(s_tv),   log q_tv = s_tv - lse_t
    loss_t    = sum_k p_tk (log p_tk - log q_t,idx_tk)          (forward KL)
    loss      = sum over valid rows of loss_t / N,   N = number of valid rows
    dz_tv     = g (q_tv - sum_k p_tk [idx_tk = v]) / (tau N)    (valid rows; 0 else)
    dH        = dz . W,     dW = dz^T . H

N = 0 gives loss 0 and zero gradients.  Duplicate ids in a row add up
termwise.  A cached logit of -inf is an entry the cache does not hold: its p is
0 and its KL term is 0 (the divergence sums over the support of p, the usual
0 log 0 = 0), so it is the same as leaving the entry out; every valid row needs
at least one finite logit.  Ignored rows contribute nothing whatever their
teacher logits hold.  Everything is fp64; the full logit row of every row is built
(row blocks only bound host memory), and the gradients are the analytic
ones above.
"""

from __future__ import annotations

import numpy as np

__all__ = ["teacher_log_probs", "student_lse", "fwd_bwd"]


def teacher_log_probs(topk_logits, tau):
    """log p over the K cached ids of each row: log-softmax of topk_logits / tau."""
    a = np.asarray(topk_logits, dtype=np.float64) / float(tau)
    amax = a.max(axis=1, keepdims=True)
    lse_a = amax + np.log(np.exp(a - amax).sum(axis=1, keepdims=True))
    return a - lse_a


def student_lse(s):
    """Row-wise logsumexp of the tempered student logits s[n, V]."""
    m = s.max(axis=1, keepdims=True)
    return (m + np.log(np.exp(s - m).sum(axis=1, keepdims=True)))[:, 0]


def fwd_bwd(H, W, topk_idx, topk_logits, valid, tau, grad=1.0, N=None, want_grads=True,
            dW_rows=None, row_block=64, return_dz=False):
    """Loss, per-row logsumexp, per-row loss and the gradients dH, dW.

    H[T, d], W[V, d]: float arrays (upcast to fp64).  topk_idx[T, K] ints in
    [0, V), topk_logits[T, K] floats, valid[T] (nonzero = the row counts).
    N: the number of valid rows the mean divides by; defaults to valid.sum()
    (pass the global count when H is a subset of a larger batch).
    dW_rows: vocab rows of dW to return (all when None).
    Returns a dict with loss, lse[T], row_loss[T], N and, when want_grads,
    dH[T, d] and dW[len(dW_rows) or V, d] (and dz[T, V] if return_dz).
    """
    H = np.asarray(H, dtype=np.float64)
    W = np.asarray(W, dtype=np.float64)
    idx = np.asarray(topk_idx, dtype=np.int64)
    valid = np.asarray(valid).astype(bool)
    T, d = H.shape
    V = W.shape[0]
    if idx.size and (idx.min() < 0 or idx.max() >= V):
        raise ValueError("teacher id out of range")
    if N is None:
        N = int(valid.sum())
    tau = float(tau)
    logp = teacher_log_probs(topk_logits, tau) if T else np.zeros((0, idx.shape[1]))
    p = np.exp(logp)

    lse = np.zeros(T)
    row_loss = np.zeros(T)
    dH = np.zeros((T, d)) if want_grads else None
    Wsel = W if dW_rows is None else W[np.asarray(dW_rows, dtype=np.int64)]
    dW = np.zeros((Wsel.shape[0], d)) if want_grads else None
    dz_all = np.zeros((T, V)) if return_dz else None
    scale = float(grad) / (tau * N) if N > 0 else 0.0

    for b0 in range(0, T, row_block):
        b1 = min(T, b0 + row_block)
        s = (H[b0:b1] @ W.T) / tau  # full tempered logit rows
        lse_b = student_lse(s)
        lse[b0:b1] = lse_b
        rows = np.arange(b1 - b0)[:, None]
        log_q_at = s[rows, idx[b0:b1]] - lse_b[:, None]
        pb = p[b0:b1]
        with np.errstate(invalid="ignore"):
            terms = pb * (logp[b0:b1] - log_q_at)
        rl = np.where(pb > 0, terms, 0.0).sum(axis=1)  # terms outside the support of p are 0
        row_loss[b0:b1] = np.where(valid[b0:b1], rl, 0.0)
        if not want_grads:
            continue
        q = np.exp(s - lse_b[:, None])
        dz = q
        np.add.at(dz, (np.repeat(np.arange(b1 - b0), idx.shape[1]), idx[b0:b1].ravel()),
                  -p[b0:b1].ravel())
        dz *= scale
        dz[~valid[b0:b1]] = 0.0
        if return_dz:
            dz_all[b0:b1] = dz
        dH[b0:b1] = dz @ W
        dzs = dz if dW_rows is None else dz[:, np.asarray(dW_rows, dtype=np.int64)]
        dW += dzs.T @ H[b0:b1]

    loss = float(row_loss.sum() / N) if N > 0 else 0.0
    out = dict(loss=loss, lse=lse, row_loss=row_loss, N=N)
    if want_grads:
        out["dH"] = dH
        out["dW"] = dW
    if return_dz:
        out["dz"] = dz_all
    return out
