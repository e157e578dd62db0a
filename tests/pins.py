"""Pins of the fp64 oracle against facts fixed by the mathematics, not by the
oracle itself.  Each pin takes a ``fwd_bwd`` callable with the oracle's
signature and raises AssertionError when the callable disagrees with the
fact it checks, so the same pins run on the oracle and on deliberately
broken copies of it (tests/test_oracle_pins.py).

The pages print no worked example and no formula for the loss; what is
pinned here is the definition written in the oracle's header (forward KL of
the tempered top-K teacher softmax against the tempered full-vocabulary
student softmax, mean over valid rows), through:

* central finite differences of the loss against the analytic gradients;
* library routines on special cases (torch's kl_div on the dense teacher,
  torch's cross_entropy when K = 1, torch's logsumexp for lse);
* Gibbs' inequality (KL >= 0) and KL = 0 when teacher = student;
* rows of the logit gradient summing to zero;
* the closed form at W = 0 (uniform student);
* the temperature identity, shift / permutation invariance of the teacher,
  additivity over row subsets and the ignored-row contract;
* entries of logit -inf being the same as entries left out (KL sums over the
  support of p).
"""

from __future__ import annotations

import numpy as np
import torch
import torch.nn.functional as F


def _tiny(seed=0, T=3, d=5, V=11, K=4, ignored=(1,), scale_w=1.0, scale_h=1.0):
    rng = np.random.default_rng(seed)
    H = rng.standard_normal((T, d)) * scale_h
    W = rng.standard_normal((V, d)) * scale_w
    idx = np.stack([rng.choice(V, K, replace=False) for _ in range(T)])
    lg = rng.standard_normal((T, K)) * 2.0 + 3.0
    valid = np.ones(T, np.uint8)
    for r in ignored:
        if r < T:
            valid[r] = 0
    return H, W, idx, lg, valid


def _rel(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    den = max(np.abs(b).max(initial=0.0), 1e-300)
    return np.abs(a - b).max(initial=0.0) / den


# ------------------------------------------------------------------------------------------


def pin_finite_differences(f):
    """Analytic dH, dW equal central differences of g*loss (fp64, rel <= 1e-7)."""
    for tau, g in ((1.0, 1.0), (2.0, 1.7)):
        H, W, idx, lg, valid = _tiny(seed=3)
        out = f(H=H, W=W, topk_idx=idx, topk_logits=lg, valid=valid, tau=tau, grad=g)
        h = 1e-6

        def L(H_, W_):
            return g * f(H=H_, W=W_, topk_idx=idx, topk_logits=lg, valid=valid, tau=tau,
                         grad=g, want_grads=False)["loss"]

        fdH = np.zeros_like(H)
        for i in np.ndindex(H.shape):
            Hp, Hm = H.copy(), H.copy()
            Hp[i] += h
            Hm[i] -= h
            fdH[i] = (L(Hp, W) - L(Hm, W)) / (2 * h)
        fdW = np.zeros_like(W)
        for i in np.ndindex(W.shape):
            Wp, Wm = W.copy(), W.copy()
            Wp[i] += h
            Wm[i] -= h
            fdW[i] = (L(H, Wp) - L(H, Wm)) / (2 * h)
        assert _rel(out["dH"], fdH) <= 1e-7, ("dH vs finite differences", tau, _rel(out["dH"], fdH))
        assert _rel(out["dW"], fdW) <= 1e-7, ("dW vs finite differences", tau, _rel(out["dW"], fdW))


def pin_library_kl(f):
    """loss = torch kl_div(log_softmax(Z/tau), dense p) summed over valid rows / N."""
    for tau in (1.0, 2.0, 0.7):
        H, W, idx, lg, valid = _tiny(seed=5, T=6, d=7, V=19, K=5, ignored=(2, 4))
        out = f(H=H, W=W, topk_idx=idx, topk_logits=lg, valid=valid, tau=tau, want_grads=False)
        Z = torch.from_numpy(H) @ torch.from_numpy(W).T
        log_q = F.log_softmax(Z / tau, dim=1)
        p_k = torch.softmax(torch.from_numpy(lg) / tau, dim=1)
        P = torch.zeros_like(Z).scatter_add_(1, torch.from_numpy(idx).long(), p_k)
        per_row = F.kl_div(log_q, P, reduction="none").sum(dim=1).numpy()
        m = valid.astype(bool)
        ref = per_row[m].sum() / m.sum()
        assert abs(out["loss"] - ref) <= 1e-12 * max(1.0, abs(ref)), ("kl_div", tau, out["loss"], ref)
        lse_ref = torch.logsumexp(Z / tau, dim=1).numpy()
        assert _rel(out["lse"], lse_ref) <= 1e-13, ("lse vs torch.logsumexp", tau)
        assert _rel(out["row_loss"][m], per_row[m]) <= 1e-12, "per-row loss vs kl_div"
        assert np.all(out["row_loss"][~m] == 0.0), "ignored rows carry loss"


def pin_cross_entropy_k1(f):
    """With K = 1 the teacher is one-hot: loss = textbook cross-entropy of Z/tau."""
    for tau in (1.0, 3.0):
        H, W, idx, lg, valid = _tiny(seed=7, T=8, d=6, V=13, K=1, ignored=(0, 5))
        out = f(H=H, W=W, topk_idx=idx, topk_logits=lg, valid=valid, tau=tau, want_grads=False)
        Z = torch.from_numpy(H) @ torch.from_numpy(W).T
        m = torch.from_numpy(valid.astype(bool))
        ref = F.cross_entropy((Z / tau)[m], torch.from_numpy(idx[:, 0]).long()[m]).item()
        assert abs(out["loss"] - ref) <= 1e-12 * max(1.0, abs(ref)), ("cross_entropy", out["loss"], ref)


def pin_kl_nonneg(f):
    """Gibbs' inequality: every valid row's KL is >= 0."""
    for seed in range(4):
        H, W, idx, lg, valid = _tiny(seed=seed, T=16, d=8, V=40, K=6, ignored=(3,), scale_w=2.0)
        out = f(H=H, W=W, topk_idx=idx, topk_logits=lg, valid=valid, tau=1.3, want_grads=False)
        assert np.all(out["row_loss"] >= -1e-12), "negative KL"
        assert out["loss"] > 0.0


def pin_kl_zero(f):
    """K = V, teacher logits = student logits: loss = 0 and gradients = 0."""
    for tau in (1.0, 2.5):
        rng = np.random.default_rng(11)
        T, d, V = 4, 6, 9
        H = rng.standard_normal((T, d))
        W = rng.standard_normal((V, d))
        Z = H @ W.T
        idx = np.stack([rng.permutation(V) for _ in range(T)])
        lg = np.take_along_axis(Z, idx, axis=1)
        valid = np.ones(T, np.uint8)
        out = f(H=H, W=W, topk_idx=idx, topk_logits=lg, valid=valid, tau=tau)
        assert abs(out["loss"]) <= 1e-12, ("KL(p||p) != 0", out["loss"])
        assert np.abs(out["dH"]).max() <= 1e-12 and np.abs(out["dW"]).max() <= 1e-12


def pin_dz_rows_sum_zero(f):
    """sum_v dz_tv = 0 on every row (q and p both sum to one); dz = 0 on ignored rows."""
    H, W, idx, lg, valid = _tiny(seed=13, T=5, d=4, V=17, K=3, ignored=(4,))
    out = f(H=H, W=W, topk_idx=idx, topk_logits=lg, valid=valid, tau=1.5, return_dz=True)
    dz = out["dz"]
    assert np.abs(dz.sum(axis=1)).max() <= 1e-15, "logit-gradient rows do not sum to 0"
    assert np.all(dz[4] == 0.0)
    assert np.abs(dz[:4]).max() > 1e-3


def pin_closed_form_uniform_student(f):
    """W = 0: q uniform, loss_t = sum p log p + log V, dH = 0,
    dW_v = g * sum_t (1/V - p_tv) H_t / (tau N)."""
    tau, g = 2.0, 0.6
    H, W, idx, lg, valid = _tiny(seed=17, T=5, d=3, V=7, K=3, ignored=(2,))
    W[:] = 0.0
    out = f(H=H, W=W, topk_idx=idx, topk_logits=lg, valid=valid, tau=tau, grad=g)
    e = np.exp(lg / tau)
    p = e / e.sum(axis=1, keepdims=True)
    V = W.shape[0]
    m = valid.astype(bool)
    rl = (p * np.log(p)).sum(axis=1) + np.log(V)
    assert abs(out["loss"] - rl[m].mean()) <= 1e-13 * abs(rl[m].mean())
    assert np.abs(out["dH"]).max() == 0.0
    Pd = np.zeros((H.shape[0], V))
    for t in range(H.shape[0]):
        for k in range(idx.shape[1]):
            Pd[t, idx[t, k]] += p[t, k]
    dW = np.zeros((V, H.shape[1]))
    for t in np.nonzero(m)[0]:
        for v in range(V):
            dW[v] += (1.0 / V - Pd[t, v]) * H[t]
    dW *= g / (tau * m.sum())
    assert _rel(out["dW"], dW) <= 1e-13, "dW closed form at W=0"


def pin_tau_identity(f):
    """loss(H, W, tau, L) = loss(H/tau, W, 1, L/tau); dH scales by 1/tau, dW is unchanged."""
    tau = 2.7
    H, W, idx, lg, valid = _tiny(seed=19, T=6, d=5, V=12, K=4, ignored=(1,))
    a = f(H=H, W=W, topk_idx=idx, topk_logits=lg, valid=valid, tau=tau)
    b = f(H=H / tau, W=W, topk_idx=idx, topk_logits=lg / tau, valid=valid, tau=1.0)
    assert abs(a["loss"] - b["loss"]) <= 1e-13 * abs(b["loss"])
    assert _rel(a["dH"], b["dH"] / tau) <= 1e-12
    assert _rel(a["dW"], b["dW"]) <= 1e-12
    assert _rel(a["lse"], b["lse"]) <= 1e-13


def pin_shift_and_permutation(f):
    """A per-row constant added to the teacher logits, or a permutation of the
    K (id, logit) pairs of a row, changes nothing."""
    H, W, idx, lg, valid = _tiny(seed=23, T=5, d=6, V=15, K=5, ignored=(0,))
    a = f(H=H, W=W, topk_idx=idx, topk_logits=lg, valid=valid, tau=1.2)
    shift = np.arange(5)[:, None] * 3.5 - 4.0
    b = f(H=H, W=W, topk_idx=idx, topk_logits=lg + shift, valid=valid, tau=1.2)
    rng = np.random.default_rng(1)
    perm = np.stack([rng.permutation(5) for _ in range(5)])
    c = f(H=H, W=W, topk_idx=np.take_along_axis(idx, perm, 1),
          topk_logits=np.take_along_axis(lg, perm, 1), valid=valid, tau=1.2)
    for o in (b, c):
        assert abs(o["loss"] - a["loss"]) <= 1e-13 * abs(a["loss"])
        assert _rel(o["dH"], a["dH"]) <= 1e-12 and _rel(o["dW"], a["dW"]) <= 1e-12


def pin_additivity(f):
    """Rows are independent: dW and the loss sum over row subsets (global N);
    dH rows of a subset equal the corresponding rows of the whole."""
    H, W, idx, lg, valid = _tiny(seed=29, T=9, d=4, V=10, K=3, ignored=(2, 7))
    whole = f(H=H, W=W, topk_idx=idx, topk_logits=lg, valid=valid, tau=1.1, grad=1.3)
    N = int(valid.sum())
    dW = np.zeros_like(whole["dW"])
    tot = 0.0
    for sl in (slice(0, 4), slice(4, 5), slice(5, 9)):
        part = f(H=H[sl], W=W, topk_idx=idx[sl], topk_logits=lg[sl], valid=valid[sl], tau=1.1,
                 grad=1.3, N=N)
        dW += part["dW"]
        tot += part["row_loss"].sum()
        assert _rel(part["dH"], whole["dH"][sl]) <= 1e-13
    assert _rel(dW, whole["dW"]) <= 1e-13
    assert abs(tot / N - whole["loss"]) <= 1e-13 * abs(whole["loss"])


def pin_ignored_rows(f):
    """Ignored rows: dH rows exactly 0, and changing their data changes nothing."""
    H, W, idx, lg, valid = _tiny(seed=31, T=6, d=5, V=14, K=4, ignored=(1, 4))
    a = f(H=H, W=W, topk_idx=idx, topk_logits=lg, valid=valid, tau=1.0)
    assert np.all(a["dH"][[1, 4]] == 0.0)
    H2, idx2, lg2 = H.copy(), idx.copy(), lg.copy()
    H2[[1, 4]] *= -3.0
    idx2[[1, 4]] = idx2[[1, 4]][:, ::-1]
    lg2[[1, 4]] += 5.0 * np.arange(4)
    b = f(H=H2, W=W, topk_idx=idx2, topk_logits=lg2, valid=valid, tau=1.0)
    assert b["loss"] == a["loss"]
    assert _rel(b["dW"], a["dW"]) <= 1e-15
    assert np.array_equal(b["dH"][[0, 2, 3, 5]], a["dH"][[0, 2, 3, 5]])


def pin_absent_entries(f):
    """A cached logit of -inf is an entry the cache does not hold: appending (id, -inf)
    pairs to every row (ids already in the row or not) changes nothing, since the KL
    divergence sums over the support of p (0 log 0 = 0)."""
    H, W, idx, lg, valid = _tiny(seed=53, T=6, d=5, V=16, K=4, ignored=(2,))
    a = f(H=H, W=W, topk_idx=idx, topk_logits=lg, valid=valid, tau=1.3, grad=0.8)
    extra_idx = np.stack([np.array([(t * 5 + 3) % 16, idx[t, 0]]) for t in range(6)])
    idx2 = np.concatenate([idx, extra_idx], axis=1)
    lg2 = np.concatenate([lg, np.full((6, 2), -np.inf)], axis=1)
    b = f(H=H, W=W, topk_idx=idx2, topk_logits=lg2, valid=valid, tau=1.3, grad=0.8)
    assert np.isfinite(b["loss"]) and abs(b["loss"] - a["loss"]) <= 1e-13 * abs(a["loss"]), "-inf entries"
    assert _rel(b["row_loss"], a["row_loss"]) <= 1e-13
    assert _rel(b["dH"], a["dH"]) <= 1e-13 and _rel(b["dW"], a["dW"]) <= 1e-13


def pin_ignored_rows_hold_anything(f):
    """An ignored row's teacher logits are never used: NaN or infinite values there give
    the same loss and gradients as finite ones, and its dH row stays exactly 0."""
    H, W, idx, lg, valid = _tiny(seed=59, T=5, d=4, V=12, K=3, ignored=(0, 3))
    a = f(H=H, W=W, topk_idx=idx, topk_logits=lg, valid=valid, tau=0.9)
    lg2 = lg.copy()
    lg2[0] = np.nan
    lg2[3] = [np.inf, -np.inf, np.nan]
    b = f(H=H, W=W, topk_idx=idx, topk_logits=lg2, valid=valid, tau=0.9)
    assert b["loss"] == a["loss"], "ignored rows' teacher data reach the loss"
    assert np.array_equal(b["row_loss"], a["row_loss"])
    assert np.array_equal(b["dH"], a["dH"]) and np.array_equal(b["dW"], a["dW"])
    assert np.all(b["dH"][[0, 3]] == 0.0)


def pin_no_valid_rows(f):
    """N = 0: loss 0 and zero gradients (the reading that avoids 0/0)."""
    H, W, idx, lg, valid = _tiny(seed=37, T=3, d=4, V=8, K=2, ignored=(0, 1, 2))
    out = f(H=H, W=W, topk_idx=idx, topk_logits=lg, valid=valid, tau=1.0)
    assert out["loss"] == 0.0 and not out["dH"].any() and not out["dW"].any()


ALL_PINS = [
    pin_finite_differences,
    pin_library_kl,
    pin_cross_entropy_k1,
    pin_kl_nonneg,
    pin_kl_zero,
    pin_dz_rows_sum_zero,
    pin_closed_form_uniform_student,
    pin_tau_identity,
    pin_shift_and_permutation,
    pin_additivity,
    pin_ignored_rows,
    pin_absent_entries,
    pin_ignored_rows_hold_anything,
    pin_no_valid_rows,
]
