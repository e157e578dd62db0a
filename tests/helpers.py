"""Shared test plumbing: moving generated inputs to the GPU, running the oracle on
them, and the tolerances of the parity bar."""

from __future__ import annotations

import numpy as np
import torch

from gen import bf16_bits_to_f32

# Parity bar: fp32 inputs -> loss rel 1e-5, gradients max|diff| / max|ref| <= 1e-4;
# bf16 inputs -> loss rel 2e-3, gradients within 1e-2 * max|ref|.  lse and per-row
# losses use the loss tolerances, scaled to each row.
TOL = {"f32": dict(loss=1e-5, grad=1e-4), "bf16": dict(loss=2e-3, grad=1e-2)}


def host_f64(x):
    """Generated H / W (bf16 bit patterns or float32) as exact float64."""
    return bf16_bits_to_f32(x).astype(np.float64) if x.dtype == np.uint16 else x.astype(np.float64)


def to_device(x: dict, device="cuda"):
    def dense(a):
        if a.dtype == np.uint16:
            return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(device)
        return torch.from_numpy(np.ascontiguousarray(a)).to(device)

    out = dict(H=dense(x["H"]), topk_idx=torch.from_numpy(x["topk_idx"]).to(device),
               topk_logits=torch.from_numpy(x["topk_logits"]).to(device),
               valid=torch.from_numpy(np.ascontiguousarray(x["valid"])).to(device))
    if "W" in x:
        out["W"] = dense(x["W"])
    return out


def oracle_of(x, **kw):
    from oracle import fwd_bwd

    return fwd_bwd(host_f64(x["H"]), host_f64(x["W"]), x["topk_idx"], x["topk_logits"], x["valid"],
                   x["cfg"].tau, **kw)


def rel_max(got, ref):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    den = np.abs(ref).max(initial=0.0)
    err = np.abs(got - ref).max(initial=0.0)
    return err / den if den > 0 else err


def rel(a, b):
    return abs(a - b) / max(abs(b), 1e-30)
