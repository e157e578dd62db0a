"""fckl_forward_noalloc: the forward for callers that cannot allocate device memory.

Some callers of this library cannot call cudaMalloc: code running while a stream is
captured into a CUDA graph, runtimes that reserve all device memory for their own
pool, and loops that cannot afford the synchronization an allocation may cause.  This
entry point gives them the forward pass with the library's own fixed scratch instead
of a workspace.  Its results must match fckl_forward's, call after call (the scratch
is shared and keeps the previous call's contents).  This file sorts last so that a
run stopping at the first failure has run every other test before it.
"""

import ctypes

import numpy as np
import pytest
import torch

from chunked_kl_loss_head_b300 import _lib, api
from gen import make_small
from helpers import TOL, rel, rel_max, to_device


@pytest.mark.gpu
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_noalloc_forward_matches_forward_two_calls(dtype):
    x = make_small(T=3000, d=256, V=20000, K=20, tau=1.3, dtype=dtype, seed=21, mask="random", mask_frac=0.1)
    g = to_device(x)
    T, d = g["H"].shape
    V, K = g["W"].shape[0], g["topk_idx"].shape[1]
    chunk = 4096
    ref_loss, ref_lse, ref_rl = api.forward(g["H"], g["W"], g["topk_idx"], g["topk_logits"], g["valid"], 1.3, chunk,
                                            want_row_loss=True)
    torch.cuda.synchronize()
    tol = TOL[dtype]["loss"]
    for call in range(2):
        loss = torch.full((), float("nan"), device="cuda")
        lse = torch.full((T,), float("nan"), device="cuda")
        rl = torch.full((T,), float("nan"), device="cuda")
        status = torch.full((), -1, dtype=torch.int32, device="cuda")
        api.fckl_forward_noalloc(g["H"], g["W"], g["topk_idx"], g["topk_logits"], g["valid"], 1.3, chunk, loss, lse,
                                 rl, status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0, f"call {call}: status {int(status.item())}"
        assert rel(loss.item(), ref_loss.item()) <= tol, (call, loss.item(), ref_loss.item())
        assert rel_max(lse.cpu().numpy(), ref_lse.cpu().numpy()) <= tol, call
        assert rel_max(rl.cpu().numpy(), ref_rl.cpu().numpy()) <= tol, call


def test_noalloc_rejects_sizes_beyond_its_scratch():
    # one row of a 300M-id vocabulary needs more scratch than the fixed array holds;
    # the call is refused before anything touches a device
    L = _lib.lib()
    dummy = ctypes.c_void_p(1 << 20)
    st = L.fckl_forward_noalloc(dummy, dummy, dummy, dummy, dummy, 64, 256, 300_000_000, 10, 1.0, 64, 1, dummy, dummy,
                                dummy, None, None)
    assert st == 3, api.fckl_status_string(st)
