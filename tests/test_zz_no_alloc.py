"""fckl_forward_noalloc: the forward for callers that cannot allocate device memory.

Some callers of this library cannot call cudaMalloc: code running while a stream is
captured into a CUDA graph, runtimes that reserve all device memory for their own
pool, and loops that cannot afford the synchronization an allocation may cause.  This
entry point gives them the forward pass with the library's own fixed scratch instead
of a workspace.  Its results must match fckl_forward's and the oracle's, call after
call (the scratch is shared and keeps the previous call's contents), including when
the rows go through in several chunks: the caller's chunk smaller than T, or a chunk
the entry point shrinks itself because its rows would not fit the fixed scratch.
This file sorts last so that a run stopping at the first failure has run every other
test before it.
"""

import ctypes

import numpy as np
import pytest
import torch

from chunked_kl_loss_head_b300 import _lib, api
from gen import make_small
from helpers import TOL, oracle_of, rel, rel_max, to_device

SCRATCH_BYTES = 8 << 20  # FCKL_NOALLOC_SCRATCH_BYTES


def _scratch_rows(T, V, K, chunk):
    """Rows per internal chunk: the caller's chunk, shrunk (to a multiple of 128 rows
    while above 256) until a chunk's scratch fits the fixed array."""
    def up(x):
        return (x + 255) // 256 * 256

    nvt = (V + 255) // 256

    def need(r):
        return up(64) + 4 * up(4 * r * K) + up(8 * r * nvt)

    r = min(chunk, T)
    while r > 1 and need(r) > SCRATCH_BYTES:
        r = (r - 1) // 128 * 128 if r > 256 else r // 2
    return r


CASES = [
    # T, d, V, K, tau, chunk, dtype: one chunk; the caller's chunk below T; the scratch
    # forcing 1024-row chunks (7888 bytes per row at V = 201088, K = 100)
    (3000, 256, 20000, 20, 1.3, 4096, "bf16"),
    (3000, 256, 20000, 20, 1.3, 1000, "bf16"),
    (2500, 256, 201088, 100, 1.0, 4096, "bf16"),
    (3000, 256, 20000, 20, 1.3, 4096, "f32"),
    (2500, 64, 201088, 100, 2.0, 4096, "f32"),
]


@pytest.mark.gpu
@pytest.mark.parametrize("T,d,V,K,tau,chunk,dtype", CASES)
def test_noalloc_forward_matches_forward_and_oracle_two_calls(T, d, V, K, tau, chunk, dtype):
    x = make_small(T=T, d=d, V=V, K=K, tau=tau, dtype=dtype, seed=21, mask="random", mask_frac=0.1)
    g = to_device(x)
    ref_loss, ref_lse, ref_rl = api.forward(g["H"], g["W"], g["topk_idx"], g["topk_logits"], g["valid"], tau, chunk,
                                            want_row_loss=True)
    torch.cuda.synchronize()
    ora = oracle_of(x, want_grads=False)
    tol = TOL[dtype]["loss"]
    rows = _scratch_rows(T, V, K, chunk)
    n_chunks = -(-T // rows)
    if (V, K) == (201088, 100):
        assert rows == 1024 and n_chunks == 3  # the shrinking loop runs
    for call in range(2):
        loss = torch.full((), float("nan"), device="cuda")
        lse = torch.full((T,), float("nan"), device="cuda")
        rl = torch.full((T,), float("nan"), device="cuda")
        status = torch.full((), -1, dtype=torch.int32, device="cuda")
        n0 = api.fckl_launch_count()
        api.fckl_forward_noalloc(g["H"], g["W"], g["topk_idx"], g["topk_logits"], g["valid"], tau, chunk, loss, lse,
                                 rl, status)
        launches = api.fckl_launch_count() - n0
        torch.cuda.synchronize()
        # a clear of the control words, three launches per chunk, the mean, the status copy
        assert launches == 3 + 3 * n_chunks, (call, launches, n_chunks)
        assert int(status.item()) == 0, f"call {call}: status {int(status.item())}"
        got = dict(loss=loss.item(), lse=lse.cpu().numpy(), row_loss=rl.cpu().numpy())
        errs = dict(fwd_loss=rel(got["loss"], ref_loss.item()),
                    fwd_lse=rel_max(got["lse"], ref_lse.cpu().numpy()),
                    fwd_row_loss=rel_max(got["row_loss"], ref_rl.cpu().numpy()),
                    oracle_loss=rel(got["loss"], ora["loss"]), oracle_lse=rel_max(got["lse"], ora["lse"]),
                    oracle_row_loss=rel_max(got["row_loss"], ora["row_loss"]))
        print(f"call {call}: {n_chunks} chunks of {rows} rows", {k: f"{v:.2e}" for k, v in errs.items()})
        assert all(v <= tol for v in errs.values()), (call, errs)
        assert np.all(got["row_loss"][~np.asarray(x["valid"]).astype(bool)] == 0.0)


def test_noalloc_rejects_sizes_beyond_its_scratch():
    # one row of a 300M-id vocabulary needs more scratch than the fixed array holds;
    # the call is refused before anything touches a device
    L = _lib.lib()
    dummy = ctypes.c_void_p(1 << 20)
    st = L.fckl_forward_noalloc(dummy, dummy, dummy, dummy, dummy, 64, 256, 300_000_000, 10, 1.0, 64, 1, dummy, dummy,
                                dummy, None, None)
    assert st == 3, api.fckl_status_string(st)
