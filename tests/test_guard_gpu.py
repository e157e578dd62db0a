"""Out-of-bounds writes, checked without a sanitizer: every buffer the library writes
(the workspace, loss, lse, per-row losses, dH, dW, the top-K outputs, and the outputs of
the allocation-free forward) is carved out of
a larger allocation whose margins hold a known byte pattern; after the calls the margins
must be untouched and the results must still match the oracle.  The shapes put ragged
edges everywhere: rows not a multiple of the 256-row tile, a vocabulary not a multiple of
the 256-column tile or of the stripe, several chunks and stripes, and odd top-K rows."""

import numpy as np
import pytest
import torch

from chunked_kl_loss_head_b300 import api
from gen import bf16_bits_to_f32, f32_to_bf16_bits, make_small
from helpers import TOL, oracle_of, rel, rel_max, to_device
from oracle import topk_rows

pytestmark = pytest.mark.gpu

MARGIN = 8192  # bytes of pattern before and after each buffer (a multiple of 256)
PATTERN = 0xA5


class Guarded:
    """A device buffer of `nbytes` between two margins of PATTERN bytes."""

    def __init__(self, nbytes):
        self.n = int(nbytes)
        self.raw = torch.full((self.n + 2 * MARGIN,), PATTERN, dtype=torch.uint8, device="cuda")

    def view(self, dtype, shape):
        return self.raw[MARGIN:MARGIN + self.n].view(dtype).view(shape)

    def margins_intact(self):
        head = self.raw[:MARGIN]
        tail = self.raw[MARGIN + self.n:]
        return bool((head == PATTERN).all().item()) and bool((tail == PATTERN).all().item())


def _nbytes(dtype, shape):
    return int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("T,d,V,K,chunk", [(300, 64, 1000, 7, 128), (1000, 256, 50001, 20, 384),
                                           (5000, 64, 9000, 5, 4500)])
def test_loss_writes_stay_in_bounds(dtype, T, d, V, K, chunk):
    x = make_small(T, d, V, K, tau=1.5, dtype=dtype, seed=11, mask="random", mask_frac=0.1)
    dev = to_device(x)
    tdt = dev["H"].dtype
    ws_n = api.fckl_workspace_size(T, d, V, K, chunk, tdt)
    bufs = dict(ws=Guarded(ws_n), loss=Guarded(4), lse=Guarded(4 * T), rl=Guarded(4 * T),
                dH=Guarded(_nbytes(tdt, (T, d))), dW=Guarded(4 * V * d))
    ws = bufs["ws"].view(torch.uint8, (ws_n,))
    ws.zero_()
    loss = bufs["loss"].view(torch.float32, ())
    lse = bufs["lse"].view(torch.float32, (T,))
    rl = bufs["rl"].view(torch.float32, (T,))
    dH = bufs["dH"].view(tdt, (T, d))
    dW = bufs["dW"].view(torch.float32, (V, d))
    api.fckl_forward(dev["H"], dev["W"], dev["topk_idx"], dev["topk_logits"], dev["valid"], x["cfg"].tau, chunk,
                     loss, lse, rl, ws)
    api.fckl_backward(dev["H"], dev["W"], dev["topk_idx"], dev["topk_logits"], dev["valid"], x["cfg"].tau, chunk,
                      lse, 1.0, dH, dW, ws)
    torch.cuda.synchronize()
    assert api.fckl_get_error(ws) == 0
    for name, b in bufs.items():
        assert b.margins_intact(), f"write outside {name}"
    ref = oracle_of(x)
    tol = TOL[dtype]
    assert rel(loss.item(), ref["loss"]) <= tol["loss"]
    assert rel_max(dH.float().cpu().numpy(), ref["dH"]) <= tol["grad"]
    assert rel_max(dW.cpu().numpy(), ref["dW"]) <= tol["grad"]


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("T,d,V,K,chunk", [(300, 64, 1000, 7, 128), (1000, 256, 50001, 20, 384),
                                           (1300, 64, 201088, 100, 4096)])
def test_noalloc_forward_writes_stay_in_bounds(dtype, T, d, V, K, chunk):
    """fckl_forward_noalloc's outputs (loss, lse, per-row losses, status) between guarded
    margins; the last shape makes the call shrink its chunk to fit its fixed scratch."""
    x = make_small(T, d, V, K, tau=1.5, dtype=dtype, seed=12, mask="random", mask_frac=0.1)
    dev = to_device(x)
    bufs = dict(loss=Guarded(4), lse=Guarded(4 * T), rl=Guarded(4 * T), status=Guarded(4))
    loss = bufs["loss"].view(torch.float32, ())
    lse = bufs["lse"].view(torch.float32, (T,))
    rl = bufs["rl"].view(torch.float32, (T,))
    status = bufs["status"].view(torch.int32, ())
    api.fckl_forward_noalloc(dev["H"], dev["W"], dev["topk_idx"], dev["topk_logits"], dev["valid"], x["cfg"].tau,
                             chunk, loss, lse, rl, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    for name, b in bufs.items():
        assert b.margins_intact(), f"write outside {name}"
    ref = oracle_of(x, want_grads=False)
    tol = TOL[dtype]
    assert rel(loss.item(), ref["loss"]) <= tol["loss"]
    assert rel_max(lse.cpu().numpy(), ref["lse"]) <= tol["loss"]
    assert rel_max(rl.cpu().numpy(), ref["row_loss"]) <= tol["loss"]


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("T,V,K", [(9, 20011, 100), (5, 37, 37), (3, 201088, 1024)])
def test_topk_writes_stay_in_bounds(dtype, T, V, K):
    rng = np.random.default_rng(V + K)
    x = rng.standard_normal((T, V)).astype(np.float32)
    if dtype == "bf16":
        bits = f32_to_bf16_bits(x)
        ref_in = bf16_bits_to_f32(bits)
        src = Guarded(2 * T * V)
        logits = src.view(torch.bfloat16, (T, V))
        logits.copy_(torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16))
    else:
        ref_in = x
        src = Guarded(4 * T * V)
        logits = src.view(torch.float32, (T, V))
        logits.copy_(torch.from_numpy(x))
    gi, gv = Guarded(4 * T * K), Guarded(4 * T * K)
    idx, val = gi.view(torch.int32, (T, K)), gv.view(torch.float32, (T, K))
    api.fckl_topk_extract(logits, K, idx, val)
    torch.cuda.synchronize()
    assert gi.margins_intact() and gv.margins_intact() and src.margins_intact()
    ref_idx, ref_val = topk_rows(ref_in, K)
    assert np.array_equal(idx.cpu().numpy(), ref_idx)
    assert np.array_equal(val.cpu().numpy().view(np.uint32), ref_val.view(np.uint32))
