"""The C-ABI library on the CPU: it loads, exports every symbol include/fckl.h
declares, sizes workspaces, and rejects bad arguments before touching a GPU."""

import ctypes
import os
import re

import pytest

from chunked_kl_loss_head_b300 import _lib
from chunked_kl_loss_head_b300.api import BF16, F32

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_symbols():
    src = open(os.path.join(ROOT, "include", "fckl.h")).read()
    return sorted(set(re.findall(r"FCKL_API\s+[\w\s\*]+?\b(fckl_\w+)\s*\(", src)))


def test_library_exports_every_declared_symbol():
    L = _lib.lib()
    names = declared_symbols()
    assert len(names) >= 9
    for n in names:
        assert hasattr(L, n), f"{n} declared in fckl.h but not exported"
        assert n in _lib.PROTOTYPES, f"{n} has no ctypes prototype"


def test_status_strings():
    L = _lib.lib()
    seen = set()
    for code in range(7):
        s = L.fckl_status_string(code).decode()
        assert s and s != "unknown status"
        seen.add(s)
    assert len(seen) == 7
    assert L.fckl_status_string(99).decode() == "unknown status"


def test_workspace_size():
    ws = _lib.lib().fckl_workspace_size
    a = ws(131072, 2880, 201088, 100, 4096, BF16)
    assert 0 < a < 512 << 20, a  # O(chunk * vocab tile), never O(T * V)
    # T enters only through the per-row loss buffer (4 bytes per row)
    b = ws(262144, 2880, 201088, 100, 4096, BF16)
    assert 0 <= b - a <= 4 * 131072 + 256
    assert ws(131072, 2880, 201088, 100, 16384, BF16) > ws(131072, 2880, 201088, 100, 1024, BF16) / 2
    assert ws(64, 256, 4096, 10, 64, F32) > 0
    for bad in [(-1, 8, 8, 1, 1, 0), (8, 0, 8, 1, 1, 0), (8, 8, 0, 1, 1, 0), (8, 8, 8, 0, 1, 0),
                (8, 8, 8, 2000, 1, 0), (8, 8, 8, 1, 0, 0), (8, 8, 8, 1, 1, 7)]:
        assert ws(*bad) == 0, bad


def _fwd(**over):
    a = dict(H=1024, W=2048, idx=4096, lg=8192, valid=16384, T=64, d=256, V=4096, K=10, tau=1.0, chunk=64,
             dt=F32, loss=32768, lse=65536, rl=None, ws=1 << 20, ws_bytes=1 << 30, stream=None)
    a.update(over)
    return _lib.lib().fckl_forward(a["H"], a["W"], a["idx"], a["lg"], a["valid"], a["T"], a["d"], a["V"], a["K"],
                                   a["tau"], a["chunk"], a["dt"], a["loss"], a["lse"], a["rl"], a["ws"],
                                   a["ws_bytes"], a["stream"])


@pytest.mark.parametrize("over,code", [
    (dict(H=None), 1), (dict(valid=None), 1), (dict(loss=None), 1), (dict(tau=0.0), 1),
    (dict(tau=float("nan")), 1), (dict(tau=-1.0), 1), (dict(chunk=0), 1), (dict(K=0), 1), (dict(K=5000), 1),
    (dict(dt=3), 1), (dict(ws=None), 3), (dict(ws=1 << 20 | 8), 3), (dict(ws_bytes=100), 3),
    (dict(dt=BF16, d=250), 2), (dict(dt=BF16, H=1032), 2),
])
def test_forward_rejects_bad_arguments(over, code):
    assert _fwd(**over) == code


def test_backward_rejects_bad_arguments():
    L = _lib.lib()
    base = [1024, 2048, 4096, 8192, 16384, 64, 256, 4096, 10, 1.0, 64, F32, 32768, 1.0, None, 65536, 131072,
            1 << 20, 1 << 30, None]
    args = list(base)
    args[16] = None  # dW
    assert L.fckl_backward(*args) == 1
    args = list(base)
    args[13] = float("inf")  # grad_loss
    assert L.fckl_backward(*args) == 1
    args = list(base)
    args[18] = 10  # workspace too small
    assert L.fckl_backward(*args) == 3


def test_valid_arguments_need_a_device():
    # arguments pass the checks; with no usable GPU the call fails cleanly with a status
    import torch

    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert _fwd() in (2, 4)


def test_topk_rejects_bad_arguments():
    L = _lib.lib()
    p = ctypes.c_void_p(1 << 20)
    # K > V, K < 1, K above the limit, a bad dtype, T < 0: refused before any device work
    for T, V, K, dt in ((4, 100, 101, BF16), (4, 100, 0, BF16), (4, 5000, 1025, F32), (4, 100, 10, 7),
                        (-1, 100, 10, BF16)):
        assert L.fckl_topk_extract(p, T, V, K, dt, p, p, None) == 1
    # misaligned logits for fp32
    assert L.fckl_topk_extract(ctypes.c_void_p((1 << 20) + 2), 4, 100, 10, F32, p, p, None) == 2


def test_data_parallel_calls_reject_bad_arguments():
    L = _lib.lib()
    p = ctypes.c_void_p(1 << 20)
    # partials: no workspace, a workspace off 256 bytes or too small, no or misaligned output
    assert L.fckl_loss_partials(None, 1 << 20, p, None) == 3
    assert L.fckl_loss_partials(ctypes.c_void_p((1 << 20) + 8), 1 << 20, p, None) == 3
    assert L.fckl_loss_partials(p, 64, p, None) == 3
    assert L.fckl_loss_partials(p, 1 << 20, None, None) == 1
    assert L.fckl_loss_partials(p, 1 << 20, ctypes.c_void_p((1 << 20) + 4), None) == 1
    # finish: any null pointer, or a misaligned one
    for k in range(4):
        args = [p, p, p, p]
        args[k] = None
        assert L.fckl_loss_finish(*args, None) == 1
    assert L.fckl_loss_finish(ctypes.c_void_p((1 << 20) + 4), p, p, p, None) == 1
    assert L.fckl_loss_finish(p, p, ctypes.c_void_p((1 << 20) + 2), p, None) == 1


def test_cast_rejects_bad_arguments():
    L = _lib.lib()
    p = ctypes.c_void_p(1 << 20)
    assert L.fckl_cast_f32_to_bf16(None, p, 8, None) == 1
    assert L.fckl_cast_f32_to_bf16(p, p, -4, None) == 1
    assert L.fckl_cast_f32_to_bf16(p, p, 6, None) == 2  # not a multiple of 4
    assert L.fckl_cast_f32_to_bf16(ctypes.c_void_p((1 << 20) + 8), p, 8, None) == 2
    assert L.fckl_cast_f32_to_bf16(p, ctypes.c_void_p((1 << 20) + 4), 8, None) == 2
    assert L.fckl_cast_f32_to_bf16(None, None, 0, None) == 0  # nothing to do
