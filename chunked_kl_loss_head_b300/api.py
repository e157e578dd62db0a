"""Python binding of the C-ABI (argument marshalling only).

The functions named like the C entry points take torch tensors that already
live on the current CUDA device and pass their pointers through; every step of
the loss runs in libfckl.so's kernels.  ``forward`` / ``backward`` are
conveniences that also allocate the outputs and the workspace with torch.
"""

from __future__ import annotations

import ctypes

import torch

from ._lib import lib

F32, BF16 = 0, 1
STATUS = {0: "FCKL_OK", 1: "FCKL_ERR_INVALID_ARG", 2: "FCKL_ERR_UNSUPPORTED", 3: "FCKL_ERR_WORKSPACE",
          4: "FCKL_ERR_CUDA", 5: "FCKL_ERR_BAD_INDEX", 6: "FCKL_ERR_TIMEOUT"}
KERNEL_CLASSES = ["prep", "fwd_tiles", "combine", "reduce", "bwd_tiles", "grad_gemm", "other", "topk"]


class FcklError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = int(status)
        super().__init__(f"{where}: {STATUS.get(self.status, self.status)} ({fckl_status_string(self.status)})")


def _check(status: int, where: str) -> None:
    if status != 0:
        raise FcklError(status, where)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return F32
    if t.dtype == torch.bfloat16:
        return BF16
    raise TypeError(f"H / W must be float32 or bfloat16, got {t.dtype}")


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensors must be on a CUDA device")
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _shapes(H, W, topk_idx, topk_logits, valid):
    T, d = H.shape
    V, d2 = W.shape
    K = topk_idx.shape[1]
    if d2 != d or H.dtype != W.dtype:
        raise ValueError("H and W must share d and dtype")
    if topk_idx.shape != (T, K) or topk_logits.shape != (T, K) or valid.shape != (T,):
        raise ValueError("topk_idx / topk_logits must be [T, K] and valid [T]")
    if topk_idx.dtype != torch.int32 or topk_logits.dtype != torch.float32 or valid.dtype != torch.uint8:
        raise TypeError("topk_idx int32, topk_logits float32, valid uint8 expected")
    return T, d, V, K


# ------------------------------------------------------------------------------ C-ABI names


def fckl_status_string(status: int) -> str:
    return lib().fckl_status_string(int(status)).decode()


def fckl_workspace_size(T: int, d: int, V: int, K: int, chunk: int, dtype) -> int:
    code = dtype if isinstance(dtype, int) else (F32 if dtype == torch.float32 else BF16)
    return int(lib().fckl_workspace_size(T, d, V, K, chunk, code))


def fckl_forward(H, W, topk_idx, topk_logits, valid, tau, chunk, loss, lse, row_loss, ws, stream=None):
    T, d, V, K = _shapes(H, W, topk_idx, topk_logits, valid)
    st = lib().fckl_forward(_ptr(H), _ptr(W), _ptr(topk_idx), _ptr(topk_logits), _ptr(valid), T, d, V, K,
                            float(tau), int(chunk), _dtype_code(H), _ptr(loss), _ptr(lse), _ptr(row_loss),
                            _ptr(ws), ws.numel() * ws.element_size(), _stream(stream))
    _check(st, "fckl_forward")


def fckl_backward(H, W, topk_idx, topk_logits, valid, tau, chunk, lse, grad_loss, dH, dW, ws, grad_scale=None,
                  stream=None):
    T, d, V, K = _shapes(H, W, topk_idx, topk_logits, valid)
    st = lib().fckl_backward(_ptr(H), _ptr(W), _ptr(topk_idx), _ptr(topk_logits), _ptr(valid), T, d, V, K,
                             float(tau), int(chunk), _dtype_code(H), _ptr(lse), float(grad_loss),
                             _ptr(grad_scale), _ptr(dH), _ptr(dW), _ptr(ws), ws.numel() * ws.element_size(),
                             _stream(stream))
    _check(st, "fckl_backward")


def fckl_forward_noalloc(H, W, topk_idx, topk_logits, valid, tau, chunk, loss, lse, row_loss, status=None,
                         stream=None):
    """fckl_forward for callers that cannot allocate device memory: no workspace, the
    library's own fixed scratch instead; row_loss is required, status optional."""
    T, d, V, K = _shapes(H, W, topk_idx, topk_logits, valid)
    st = lib().fckl_forward_noalloc(_ptr(H), _ptr(W), _ptr(topk_idx), _ptr(topk_logits), _ptr(valid), T, d, V, K,
                                    float(tau), int(chunk), _dtype_code(H), _ptr(loss), _ptr(lse), _ptr(row_loss),
                                    _ptr(status), _stream(stream))
    _check(st, "fckl_forward_noalloc")


def fckl_loss_partials(ws, partials, stream=None):
    """partials (float64 [2] on the device) = (sum of loss_t over valid rows, N) of the last
    fckl_forward on ws."""
    _check(lib().fckl_loss_partials(_ptr(ws), ws.numel() * ws.element_size(), _ptr(partials), _stream(stream)),
           "fckl_loss_partials")


def fckl_loss_finish(total, local, loss, grad_scale, stream=None):
    """loss = total[0] / total[1]; grad_scale = local[1] / total[1] (both 0 when total[1] is 0)."""
    _check(lib().fckl_loss_finish(_ptr(total), _ptr(local), _ptr(loss), _ptr(grad_scale), _stream(stream)),
           "fckl_loss_finish")


def fckl_cast_f32_to_bf16(src, dst, stream=None):
    """dst (bfloat16) = src (float32) rounded to nearest even, element by element."""
    if src.dtype != torch.float32 or dst.dtype != torch.bfloat16 or src.numel() != dst.numel():
        raise TypeError("float32 source and bfloat16 destination of the same size expected")
    _check(lib().fckl_cast_f32_to_bf16(_ptr(src), _ptr(dst), src.numel(), _stream(stream)), "fckl_cast_f32_to_bf16")


def to_dtype(dW, dtype, stream=None):
    """dW in `dtype`: itself when it already has it, the library's cast from float32 to
    bfloat16 otherwise (any other pair is refused)."""
    if dW.dtype == dtype:
        return dW
    if dW.dtype != torch.float32 or dtype != torch.bfloat16:
        raise TypeError(f"no cast from {dW.dtype} to {dtype}")
    out = torch.empty(dW.shape, dtype=dtype, device=dW.device)
    fckl_cast_f32_to_bf16(dW, out, stream)
    return out


def fckl_topk_extract(logits, K, topk_idx, topk_logits, stream=None):
    """Per row of logits [T, V] (float32 or bfloat16): the K largest values and their ids,
    value descending then id ascending, into topk_idx [T, K] int32 / topk_logits float32."""
    if logits.dim() != 2:
        raise ValueError("logits must be [T, V]")
    T, V = logits.shape
    if topk_idx.shape != (T, K) or topk_logits.shape != (T, K):
        raise ValueError("outputs must be [T, K]")
    if topk_idx.dtype != torch.int32 or topk_logits.dtype != torch.float32:
        raise TypeError("topk_idx int32 and topk_logits float32 expected")
    _check(lib().fckl_topk_extract(_ptr(logits), T, V, int(K), _dtype_code(logits), _ptr(topk_idx),
                                   _ptr(topk_logits), _stream(stream)), "fckl_topk_extract")


def topk_extract(logits, K, stream=None):
    """(topk_idx [T, K] int32, topk_logits [T, K] float32) on logits' device."""
    T = logits.shape[0]
    idx = torch.empty((T, K), dtype=torch.int32, device=logits.device)
    val = torch.empty((T, K), dtype=torch.float32, device=logits.device)
    fckl_topk_extract(logits, K, idx, val, stream)
    return idx, val


def fckl_get_error(ws, stream=None) -> int:
    return int(lib().fckl_get_error(_ptr(ws), _stream(stream)))


def fckl_launch_count() -> int:
    return int(lib().fckl_launch_count())


def fckl_profile_enable(on: bool) -> None:
    lib().fckl_profile_enable(1 if on else 0)


def fckl_profile_read(kernel_class, reset: bool = False):
    """(launches, total device ms) of one kernel class since the last reset."""
    cls = KERNEL_CLASSES.index(kernel_class) if isinstance(kernel_class, str) else int(kernel_class)
    n = ctypes.c_int64(0)
    ms = ctypes.c_double(0.0)
    _check(lib().fckl_profile_read(cls, ctypes.byref(n), ctypes.byref(ms), 1 if reset else 0), "fckl_profile_read")
    return int(n.value), float(ms.value)


def fckl_debug_wait_timeout(ws, stream=None):
    _check(lib().fckl_debug_wait_timeout(_ptr(ws), ws.numel() * ws.element_size(), _stream(stream)),
           "fckl_debug_wait_timeout")


def fckl_debug_gemm_bf16(A, B, D, M, N, K, a_mn, b_mn, cta_pair=1, stream=None):
    _check(lib().fckl_debug_gemm_bf16(_ptr(A), _ptr(B), _ptr(D), M, N, K, int(a_mn), int(b_mn), int(cta_pair),
                                      _stream(stream)), "fckl_debug_gemm_bf16")


# ------------------------------------------------------------------------------ conveniences


def workspace(T, d, V, K, chunk, dtype, device=None) -> torch.Tensor:
    n = fckl_workspace_size(T, d, V, K, chunk, dtype)
    if n == 0:
        raise ValueError("invalid sizes for a workspace")
    return torch.zeros(n, dtype=torch.uint8, device=device or torch.device("cuda"))


def forward(H, W, topk_idx, topk_logits, valid, tau=1.0, chunk=4096, ws=None, want_row_loss=False, stream=None):
    """(loss scalar, lse[T]) (and row_loss[T] when asked) on H's device."""
    T, d, V, K = _shapes(H, W, topk_idx, topk_logits, valid)
    dev = H.device
    if ws is None:
        ws = workspace(T, d, V, K, chunk, H.dtype, dev)
    loss = torch.empty((), dtype=torch.float32, device=dev)
    lse = torch.empty(T, dtype=torch.float32, device=dev)
    rl = torch.empty(T, dtype=torch.float32, device=dev) if want_row_loss else None
    fckl_forward(H, W, topk_idx, topk_logits, valid, tau, chunk, loss, lse, rl, ws, stream)
    return (loss, lse, rl) if want_row_loss else (loss, lse)


def backward(H, W, topk_idx, topk_logits, valid, lse, tau=1.0, chunk=4096, grad_loss=1.0, ws=None,
             grad_scale=None, stream=None):
    """(dH[T, d] in H's dtype, dW[V, d] float32)."""
    T, d, V, K = _shapes(H, W, topk_idx, topk_logits, valid)
    dev = H.device
    if ws is None:
        ws = workspace(T, d, V, K, chunk, H.dtype, dev)
    dH = torch.empty((T, d), dtype=H.dtype, device=dev)
    dW = torch.empty((V, d), dtype=torch.float32, device=dev)
    fckl_backward(H, W, topk_idx, topk_logits, valid, tau, chunk, lse, grad_loss, dH, dW, ws, grad_scale, stream)
    return dH, dW
