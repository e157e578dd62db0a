"""ctypes loader of libfckl.so with the prototypes of include/fckl.h.

The library is built in-tree (``python -m chunked_kl_loss_head_b300.build``).
There is no fallback: if it is missing, importing the package's compute
functions raises, so nothing can silently run elsewhere.
"""

from __future__ import annotations

import ctypes
import os

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libfckl.so")

c_i64, c_i32, c_f32, c_f64, c_vp, c_sz = (ctypes.c_int64, ctypes.c_int32, ctypes.c_float, ctypes.c_double,
                                           ctypes.c_void_p, ctypes.c_size_t)

PROTOTYPES = {
    "fckl_workspace_size": (c_sz, [c_i64, c_i64, c_i64, c_i32, c_i64, c_i32]),
    "fckl_forward": (c_i32, [c_vp, c_vp, c_vp, c_vp, c_vp, c_i64, c_i64, c_i64, c_i32, c_f32, c_i64, c_i32,
                             c_vp, c_vp, c_vp, c_vp, c_sz, c_vp]),
    "fckl_backward": (c_i32, [c_vp, c_vp, c_vp, c_vp, c_vp, c_i64, c_i64, c_i64, c_i32, c_f32, c_i64, c_i32,
                              c_vp, c_f32, c_vp, c_vp, c_vp, c_vp, c_sz, c_vp]),
    "fckl_get_error": (c_i32, [c_vp, c_vp]),
    "fckl_loss_partials": (c_i32, [c_vp, c_sz, c_vp, c_vp]),
    "fckl_loss_finish": (c_i32, [c_vp, c_vp, c_vp, c_vp, c_vp]),
    "fckl_cast_f32_to_bf16": (c_i32, [c_vp, c_vp, c_i64, c_vp]),
    "fckl_status_string": (ctypes.c_char_p, [c_i32]),
    "fckl_launch_count": (c_i64, []),
    "fckl_profile_enable": (None, [ctypes.c_int]),
    "fckl_profile_read": (c_i32, [c_i32, ctypes.POINTER(c_i64), ctypes.POINTER(c_f64), ctypes.c_int]),
    "fckl_debug_gemm_bf16": (c_i32, [c_vp, c_vp, c_vp, c_i64, c_i64, c_i64, c_i32, c_i32, c_i32, c_vp]),
    "fckl_debug_wait_timeout": (c_i32, [c_vp, c_sz, c_vp]),
    "fckl_topk_extract": (c_i32, [c_vp, c_i64, c_i64, c_i32, c_i32, c_vp, c_vp, c_vp]),
    "fckl_forward_noalloc": (c_i32, [c_vp, c_vp, c_vp, c_vp, c_vp, c_i64, c_i64, c_i64, c_i32, c_f32, c_i64, c_i32,
                                     c_vp, c_vp, c_vp, c_vp, c_vp]),
}

_lib = None


def lib() -> ctypes.CDLL:
    """The loaded library (loaded once).  Raises ImportError when it is not built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: build it with `python -m chunked_kl_loss_head_b300.build`")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in PROTOTYPES.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib
