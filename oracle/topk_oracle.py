"""CPU oracle for teacher top-K extraction: the offline step that builds the cache.

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import or run this module.  It shares no code
with the CUDA library and never calls it.

What it computes
----------------
The teacher's knowledge is cached offline as, per token position, only its K
largest logits and the ids they belong to, so that the teacher never has to be
resident during student training (getaibook.com, "Preparing Offline Top-K
Logits"; axbrief.com, "Breaking the Bottleneck with Offline Caching and Chunked
Loss"; top-100 in calcaas.com, "What actually changed?").  For every row of a
[T, V] teacher logit matrix this returns the K entries that come first in the
order

    value descending, then id ascending,

so the result is unique even when values tie (bf16 logits tie often).  Values
are ordered by their IEEE-754 bit patterns read as sign-magnitude numbers:
that is the numeric order for all non-NaN values, with -0 placed just below +0,
and puts NaNs with the sign bit clear above +inf and NaNs with it set below
-inf.  The returned values are the inputs widened exactly to float32.
"""

from __future__ import annotations

import numpy as np

__all__ = ["order_keys", "topk_rows"]


def order_keys(values_f32: np.ndarray) -> np.ndarray:
    """uint32 keys whose unsigned order is the value order above (float32 input)."""
    u = np.ascontiguousarray(values_f32, dtype=np.float32).view(np.uint32)
    neg = (u >> np.uint32(31)).astype(bool)
    return np.where(neg, ~u, u | np.uint32(0x80000000)).astype(np.uint32)


def topk_rows(logits: np.ndarray, K: int):
    """(ids[T, K] int32, values[T, K] float32): per row, the first K entries by
    (value descending, id ascending).  `logits` is float32 [T, V] (bf16 inputs are
    passed widened to float32, which is exact)."""
    x = np.ascontiguousarray(logits, dtype=np.float32)
    T, V = x.shape
    if not 1 <= K <= V:
        raise ValueError("need 1 <= K <= V")
    ids = np.empty((T, K), np.int32)
    vals = np.empty((T, K), np.float32)
    col = np.arange(V, dtype=np.int64)
    for t in range(T):
        key = order_keys(x[t]).astype(np.int64)
        # lexsort sorts by the last key first: primary -key (value descending), then id
        order = np.lexsort((col, -key))[:K]
        ids[t] = order
        vals[t] = x[t, order]
    return ids, vals
