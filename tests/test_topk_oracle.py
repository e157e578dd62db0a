"""The top-K extraction oracle against what fixes it independently (CPU):

* a library routine: with distinct values, the K largest by numpy's sort agree;
* brute force on tiny rows with heavy ties: every K-subset rule checked by
  comparing against a pure-Python selection written from the definition;
* invariants: values non-increasing, ids distinct, each value equals the logit
  at its id, nothing left out exceeds the K-th value, ties resolved by id;
* special cases: K = V returns the full order; the key order matches float
  order, with -0 below +0 and NaNs outside +-inf.
A planted mistake in a copy of the oracle (ties by id descending, ascending
values, a dropped sign flip in the key) must fail one of these checks.
"""

import inspect

import numpy as np
import pytest

from oracle import topk_oracle
from oracle.topk_oracle import order_keys, topk_rows


def _brute(row, K):
    # selection sort written from the definition: repeatedly take the largest value,
    # the smallest id among equals; values compared as Python floats (no NaN here)
    left = list(range(len(row)))
    out = []
    for _ in range(K):
        best = None
        for i in left:
            if best is None or row[i] > row[best] or (row[i] == row[best] and i < best):
                best = i
        out.append(best)
        left.remove(best)
    return out


def check_topk(f):
    rng = np.random.default_rng(0)
    # distinct values: agrees with numpy's descending sort
    x = rng.standard_normal((7, 300)).astype(np.float32)
    ids, vals = f(x, 17)
    ref = np.argsort(-x, axis=1, kind="stable")[:, :17]
    assert np.array_equal(ids, ref)
    assert np.array_equal(vals, np.take_along_axis(x, ref, 1))
    # heavy ties (values from a set of 5): brute force
    x = rng.integers(-2, 3, size=(9, 23)).astype(np.float32)
    for K in (1, 4, 11, 23):
        ids, vals = f(x, K)
        for t in range(x.shape[0]):
            assert list(ids[t]) == _brute([float(v) for v in x[t]], K), (t, K)
    # invariants on a bf16-like grid (many ties)
    x = (np.round(rng.standard_normal((5, 1000)) * 8) / 8).astype(np.float32)
    ids, vals = f(x, 50)
    for t in range(5):
        assert len(set(ids[t].tolist())) == 50
        assert np.all(np.diff(vals[t]) <= 0)
        assert np.array_equal(vals[t], x[t, ids[t]])
        rest = np.setdiff1d(np.arange(1000), ids[t])
        assert x[t, rest].max() <= vals[t, -1]
        tied = rest[x[t, rest] == vals[t, -1]]
        assert tied.size == 0 or tied.min() > ids[t][vals[t] == vals[t, -1]].max()


def test_topk_oracle_pins():
    check_topk(topk_rows)


def test_order_keys():
    v = np.array([-np.inf, -3.5, -1e-30, -0.0, 0.0, 1e-30, 2.0, np.inf], np.float32)
    k = order_keys(v)
    assert np.all(np.diff(k.astype(np.int64)) > 0)
    nan_pos = np.array([np.nan], np.float32)
    nan_neg = (nan_pos.view(np.uint32) | np.uint32(0x80000000)).view(np.float32)
    assert order_keys(nan_pos)[0] > order_keys(np.array([np.inf], np.float32))[0]
    assert order_keys(nan_neg)[0] < order_keys(np.array([-np.inf], np.float32))[0]


def test_k_equals_v_is_full_order():
    x = np.array([[3.0, 1.0, 3.0, -2.0, 1.0]], np.float32)
    ids, vals = topk_rows(x, 5)
    assert ids.tolist() == [[0, 2, 1, 4, 3]]
    assert vals.tolist() == [[3.0, 3.0, 1.0, 1.0, -2.0]]


MUTATIONS = {
    "ties_by_id_descending": ("order = np.lexsort((col, -key))[:K]", "order = np.lexsort((-col, -key))[:K]"),
    "ascending_values": ("order = np.lexsort((col, -key))[:K]", "order = np.lexsort((col, key))[:K]"),
    "no_sign_flip": ("return np.where(neg, ~u, u | np.uint32(0x80000000)).astype(np.uint32)",
                     "return (u | np.uint32(0x80000000)).astype(np.uint32)"),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_reject_planted_mistake(name):
    old, new = MUTATIONS[name]
    src = inspect.getsource(topk_oracle)
    assert src.count(old) == 1
    ns = {}
    exec(compile(src.replace(old, new), "<mutant>", "exec"), ns)
    with pytest.raises(AssertionError):
        check_topk(ns["topk_rows"])
