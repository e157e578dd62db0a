"""The oracle against its pins (CPU), and the pins against planted mistakes.

Each mutation below plants one plausible mistake in a copy of the oracle's
source (a dropped term, a wrong sign, a dropped temperature, a transposed or
shifted index, a wrong divisor, a leak through ignored rows); the pin suite
must reject every mutant, which shows the pins can tell a wrong oracle from
the right one.
"""

import inspect

import numpy as np
import pytest

import pins
from oracle import kl_oracle

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda p: p.__name__)
def test_oracle_pin(pin):
    pin(kl_oracle.fwd_bwd)


def test_row_block_invariance():
    H, W, idx, lg, valid = pins._tiny(seed=41, T=13, d=6, V=21, K=4, ignored=(3, 9))
    a = kl_oracle.fwd_bwd(H, W, idx, lg, valid, 1.4, row_block=1)
    b = kl_oracle.fwd_bwd(H, W, idx, lg, valid, 1.4, row_block=64)
    c = kl_oracle.fwd_bwd(H, W, idx, lg, valid, 1.4, row_block=5)
    for o in (b, c):
        assert abs(o["loss"] - a["loss"]) <= 1e-14 * abs(a["loss"])
        np.testing.assert_allclose(o["dW"], a["dW"], rtol=0, atol=1e-15 * np.abs(a["dW"]).max() * 10)
        np.testing.assert_allclose(o["lse"], a["lse"], rtol=1e-15, atol=0)


def test_dW_rows_subset():
    H, W, idx, lg, valid = pins._tiny(seed=43, T=7, d=5, V=30, K=4, ignored=(2,))
    full = kl_oracle.fwd_bwd(H, W, idx, lg, valid, 1.0)
    rows = [0, 5, 17, 29]
    sub = kl_oracle.fwd_bwd(H, W, idx, lg, valid, 1.0, dW_rows=rows)
    np.testing.assert_array_equal(sub["dW"], full["dW"][rows])


def test_rejects_out_of_range_ids():
    H, W, idx, lg, valid = pins._tiny(seed=47, T=3, d=4, V=8, K=2)
    idx[1, 0] = 8
    with pytest.raises(ValueError):
        kl_oracle.fwd_bwd(H, W, idx, lg, valid, 1.0)


MUTATIONS = {
    "dropped_student_lse": ("log_q_at = s[rows, idx[b0:b1]] - lse_b[:, None]",
                            "log_q_at = s[rows, idx[b0:b1]]"),
    "wrong_sign_teacher_in_dz": ("-p[b0:b1].ravel())", "p[b0:b1].ravel())"),
    "dropped_tau_in_gradient": ("scale = float(grad) / (tau * N)", "scale = float(grad) / N"),
    "dW_with_reversed_rows": ("dW += dzs.T @ H[b0:b1]", "dW += dzs.T @ H[b0:b1][::-1]"),
    "teacher_without_tau": ("a = np.asarray(topk_logits, dtype=np.float64) / float(tau)",
                            "a = np.asarray(topk_logits, dtype=np.float64)"),
    "ignored_rows_leak_into_grad": ("dz[~valid[b0:b1]] = 0.0", "pass"),
    "mean_over_all_rows": ("loss = float(row_loss.sum() / N)", "loss = float(row_loss.sum() / T)"),
    "teacher_lse_missing_max": ("lse_a = amax + np.log(", "lse_a = np.log("),
    "student_without_tau": ("s = (H[b0:b1] @ W.T) / tau", "s = (H[b0:b1] @ W.T)"),
    "teacher_scattered_to_wrong_ids": ("idx[b0:b1].ravel()),", "np.roll(idx[b0:b1], 1, axis=1).ravel()),"),
    "transposed_dH": ("dH[b0:b1] = dz @ W", "dH[b0:b1] = (W.T @ dz.T).T[:, ::-1]"),
    "terms_outside_support_kept": ("rl = np.where(pb > 0, terms, 0.0).sum(axis=1)", "rl = terms.sum(axis=1)"),
    "ignored_rows_masked_by_product": ("dz[~valid[b0:b1]] = 0.0", "dz *= valid[b0:b1, None]"),
}


def _mutant(old, new):
    src = inspect.getsource(kl_oracle)
    assert src.count(old) == 1, f"mutation site not found exactly once: {old!r}"
    ns = {}
    exec(compile(src.replace(old, new), "<mutant>", "exec"), ns)
    return ns["fwd_bwd"]


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_reject_planted_mistake(name):
    bad = _mutant(*MUTATIONS[name])
    caught = []
    for pin in pins.ALL_PINS:
        try:
            pin(bad)
        except (AssertionError, ValueError, IndexError):
            caught.append(pin.__name__)
    assert caught, f"no pin catches the planted mistake {name}"
