"""The seeded input generators: determinism, shapes and the stated structure."""

import numpy as np
import pytest

from gen import CONFIGS, bf16_bits_to_f32, f32_to_bf16_bits, make_inputs, make_rows, valid_mask
from gen.synthetic import _topk_rows


def test_tiny_deterministic_and_shaped():
    cfg = CONFIGS["tiny_fp32"]
    a = make_inputs(cfg)
    b = make_inputs(cfg)
    for k in ("H", "W", "topk_idx", "topk_logits", "valid"):
        np.testing.assert_array_equal(a[k], b[k])
    assert a["H"].shape == (64, 256) and a["H"].dtype == np.float32
    assert a["W"].shape == (4096, 256)
    assert a["topk_idx"].shape == (64, 10) and a["topk_idx"].dtype == np.int32
    assert a["topk_logits"].dtype == np.float32
    assert a["valid"].all()
    # W ~ N(0, 1/d): z = H W^T ~ N(0, 1)
    assert abs(a["W"].std() * np.sqrt(256) - 1.0) < 0.02


@pytest.mark.parametrize("name", ["llama_bf16", "gptoss_bf16", "longctx_bf16", "stress_bf16"])
def test_topk_structure(name):
    cfg = CONFIGS[name]
    rows = np.unique(np.concatenate([np.arange(0, 300), np.arange(cfg.T - 300, cfg.T)]))
    idx, lg = _topk_rows(cfg, rows)
    assert idx.shape == (len(rows), cfg.K)
    assert idx.min() >= 0 and idx.max() < cfg.V
    assert all(len(set(r)) == cfg.K for r in idx)
    assert np.all(np.diff(lg, axis=1) <= 0), "teacher logits not sorted descending"
    if cfg.ids == "zipf":
        assert np.median(idx[:, 0]) < 500  # heavy head (uniform: ~V/2)
    else:
        assert np.median(idx) > cfg.V / 4


def test_masks_and_onehot():
    assert int((valid_mask(CONFIGS["llama_bf16"]) == 0).sum()) == 410
    v = valid_mask(CONFIGS["gptoss_bf16"])
    assert int((v == 0).sum()) == 4 * 655
    assert v[32768 - 655:32768].sum() == 0 and v[32768 - 656] == 1
    v = valid_mask(CONFIGS["longctx_bf16"])
    assert int((v == 0).sum()) == 5242 and v[-5242:].sum() == 0
    assert valid_mask(CONFIGS["stress_bf16"]).all()
    cfg = CONFIGS["stress_bf16"]
    _, lg = _topk_rows(cfg, np.arange(4096))
    hot = (lg[:, 0] - lg[:, 1]) > 25
    assert 0.07 < hot.mean() < 0.13


def test_rows_match_full():
    cfg = CONFIGS["llama_bf16"].with_(T=3000, V=5000, d=64)
    full = make_inputs(cfg)
    rows = [0, 1023, 1024, 2999, 17]
    r = make_rows(cfg, rows)
    for k in ("H", "topk_idx", "topk_logits", "valid"):
        np.testing.assert_array_equal(r[k], full[k][rows])


def test_bf16_round_trip():
    x = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5, 3.0e38, 1e-40], np.float32)
    b = f32_to_bf16_bits(x)
    y = bf16_bits_to_f32(b)
    assert y[0] == 1.0 and y[1] == 1.0  # tie to even
    assert y[2] == 1.0 + 2 ** -6  # 1 + 3*2^-8 rounds up to the even neighbour
    assert y[3] == -2.5
