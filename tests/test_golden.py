"""Stored values: the pages' printed figures and the oracle's regression values."""

import json
import os

import numpy as np

from gen import CONFIGS, bf16_bits_to_f32, make_inputs, make_small
from oracle import fwd_bwd

HERE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def test_pages_dense_tensor_figure():
    g = json.load(open(os.path.join(HERE, "pages_figures.json")))
    t = g["dense_teacher_tensor"]
    from chunked_kl_loss_head_b300.memory import dense_logit_bytes

    nbytes = dense_logit_bytes(t["batch"] * t["seq_len"], t["vocab"], t["bytes_per_elem"])
    assert abs(nbytes / 1e9 - t["approx_gb"]) <= t["approx_rel_tol"] * t["approx_gb"]
    b = g["isolated_benchmark_32k"]
    assert abs(b["dense_gib"] / b["fused_gib"] - b["ratio"]) < 0.05


def _check(entry, x):
    H, W = x["H"], x["W"]
    if H.dtype == np.uint16:
        H, W = bf16_bits_to_f32(H), bf16_bits_to_f32(W)
    o = fwd_bwd(H, W, x["topk_idx"], x["topk_logits"], x["valid"], x["cfg"].tau)
    assert abs(o["loss"] - entry["loss"]) <= 1e-12 * abs(entry["loss"])
    assert o["N"] == entry["N"]
    np.testing.assert_allclose(o["lse"][:8], entry["lse_head"], rtol=1e-12)
    np.testing.assert_allclose(o["row_loss"][:8], entry["row_loss_head"], rtol=1e-12)
    np.testing.assert_allclose(o["dH"][0, :8], entry["dH_0_head"], rtol=1e-10, atol=1e-18)
    for v, vals in entry["dW_rows"].items():
        np.testing.assert_allclose(o["dW"][int(v), :8], vals, rtol=1e-10, atol=1e-18)


def test_oracle_regression_values():
    g = json.load(open(os.path.join(HERE, "oracle_tiny.json")))
    _check(g["tiny_fp32"], make_inputs(CONFIGS["tiny_fp32"]))
    _check(g["small_bf16"], make_small(T=40, d=72, V=700, K=7, tau=1.5, dtype="bf16", seed=5,
                                       mask="random", mask_frac=0.2, name="small_bf16"))
