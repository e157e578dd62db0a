"""Writes oracle_tiny.json: oracle values on the tiny fp32 workload and on a
small bf16 workload, stored so that a later change to the oracle's arithmetic
shows up as a diff.  Calls only the oracle and the input generators.

    python tests/golden/make_golden.py
"""

import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

from gen import CONFIGS, bf16_bits_to_f32, make_inputs, make_small  # noqa: E402
from oracle import fwd_bwd  # noqa: E402


def entry(x):
    H, W = x["H"], x["W"]
    if H.dtype == np.uint16:
        H, W = bf16_bits_to_f32(H), bf16_bits_to_f32(W)
    cfg = x["cfg"]
    o = fwd_bwd(H, W, x["topk_idx"], x["topk_logits"], x["valid"], cfg.tau)
    return dict(loss=o["loss"], N=o["N"], lse_head=o["lse"][:8].tolist(),
                row_loss_head=o["row_loss"][:8].tolist(), dH_0_head=o["dH"][0, :8].tolist(),
                dW_rows={str(v): o["dW"][v, :8].tolist() for v in (0, 1, 7, cfg.V - 1)})


def main():
    out = {
        "_about": "oracle regression values; written by tests/golden/make_golden.py (oracle + generators only)",
        "tiny_fp32": entry(make_inputs(CONFIGS["tiny_fp32"])),
        "small_bf16": entry(make_small(T=40, d=72, V=700, K=7, tau=1.5, dtype="bf16", seed=5,
                                       mask="random", mask_frac=0.2, name="small_bf16")),
    }
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "oracle_tiny.json")
    with open(path, "w") as f:
        json.dump(out, f, indent=1)
    print("wrote", path)


if __name__ == "__main__":
    main()
