"""Seeded synthetic inputs for the fused chunked KL loss (shared by the tests,
the bench and the oracle checks).  Holds no loss arithmetic."""

from .synthetic import (  # noqa: F401
    CONFIGS,
    Config,
    bf16_bits_to_f32,
    f32_to_bf16_bits,
    make_inputs,
    make_rows,
    make_small,
    make_teacher_logits,
    make_W,
    valid_mask,
)
