"""Memory accounting for the loss (what the fused path avoids and what it needs)."""


def dense_logit_bytes(tokens: int, vocab: int, bytes_per_elem: int = 2) -> int:
    """Bytes of one dense [tokens x vocab] logit (or probability) tensor: the
    tensor the fused chunked loss never builds.  For batch 4 x 32K tokens over
    the 201,088-id gpt-oss vocabulary in bfloat16 this is the ~50 GB teacher
    tensor the pages describe (axbrief.com, "The 250GB VRAM Wall in
    Long-Context Distillation")."""
    return int(tokens) * int(vocab) * int(bytes_per_elem)
