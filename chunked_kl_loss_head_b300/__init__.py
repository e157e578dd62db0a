"""Fused chunked KL distillation loss for NVIDIA B300 (sm_103a).

The loss compares a student with a teacher cached offline as top-K (id,
logit) pairs; the student's lm_head is folded into the loss, so the
[tokens x vocab] logits are never built.  All compute runs in libfckl.so
(hand-written CUDA, tcgen05 tensor cores for bf16); this package only
marshals torch tensors into its C-ABI.
"""

from .api import (  # noqa: F401
    BF16,
    F32,
    FcklError,
    backward,
    fckl_backward,
    fckl_debug_gemm_bf16,
    fckl_forward,
    fckl_get_error,
    fckl_launch_count,
    fckl_profile_enable,
    fckl_profile_read,
    fckl_status_string,
    fckl_topk_extract,
    fckl_workspace_size,
    forward,
    topk_extract,
    workspace,
)
from .autograd import FusedChunkedKLLoss, fused_chunked_kl_loss  # noqa: F401
