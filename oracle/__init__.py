"""fp64 CPU oracle of the fused chunked KL loss, and the CPU oracle of the teacher
top-K extraction that builds its cache.

Test infrastructure: only the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may use it; the CUDA library never does.
"""

from .kl_oracle import fwd_bwd, student_lse, teacher_log_probs  # noqa: F401
from .topk_oracle import order_keys, topk_rows  # noqa: F401
