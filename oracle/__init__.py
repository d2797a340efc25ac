"""CPU oracle for the fused chunked top-K KL loss. TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py`` (its CPU
baseline and reference legs) may import this package.  The product path
(``chunked_top_kl_gemm_b300``) never imports it and shares no code with it.

It is a plain, slow, dense float64 implementation in numpy that materialises
the full [tokens x vocab] logit matrix (per row block).  See ``kl_topk.py``.
"""
from .kl_topk import (  # noqa: F401
    teacher_log_probs,
    student_lse,
    fused_topk_kl,
    rows_forward,
    grad_W_rows,
    to_f64,
)
from .topk_cache import topk_cache, topk_rows  # noqa: F401
