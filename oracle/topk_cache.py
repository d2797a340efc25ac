"""Dense float64 oracle of the offline top-K teacher cache.  TEST INFRASTRUCTURE ONLY.

The method caches, per token position, the teacher's K highest logits and
their token ids, computed once offline (epoka.news, "The two proposed
changes"; glonce.com, body; ainewsbank.com, "Two changes remove different
bottlenecks": K = 100).  The pages do not say how ties are broken; this
build reads it as "lower token id first" (a stable order of the vocabulary).

    z_n       = W h_n                      (teacher LM head, no bias)
    topk_n    = the K ids v with the largest z_nv, in decreasing z_nv,
                equal logits ordered by increasing id
    logit_nk  = z_{n, topk_nk}
"""
from __future__ import annotations

import numpy as np

from .kl_topk import to_f64


def topk_rows(Z: np.ndarray, K: int):
    """Top-K ids and values of every row of Z (decreasing value, ties by
    increasing id).  Returns (idx [N,K] int64, val [N,K] float64)."""
    Z = np.asarray(Z, dtype=np.float64)
    N, V = Z.shape
    ids = np.broadcast_to(np.arange(V), (N, V))
    # lexsort: the last key is the primary one
    order = np.lexsort((ids, -Z), axis=1)[:, :K]
    return order.astype(np.int64), np.take_along_axis(Z, order, axis=1)


def topk_cache(hidden, W, K: int, chunk_rows: int | None = None) -> dict:
    """Teacher cache of the hidden states ``hidden`` [N,H] through the head
    ``W`` [V,H], with the logits in float64 (bf16 inputs upcast exactly)."""
    h = to_f64(hidden)
    Wd = to_f64(W)
    N = h.shape[0]
    V = Wd.shape[0]
    if chunk_rows is None:
        chunk_rows = max(1, min(N, (1 << 27) // max(V, 1)))
    idx = np.empty((N, K), dtype=np.int64)
    val = np.empty((N, K))
    for r0 in range(0, N, chunk_rows):
        r1 = min(N, r0 + chunk_rows)
        idx[r0:r1], val[r0:r1] = topk_rows(h[r0:r1] @ Wd.T, K)
    return {"topk_idx": idx, "topk_logit": val}
