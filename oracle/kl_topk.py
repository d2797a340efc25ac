"""Dense float64 oracle of the top-K KL distillation loss and its gradients.

TEST INFRASTRUCTURE ONLY: imported by tests, the smoke check and the
benchmark's CPU baseline, never by the product path.

What is computed
----------------
The pages describe the method but do not print its formula:

* offline top-K caching keeps, per token position, the teacher's K highest
  logits and their token ids (epoka.news, "The two proposed changes";
  ainewsbank.com, "Two changes remove different bottlenecks", which puts K
  at 100);
* the fused chunked loss works through the token positions chunk by chunk:
  a chunk's logits are formed, reduced into the running loss and dropped,
  then formed again for the gradients rather than kept (glonce.com, body,
  the paragraph on Multiverse's fix); the chunked form computes the same
  numbers as the plain one (ainewsbank.com, "Two changes remove different
  bottlenecks").

Because chunking and recomputation leave the result unchanged, this oracle
is the plain dense definition, with one row block at a time only to bound
host memory.  The loss is the standard truncated-teacher KL (the pages call
the gradient "closed-form" without printing it, glonce.com, "How to use
it"):

    z_n      = W h_n                              (LM head, no bias)
    log p_nk = l_nk/T - logsumexp_k(l_n/T)        (teacher over its K entries)
    log q_nv = z_nv/T - logsumexp_v(z_n/T)        (student over all V)
    loss     = (1/N) sum_n sum_k p_nk (log p_nk - log q_{n, idx_nk})
    dZ_nv    = (q_nv - sum_{k: idx_nk = v} p_nk) / (T N)
    grad_hidden = dZ W,   grad_W = dZ^T hidden

Readings where the pages are silent: no T^2 factor, mean over all N tokens,
no bias, the teacher's tail mass beyond K is dropped and p renormalised over
the K entries, repeated ids add up (scatter-add) in dZ and give one loss term
each.

Token mask.  The pages mention sequence-packing ablations (glonce.com, body
and "How to use it") without detail; a real training step also pads.  With
an optional per-token mask the loss is the mean over the N_v tokens whose
mask is set, and masked tokens contribute nothing:

    loss = (1/N_v) sum_{n: mask_n} sum_k p_nk (log p_nk - log q_{n, idx_nk})
    dZ_n = mask_n (q_n - scatter(p_n)) / (T N_v)

i.e. exactly the unmasked definition applied to the valid tokens alone (a
test checks that reading).  With N_v = 0 the loss and the gradients are 0.
"""
from __future__ import annotations

import numpy as np


def to_f64(x) -> np.ndarray:
    """Exact upcast of a torch tensor (bf16 / fp32 / int) or array to numpy.

    bf16 and fp32 values are exactly representable in float64, so this
    introduces no rounding.  Integer arrays are returned as int64.
    """
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().cpu()
            if x.dtype in (torch.int32, torch.int64, torch.int16):
                return x.to(torch.int64).numpy()
            return x.to(torch.float64).numpy()
    except ImportError:  # pragma: no cover
        pass
    a = np.asarray(x)
    if np.issubdtype(a.dtype, np.integer):
        return np.asarray(a, dtype=np.int64)
    return np.asarray(a, dtype=np.float64)   # no copy when already float64


def _logsumexp_rows(a: np.ndarray) -> np.ndarray:
    """logsumexp over axis 1, shifted by the row maximum."""
    m = a.max(axis=1, keepdims=True)
    return (m + np.log(np.exp(a - m).sum(axis=1, keepdims=True)))[:, 0]


def teacher_log_probs(topk_logit: np.ndarray, T: float):
    """Teacher log p and p over the K cached entries (log-softmax of l/T).

    Follows the top-K cache description (epoka.news, "The two proposed
    changes"): the cache holds only the K highest teacher logits, so the
    teacher distribution used by the loss is the softmax over those K.
    Returns (log_p [N,K], p [N,K]).
    """
    a = np.asarray(topk_logit, dtype=np.float64) / T
    lp = a - _logsumexp_rows(a)[:, None]
    return lp, np.exp(lp)


def student_lse(Z: np.ndarray, T: float) -> np.ndarray:
    """logsumexp_v(z_nv / T) over the full vocabulary, per row."""
    return _logsumexp_rows(np.asarray(Z, dtype=np.float64) / T)


def _block_terms(h_blk, W, idx_blk, logit_blk, T, N):
    """Dense logits and per-row quantities for one row block.

    Returns (Z, lse, zg, loss_rows, D) where D = dZ for the block, already
    divided by T*N (N: the number of tokens the mean runs over).
    """
    Z = h_blk @ W.T                                   # [b, V]
    lse = student_lse(Z, T)                           # [b]
    lp, p = teacher_log_probs(logit_blk, T)           # [b, K]
    rows = np.arange(Z.shape[0])[:, None]
    zg = Z[rows, idx_blk]                             # [b, K] gather
    log_q_idx = zg / T - lse[:, None]
    loss_rows = (p * (lp - log_q_idx)).sum(axis=1)    # [b]
    Q = np.exp(Z / T - lse[:, None])                  # student softmax
    P = np.zeros_like(Z)
    np.add.at(P, (np.broadcast_to(rows, idx_blk.shape), idx_blk), p)
    D = (Q - P) / (T * N)
    return Z, lse, zg, loss_rows, D


def fused_topk_kl(hidden, W, topk_idx, topk_logit, T: float,
                  chunk_rows: int | None = None, mask=None) -> dict:
    """Loss and gradients of the top-K KL loss over all N tokens.

    ``chunk_rows`` only bounds host memory (the result does not depend on
    it; a test checks that).  Inputs may be torch tensors or arrays; all
    arithmetic is float64.  ``mask`` (optional, [N], nonzero = the token
    counts) restricts the mean to the valid tokens; masked tokens get zero
    loss terms and zero gradient rows.

    Returns a dict with
      loss         float, mean over the N tokens
      loss_rows    [N]   per-token sum_k p (log p - log q_idx)
      lse          [N]   logsumexp_v(z/T)
      zg           [N,K] student logits z at the cached ids
      grad_hidden  [N,H]
      grad_W       [V,H]
    """
    h = to_f64(hidden)
    Wd = to_f64(W)
    idx = to_f64(topk_idx)
    lg = to_f64(topk_logit)
    N, H = h.shape
    V = Wd.shape[0]
    valid = np.ones(N, dtype=bool) if mask is None else (to_f64(mask) != 0)
    n_valid = int(valid.sum())
    if chunk_rows is None:
        chunk_rows = max(1, min(N, (1 << 28) // max(V, 1)))
    out_lse = np.empty(N)
    out_zg = np.empty(idx.shape)
    out_loss_rows = np.empty(N)
    gh = np.empty((N, H))
    gW = np.zeros((V, H))
    for r0 in range(0, N, chunk_rows):
        r1 = min(N, r0 + chunk_rows)
        _, lse, zg, lrow, D = _block_terms(h[r0:r1], Wd, idx[r0:r1],
                                           lg[r0:r1], T, max(n_valid, 1))
        keep = valid[r0:r1]
        lrow = np.where(keep, lrow, 0.0)
        D = D * keep[:, None]
        out_lse[r0:r1] = lse
        out_zg[r0:r1] = zg
        out_loss_rows[r0:r1] = lrow
        gh[r0:r1] = D @ Wd
        gW += D.T @ h[r0:r1]
    return {
        "loss": float(out_loss_rows.sum() / n_valid) if n_valid else 0.0,
        "n_valid": n_valid,
        "loss_rows": out_loss_rows,
        "lse": out_lse,
        "zg": out_zg,
        "grad_hidden": gh,
        "grad_W": gW,
    }


def rows_forward(hidden_rows, W, idx_rows, logit_rows, T: float,
                 N_total: int, vrows=None, grad_hidden: bool = True) -> dict:
    """Per-token quantities for a subset of token rows.

    Every per-token output (its loss term, lse, gathered logits and its row
    of grad_hidden) depends only on that token's inputs and W, so a sample
    of rows can be checked at any N.  ``N_total`` is the token count of the
    full problem (the mean's denominator).

    With ``vrows`` (vocabulary ids) the result also holds ``grad_W_rows``:
    these tokens' share sum_n dZ_nv h_n of grad_W rows ``vrows``.  grad_W
    is a sum over tokens, so the shares of disjoint token blocks add up to
    the rows of the full problem's grad_W.  ``grad_hidden=False`` skips
    the grad_hidden product (half the work of a block).
    """
    h = to_f64(hidden_rows)
    Wd = to_f64(W)
    idx = to_f64(idx_rows)
    lg = to_f64(logit_rows)
    _, lse, zg, lrow, D = _block_terms(h, Wd, idx, lg, T, N_total)
    out = {"lse": lse, "zg": zg, "loss_rows": lrow}
    if grad_hidden:
        out["grad_hidden"] = D @ Wd
    if vrows is not None:
        out["grad_W_rows"] = D[:, np.asarray(vrows, dtype=np.int64)].T @ h
    return out


def grad_W_rows(hidden, W, topk_idx, topk_logit, T: float, vrows,
                chunk_rows: int = 4096) -> np.ndarray:
    """Rows ``vrows`` of grad_W, using every token.

    grad_W[v] = sum_n dZ_nv h_n needs each token's full-vocabulary
    normaliser, so every token's full logit row is formed (in row blocks);
    only the requested vocab rows of dZ are kept.
    """
    h = to_f64(hidden)
    Wd = to_f64(W)
    idx = to_f64(topk_idx)
    lg = to_f64(topk_logit)
    vrows = np.asarray(vrows, dtype=np.int64)
    N = h.shape[0]
    out = np.zeros((len(vrows), h.shape[1]))
    for r0 in range(0, N, chunk_rows):
        r1 = min(N, r0 + chunk_rows)
        hb = h[r0:r1]
        Z = hb @ Wd.T
        lse = student_lse(Z, T)
        _, p = teacher_log_probs(lg[r0:r1], T)
        Qs = np.exp(Z[:, vrows] / T - lse[:, None])           # [b, |vrows|]
        Ps = np.zeros_like(Qs)
        for j, v in enumerate(vrows):
            Ps[:, j] = (p * (idx[r0:r1] == v)).sum(axis=1)
        out += ((Qs - Ps) / (T * N)).T @ hb
    return out
