"""Plant plausible mistakes in copies of the oracle; some pin must fail.

Every mutant below changes one thing in the oracle's per-block arithmetic
(a dropped term, a wrong sign, index or factor, a transposed operand).  The
test passes when at least one pin from ``oracle_pins`` rejects the mutant,
which shows the pins would catch that kind of mistake in the oracle itself.
Mistakes are planted only here, in the oracle, on the CPU.
"""
import numpy as np
import pytest

import oracle
from oracle import kl_topk
from tests import oracle_pins as pins


def _terms(h_blk, W, idx_blk, logit_blk, T, N, *, mut):
    Z = h_blk @ W.T
    if mut == "transposed_head":
        Z = (h_blk @ W.T) if W.shape[0] != W.shape[1] else h_blk @ W
        Z = Z[:, ::-1]
    lse = kl_topk.student_lse(Z, T)
    lg = logit_blk if mut != "teacher_no_T" else logit_blk * T
    lp, p = kl_topk.teacher_log_probs(lg, T)
    rows = np.arange(Z.shape[0])[:, None]
    gidx = idx_blk if mut != "gather_off_by_one" else (idx_blk + 1) % W.shape[0]
    zg = Z[rows, gidx]
    log_q = zg / T - (lse[:, None] if mut != "drop_lse" else 0.0)
    if mut == "drop_entropy":
        loss_rows = (p * (-log_q)).sum(axis=1)
    else:
        loss_rows = (p * (lp - log_q)).sum(axis=1)
    Q = np.exp(Z / T - lse[:, None])
    P = np.zeros_like(Z)
    np.add.at(P, (np.broadcast_to(rows, idx_blk.shape), idx_blk), p)
    sign = -1.0 if mut == "wrong_sign" else 1.0
    scale = T * N * (T if mut == "extra_T" else 1.0)
    D = (Q - sign * P) / scale
    if mut == "set_not_add":
        P2 = np.zeros_like(Z)
        P2[np.broadcast_to(rows, idx_blk.shape), idx_blk] = p
        D = (Q - P2) / (T * N)
    return Z, lse, zg, loss_rows, D


MUTANTS = ["drop_lse", "drop_entropy", "teacher_no_T", "gather_off_by_one",
           "wrong_sign", "extra_T", "set_not_add", "transposed_head"]


@pytest.mark.parametrize("mut", MUTANTS)
def test_some_pin_rejects_mutant(mut, monkeypatch):
    monkeypatch.setattr(kl_topk, "_block_terms",
                        lambda *a: _terms(*a, mut=mut))

    def impl(h, W, idx, lg, T):
        return oracle.fused_topk_kl(h, W, idx, lg, T)

    caught = []
    checks = [(p, T) for p in pins.ALL_PINS for T in (1.0, 2.0)]
    checks.append((lambda f, T: pins.pin_finite_differences(f, T, dup=True), 1.5))
    for pin, T in checks:
        try:
            pin(impl, T)
        except (AssertionError, IndexError, ValueError):
            caught.append(getattr(pin, "__name__", "fd_dup"))
    assert caught, f"no pin rejects mutant {mut}"


def test_mask_mean_over_all_tokens_is_rejected(monkeypatch):
    # planted mistake: the masked mean divides by N instead of the number of
    # valid tokens (and scales dZ the same way)
    real = kl_topk.fused_topk_kl

    def wrong(h, W, idx, lg, T, chunk_rows=None, mask=None):
        out = real(h, W, idx, lg, T, chunk_rows=chunk_rows, mask=mask)
        n = np.asarray(h).shape[0]
        if mask is not None and out["n_valid"]:
            f = out["n_valid"] / n
            out = dict(out, loss=out["loss"] * f, grad_hidden=out["grad_hidden"] * f,
                       grad_W=out["grad_W"] * f)
        return out

    caught = []
    for pin in pins.MASK_PINS:
        try:
            pin(lambda h, W, i, l, T, m: wrong(h, W, i, l, T, mask=m), 1.0)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught


def test_mask_dropped_is_rejected():
    # planted mistake: the mask is ignored
    caught = []
    for pin in pins.MASK_PINS:
        try:
            pin(lambda h, W, i, l, T, m: oracle.fused_topk_kl(h, W, i, l, T), 1.0)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught


def test_unmutated_oracle_passes_every_pin():
    for pin in pins.ALL_PINS:
        pin(lambda h, W, i, l, T: oracle.fused_topk_kl(h, W, i, l, T), 1.0)
