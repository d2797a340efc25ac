"""Checks that pin the oracle to facts outside itself.

Each ``pin_*`` function takes an implementation ``impl(hidden, W, idx,
logit, T) -> dict`` with the oracle's output keys and raises AssertionError
when the implementation disagrees with the fact the pin encodes.  The
oracle tests run every pin on the oracle; the mutant tests plant a mistake
in a copy of the oracle and check that some pin catches it.

What each pin rests on:

* ``pin_finite_differences`` -- calculus: the gradients are the derivatives
  of the loss (central differences in float64, every entry).
* ``pin_uniform_head``       -- closed form: with every row of W equal the
  student is uniform, q = 1/V, so loss = log V - mean entropy(p),
  grad_hidden = 0 and grad_W has a closed form.
* ``pin_cross_entropy``      -- textbook reduction: with K = 1 the teacher is
  one-hot and the loss is softmax cross-entropy of z/T (torch's
  ``cross_entropy`` and autograd, float64, as the independent routine).
* ``pin_library_kl``         -- library reduction of the general case: torch
  ``log_softmax`` + ``gather`` + ``kl_div`` + autograd in float64.
* ``pin_self_distillation``  -- K = V and teacher logits equal to the
  student's: KL is zero and so are both gradients.
* ``pin_two_token_vocab``    -- a hand-derived case (V = 2, H = 1, K = 1).
* ``pin_nonnegative``        -- Gibbs' inequality: loss >= 0 for distinct ids.
* ``pin_invariants``         -- sum over v of grad_W[v] = 0 (softmax minus a
  distribution sums to zero), and adding one vector u to every row of W
  changes neither the loss nor the gradients.
"""
from __future__ import annotations

import math

import numpy as np
import torch


def _rng(seed):
    return np.random.default_rng(seed)


def _distinct(rng, n, k, v):
    return np.stack([rng.choice(v, size=k, replace=False) for _ in range(n)])


def small_case(seed=0, N=6, H=8, V=40, K=4, w_std=0.3, dup=False):
    rng = _rng(seed)
    h = rng.normal(size=(N, H))
    W = rng.normal(scale=w_std, size=(V, H))
    idx = _distinct(rng, N, K, V)
    if dup:
        idx[0, 1] = idx[0, 0]   # one repeated id in row 0
    lg = np.sort(rng.normal(scale=2.0, size=(N, K)), axis=1)[:, ::-1].copy()
    return h, W, idx, lg


def pin_finite_differences(impl, T, seed=0, dup=False, eps=1e-6, tol=1e-6):
    h, W, idx, lg = small_case(seed, dup=dup)
    out = impl(h, W, idx, lg, T)

    def loss_at(hh, WW):
        return impl(hh, WW, idx, lg, T)["loss"]

    for name, X, G in (("hidden", h, out["grad_hidden"]), ("W", W, out["grad_W"])):
        fd = np.empty_like(X)
        for i in np.ndindex(X.shape):
            Xp = X.copy(); Xp[i] += eps
            Xm = X.copy(); Xm[i] -= eps
            if name == "hidden":
                fd[i] = (loss_at(Xp, W) - loss_at(Xm, W)) / (2 * eps)
            else:
                fd[i] = (loss_at(h, Xp) - loss_at(h, Xm)) / (2 * eps)
        err = np.abs(fd - G).max() / max(np.abs(fd).max(), 1e-300)
        assert err <= tol, f"FD mismatch on {name}: rel {err:.3e}"


def pin_uniform_head(impl, T, seed=1, N=5, H=6, V=17, K=4):
    rng = _rng(seed)
    h = rng.normal(size=(N, H))
    w = rng.normal(size=(H,))
    W = np.tile(w, (V, 1))
    idx = _distinct(rng, N, K, V)
    lg = rng.normal(scale=3.0, size=(N, K))
    out = impl(h, W, idx, lg, T)
    a = lg / T
    e = np.exp(a - a.max(axis=1, keepdims=True))
    p = e / e.sum(axis=1, keepdims=True)
    entropy = -(p * np.log(p)).sum(axis=1)
    want_loss = math.log(V) - entropy.mean()
    assert abs(out["loss"] - want_loss) <= 1e-12 * max(1.0, abs(want_loss)), \
        (out["loss"], want_loss)
    assert np.abs(out["grad_hidden"]).max() <= 1e-13
    Pm = np.zeros((N, V))
    for n in range(N):
        for k in range(K):
            Pm[n, idx[n, k]] += p[n, k]
    want_gW = ((1.0 / V - Pm).T @ h) / (T * N)
    assert np.allclose(out["grad_W"], want_gW, rtol=0, atol=1e-13)


def _torch_loss(h, W, idx, lg, T, K1=False):
    ht = torch.tensor(h, dtype=torch.float64, requires_grad=True)
    Wt = torch.tensor(W, dtype=torch.float64, requires_grad=True)
    Z = ht @ Wt.T
    it = torch.tensor(np.asarray(idx), dtype=torch.int64)
    if K1:
        loss = torch.nn.functional.cross_entropy(Z / T, it[:, 0],
                                                 reduction="mean")
    else:
        logq = torch.log_softmax(Z / T, dim=1).gather(1, it)
        lp = torch.log_softmax(torch.tensor(lg, dtype=torch.float64) / T, dim=1)
        loss = torch.nn.functional.kl_div(logq, lp, log_target=True,
                                          reduction="sum") / h.shape[0]
    loss.backward()
    return float(loss.detach()), ht.grad.numpy(), Wt.grad.numpy()


def _assert_matches_torch(out, ref, tol=1e-12):
    loss, gh, gW = ref
    assert abs(out["loss"] - loss) <= tol * max(1.0, abs(loss)), (out["loss"], loss)
    for got, want in ((out["grad_hidden"], gh), (out["grad_W"], gW)):
        scale = max(np.abs(want).max(), 1e-300)
        assert np.abs(got - want).max() <= tol * scale


def pin_cross_entropy(impl, T, seed=2, N=7, H=5, V=23):
    rng = _rng(seed)
    h = rng.normal(size=(N, H))
    W = rng.normal(scale=0.5, size=(V, H))
    idx = rng.integers(0, V, size=(N, 1))
    lg = rng.normal(size=(N, 1))
    out = impl(h, W, idx, lg, T)
    _assert_matches_torch(out, _torch_loss(h, W, idx, lg, T, K1=True))


def pin_library_kl(impl, T, seed=3, N=9, H=7, V=31, K=5):
    rng = _rng(seed)
    h = rng.normal(size=(N, H))
    W = rng.normal(scale=0.5, size=(V, H))
    idx = _distinct(rng, N, K, V)
    lg = rng.normal(scale=2.0, size=(N, K))
    out = impl(h, W, idx, lg, T)
    _assert_matches_torch(out, _torch_loss(h, W, idx, lg, T))


def pin_self_distillation(impl, T, seed=4, N=4, H=6, V=12):
    rng = _rng(seed)
    h = rng.normal(size=(N, H))
    W = rng.normal(scale=0.7, size=(V, H))
    idx = np.stack([rng.permutation(V) for _ in range(N)])
    Z = h @ W.T
    lg = np.take_along_axis(Z, idx, axis=1)
    out = impl(h, W, idx, lg, T)
    assert abs(out["loss"]) <= 1e-13, out["loss"]
    assert np.abs(out["grad_hidden"]).max() <= 1e-14
    assert np.abs(out["grad_W"]).max() <= 1e-14


def pin_two_token_vocab(impl, T, a=0.3, b=-1.1, x=1.7):
    # one token, H = 1, V = 2, K = 1 with the cached id 0: KL = -log q_0.
    h = np.array([[x]])
    W = np.array([[a], [b]])
    idx = np.array([[0]])
    lg = np.array([[5.0]])
    out = impl(h, W, idx, lg, T)
    d = (b - a) * x / T
    q1 = 1.0 / (1.0 + math.exp(-d))
    assert abs(out["loss"] - math.log1p(math.exp(d))) <= 1e-14
    assert abs(out["grad_hidden"][0, 0] - q1 * (b - a) / T) <= 1e-14
    assert np.allclose(out["grad_W"][:, 0], [-q1 * x / T, q1 * x / T],
                       rtol=0, atol=1e-14)


def pin_nonnegative(impl, T, seeds=range(5)):
    for s in seeds:
        h, W, idx, lg = small_case(100 + s, N=8, H=6, V=30, K=6, w_std=2.0)
        assert impl(h, W, idx, lg, T)["loss"] >= -1e-15


def pin_invariants(impl, T, seed=5):
    h, W, idx, lg = small_case(seed, N=7, H=5, V=29, K=5)
    out = impl(h, W, idx, lg, T)
    assert np.abs(out["grad_W"].sum(axis=0)).max() <= 1e-14
    u = _rng(seed + 1).normal(size=(W.shape[1],))
    out2 = impl(h, W + u[None, :], idx, lg, T)
    assert abs(out2["loss"] - out["loss"]) <= 1e-12
    assert np.abs(out2["grad_hidden"] - out["grad_hidden"]).max() <= 1e-13
    assert np.abs(out2["grad_W"] - out["grad_W"]).max() <= 1e-13


ALL_PINS = (
    pin_finite_differences, pin_uniform_head, pin_cross_entropy,
    pin_library_kl, pin_self_distillation, pin_two_token_vocab,
    pin_nonnegative, pin_invariants,
)


# ---------------------------------------------------------------- token mask
# Pins of the masked loss take ``impl_m(hidden, W, idx, logit, T, mask)``.
#
# * ``pin_mask_subset``  -- the masked loss is the unmasked loss of the valid
#   tokens alone (the definition of "mean over the valid tokens"): the same
#   loss and grad_W, the same grad_hidden rows, zero rows for masked tokens;
#   an all-ones mask changes nothing; an all-zero mask gives zeros.
# * ``pin_mask_fd``      -- calculus: the masked gradients are the derivatives
#   of the masked loss (central differences, float64).
# * ``pin_mask_torch``   -- library reduction: torch log_softmax / kl_div with
#   the mask applied per token and autograd, float64.

def _mask_case(seed=7, N=8, H=5, V=26, K=4):
    h, W, idx, lg = small_case(seed, N=N, H=H, V=V, K=K)
    mask = (_rng(seed + 50).random(N) < 0.6).astype(np.uint8)
    mask[0], mask[1] = 1, 0
    return h, W, idx, lg, mask


def pin_mask_subset(impl_m, T):
    h, W, idx, lg, mask = _mask_case()
    out = impl_m(h, W, idx, lg, T, mask)
    keep = mask != 0
    sub = impl_m(h[keep], W, idx[keep], lg[keep], T, np.ones(int(keep.sum())))
    assert abs(out["loss"] - sub["loss"]) <= 1e-12 * max(1.0, abs(sub["loss"]))
    assert np.abs(out["grad_W"] - sub["grad_W"]).max() <= 1e-14
    assert np.abs(out["grad_hidden"][keep] - sub["grad_hidden"]).max() <= 1e-14
    assert np.abs(out["grad_hidden"][~keep]).max() == 0.0
    full = impl_m(h, W, idx, lg, T, np.ones(len(mask)))
    plain = impl_m(h, W, idx, lg, T, None)
    assert full["loss"] == plain["loss"]
    assert np.array_equal(full["grad_W"], plain["grad_W"])
    none = impl_m(h, W, idx, lg, T, np.zeros(len(mask)))
    assert none["loss"] == 0.0
    assert np.abs(none["grad_W"]).max() == 0.0 and np.abs(none["grad_hidden"]).max() == 0.0


def pin_mask_fd(impl_m, T, eps=1e-6, tol=1e-6):
    h, W, idx, lg, mask = _mask_case(N=6, H=4, V=15, K=3)
    out = impl_m(h, W, idx, lg, T, mask)
    for name, X, G in (("hidden", h, out["grad_hidden"]), ("W", W, out["grad_W"])):
        fd = np.empty_like(X)
        for i in np.ndindex(X.shape):
            Xp = X.copy(); Xp[i] += eps
            Xm = X.copy(); Xm[i] -= eps
            args_p = (Xp, W) if name == "hidden" else (h, Xp)
            args_m = (Xm, W) if name == "hidden" else (h, Xm)
            fd[i] = (impl_m(*args_p, idx, lg, T, mask)["loss"]
                     - impl_m(*args_m, idx, lg, T, mask)["loss"]) / (2 * eps)
        err = np.abs(fd - G).max() / max(np.abs(fd).max(), 1e-300)
        assert err <= tol, f"masked FD mismatch on {name}: rel {err:.3e}"


def pin_mask_torch(impl_m, T):
    h, W, idx, lg, mask = _mask_case(seed=9, N=10, H=6, V=21, K=5)
    out = impl_m(h, W, idx, lg, T, mask)
    ht = torch.tensor(h, dtype=torch.float64, requires_grad=True)
    Wt = torch.tensor(W, dtype=torch.float64, requires_grad=True)
    logq = torch.log_softmax((ht @ Wt.T) / T, dim=1).gather(
        1, torch.tensor(np.asarray(idx), dtype=torch.int64))
    lp = torch.log_softmax(torch.tensor(lg, dtype=torch.float64) / T, dim=1)
    per_tok = torch.nn.functional.kl_div(logq, lp, log_target=True,
                                         reduction="none").sum(dim=1)
    m = torch.tensor(mask, dtype=torch.float64)
    loss = (per_tok * m).sum() / m.sum()
    loss.backward()
    lv = float(loss.detach())
    assert abs(out["loss"] - lv) <= 1e-12 * max(1.0, abs(lv))
    for got, want in ((out["grad_hidden"], ht.grad.numpy()), (out["grad_W"], Wt.grad.numpy())):
        assert np.abs(got - want).max() <= 1e-12 * max(np.abs(want).max(), 1e-300)


MASK_PINS = (pin_mask_subset, pin_mask_fd, pin_mask_torch)
