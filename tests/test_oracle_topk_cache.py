"""The top-K cache oracle against facts outside itself (CPU only).

* brute force: Python's own sort of (-z, id) pairs on tiny inputs;
* a closed form: with H = V and W = I the logits are the hidden entries;
* ties: equal logits come out in increasing id order (all-equal rows give
  ids 0..K-1); K = V returns a full permutation sorted by value.
A planted mistake (ties by decreasing id, or an ascending sort) is rejected.
"""
import numpy as np
import pytest

import oracle


def _brute(Z, K):
    out_i, out_v = [], []
    for row in Z:
        pairs = sorted(((-float(z), v) for v, z in enumerate(row)))[:K]
        out_i.append([v for _, v in pairs])
        out_v.append([-nz for nz, _ in pairs])
    return np.array(out_i), np.array(out_v)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_matches_brute_force(seed):
    rng = np.random.default_rng(seed)
    h = rng.normal(size=(7, 5))
    W = np.round(rng.normal(size=(40, 5)) * 4) / 4     # some exactly equal logits
    W[3] = W[11]                                        # a guaranteed tie
    out = oracle.topk_cache(h, W, 9)
    bi, bv = _brute(h @ W.T, 9)
    assert np.array_equal(out["topk_idx"], bi)
    assert np.array_equal(out["topk_logit"], bv)


def test_identity_head_closed_form():
    rng = np.random.default_rng(4)
    h = rng.normal(size=(6, 12))
    out = oracle.topk_cache(h, np.eye(12), 4)
    for n in range(6):
        want = sorted(range(12), key=lambda v: (-h[n, v], v))[:4]
        assert list(out["topk_idx"][n]) == want
        assert np.array_equal(out["topk_logit"][n], h[n, want])


def test_ties_go_to_the_lower_id_and_k_equals_v():
    h = np.ones((3, 4))
    W = np.ones((10, 4))
    out = oracle.topk_cache(h, W, 5)
    assert (out["topk_idx"] == np.arange(5)).all()
    rng = np.random.default_rng(5)
    h2 = rng.normal(size=(2, 3))
    W2 = rng.normal(size=(8, 3))
    full = oracle.topk_cache(h2, W2, 8)
    for n in range(2):
        assert sorted(full["topk_idx"][n]) == list(range(8))
        assert (np.diff(full["topk_logit"][n]) <= 0).all()


def test_planted_mistakes_are_rejected(monkeypatch):
    import importlib
    tc = importlib.import_module("oracle.topk_cache")
    h = np.ones((2, 3))
    W = np.ones((6, 3))
    W[4] *= 2
    real = tc.topk_rows

    def desc_id_ties(Z, K):
        Z = np.asarray(Z, dtype=np.float64)
        ids = np.broadcast_to(np.arange(Z.shape[1]), Z.shape)
        order = np.lexsort((-ids, -Z), axis=1)[:, :K]
        return order, np.take_along_axis(Z, order, axis=1)

    def ascending(Z, K):
        i, v = real(-np.asarray(Z), K)
        return i, -v

    for wrong in (desc_id_ties, ascending):
        monkeypatch.setattr(tc, "topk_rows", wrong)
        out = oracle.topk_cache(h, W, 3)
        assert list(out["topk_idx"][0]) != [4, 0, 1]
    monkeypatch.setattr(tc, "topk_rows", real)
    assert list(oracle.topk_cache(h, W, 3)["topk_idx"][0]) == [4, 0, 1]
