"""The offline top-K cache builder against the float64 oracle (GPU).

Exactness: with small-integer bf16 inputs every logit is an integer that
fp32 accumulates exactly, so ids and values must equal the oracle's bit for
bit -- including the tie order (lower id first) when many logits are equal.
These cases drive both selection paths: the one-pass filter behind the
per-tile-maximum threshold, and the exact radix select (K above the tile
count, or more candidates than shared memory holds).  On realistic inputs
(GPT-OSS-like head, full vocabulary) the fp32 logits must match the float64
ones closely and the returned set must be a valid top-K of them.
"""
import numpy as np
import pytest
import torch

import chunked_top_kl_gemm_b300 as kd
import oracle
import workloads
from tests.gpu_util import ensure_lib

pytestmark = pytest.mark.gpu


def _int_inputs(N, H, V, lo, hi, seed):
    g = torch.Generator().manual_seed(seed)
    h = torch.randint(lo, hi + 1, (N, H), generator=g).to(torch.bfloat16)
    W = torch.randint(lo, hi + 1, (V, H), generator=g).to(torch.bfloat16)
    return h, W


def _build(h, W, K, chunk):
    idx, val = kd.kd_topk_cache_build(h.cuda(), W.cuda(), K, chunk)
    torch.cuda.synchronize()
    return idx.cpu().numpy(), val.cpu().numpy()


@pytest.mark.parametrize("N,H,V,K,chunk", [
    (300, 64, 1000, 7, 128),      # 4 vocab tiles < K: every value a candidate, one sort
    (300, 64, 9000, 40, 128),     # 36 tiles < K and 9000 values: exact radix-select path
    (300, 64, 8192, 16, 128),     # threshold path, 32 tiles, ragged chunk
    (130, 48, 8200, 100, 256),    # ragged last vocab tile (8 columns)
    (64, 32, 2048, 2048, 64),     # K = V: a full sort per row
])
def test_exact_on_integer_logits(N, H, V, K, chunk):
    ensure_lib()
    h, W = _int_inputs(N, H, V, -2, 2, seed=N + V + K)
    want = oracle.topk_cache(h, W, K)
    idx, val = _build(h, W, K, chunk)
    assert np.array_equal(idx, want["topk_idx"])
    assert np.array_equal(val.astype(np.float64), want["topk_logit"])


@pytest.mark.parametrize("K", [50, 100])
def test_all_equal_logits_overflow_the_filter_and_keep_id_order(K):
    # every logit equal: all 16384 values pass the threshold (K = 50 <= 64
    # tiles) or there is none (K = 100), more than shared memory holds, so the
    # exact path runs and ties resolve to ids 0..K-1
    ensure_lib()
    N, H, V = 20, 16, 16384
    h = torch.ones((N, H), dtype=torch.bfloat16)
    W = torch.ones((V, H), dtype=torch.bfloat16)
    idx, val = _build(h, W, K, 128)
    assert (idx == np.arange(K)).all()
    assert (val == 16.0).all()


def test_many_ties_across_the_k_boundary():
    ensure_lib()
    N, H, V, K = 40, 8, 12000, 100
    h, W = _int_inputs(N, H, V, 0, 1, seed=9)    # logits in 0..8: heavy ties everywhere
    want = oracle.topk_cache(h, W, K)
    idx, val = _build(h, W, K, 128)
    assert np.array_equal(idx, want["topk_idx"])
    assert np.array_equal(val.astype(np.float64), want["topk_logit"])


def test_realistic_head_full_vocabulary():
    """256 tokens through a GPT-OSS-like head (H=2880, V=201,088), K = 100."""
    ensure_lib()
    cfg = workloads.CONFIGS["gptoss32k"]
    inp = workloads.make_inputs(cfg, seed=12, n_rows=256)
    h, W = inp["hidden"], inp["W"]
    K = 100
    idx, val = _build(h, W, K, 2048)
    Z = h.double().numpy() @ W.double().numpy().T
    want = oracle.topk_rows(Z, K)
    tol = 1e-5 * np.abs(Z).max()
    for n in range(Z.shape[0]):
        ids = idx[n]
        assert len(set(ids.tolist())) == K
        assert (np.diff(val[n]) <= 0).all()
        assert np.abs(val[n] - Z[n, ids]).max() <= tol
        rest = np.ones(Z.shape[1], dtype=bool)
        rest[ids] = False
        # a valid top-K of the float64 logits up to the fp32 rounding
        assert Z[n, ids].min() >= Z[n, rest].max() - 2 * tol
    agree = np.mean([len(set(idx[n]) & set(want[0][n])) / K for n in range(Z.shape[0])])
    assert agree > 0.999


def test_chunk_of_more_than_65535_rows():
    """One 70,016-row chunk: the streaming filter covers more rows than a
    grid's y dimension could hold.  Integer logits, so sampled rows must
    equal the oracle's bit for bit."""
    ensure_lib()
    N, H, V, K = 70000, 32, 512, 8
    h, W = _int_inputs(N, H, V, -2, 2, seed=17)
    idx, val = _build(h, W, K, 70000)
    rows = np.array([0, 1, 65534, 65535, 65536, 69998, 69999])
    want = oracle.topk_cache(h[rows], W, K)
    assert np.array_equal(idx[rows], want["topk_idx"])
    assert np.array_equal(val[rows].astype(np.float64), want["topk_logit"])


def test_cache_feeds_the_loss():
    """Build a cache from a teacher head, then run the loss against it."""
    ensure_lib()
    cfg = workloads.custom("cache_loss", N=384, H=256, V=4096, K=32, T=1.0, chunk=128)
    g = torch.Generator().manual_seed(3)
    h_t = torch.randn((cfg.N, cfg.H), generator=g).to(torch.bfloat16).cuda()
    W_t = (torch.randn((cfg.V, cfg.H), generator=g) * 0.05).to(torch.bfloat16).cuda()
    idx, lg = kd.kd_topk_cache_build(h_t, W_t, cfg.K, 128)
    student = workloads.make_inputs(cfg, seed=4, device="cuda")
    loss, gh, gW = kd.fwd_bwd(student["hidden"], student["W"], idx, lg, cfg.T, cfg.chunk)
    torch.cuda.synchronize()
    want = oracle.fused_topk_kl(student["hidden"].cpu(), student["W"].cpu(), idx.cpu(),
                                lg.cpu(), cfg.T)
    assert abs(loss - want["loss"]) <= 1e-3 * abs(want["loss"])


def test_bad_arguments():
    ensure_lib()
    assert kd.kd_topk_cache_workspace_size(16, 64, 128, 0, 64) == 0
    assert kd.kd_topk_cache_workspace_size(16, 64, 128, 129, 64) == 0
    assert kd.kd_topk_cache_workspace_size(16, 60, 128, 4, 64) == 0
    h = torch.zeros((16, 64), dtype=torch.bfloat16, device="cuda")
    W = torch.zeros((128, 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(kd.KdError):
        kd.kd_topk_cache_build(h, W, 200, 64)
