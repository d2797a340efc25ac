"""The CUDA path at the workloads' full sizes, in the benchmark's launch configuration.

Each workload (llama3b, gptoss32k, long64k, ext256k) runs whole on the GPU
with its own chunk size, exactly as ``bench.py`` times it.  The float64
oracle cannot redo a full call in seconds, so the checks are:

* every gathered id on every row equals the cached id (bit-exact);
* lse, gathered z, the per-token loss terms and grad_hidden of sampled
  tokens against the oracle's ``rows_forward`` (each token's outputs depend
  only on its own inputs and W);
* the loss is the mean of the per-token terms;
* grad_W through properties that hold at any size: its rows sum to zero
  (softmax minus a distribution sums to zero over the vocabulary), and
  <grad_W, W> = <grad_hidden, hidden>, both being sum_{n,v} dZ_nv z_nv;
* a 256-token run at full H and V whose sampled grad_W rows (and all other
  outputs) are compared with the oracle in full.

Inputs are drawn on the GPU with the workload's recipe; the oracle reads
the same bf16 / int32 / fp32 values copied back to the host.
"""
import numpy as np
import pytest
import torch

import chunked_top_kl_gemm_b300 as kd
import oracle
import workloads
from tests.gpu_util import (GRAD_REL_L2, LOSS_RTOL, LSE_ATOL, ZG_RTOL, assert_parity,
                            ensure_lib, rel_l2, run_debug, to_device)

pytestmark = pytest.mark.gpu

N_SAMPLES = 40


def _sample_rows(cfg, lg):
    """Evenly spaced tokens, both ends, both sides of every chunk boundary,
    and (when the workload has them) near-one-hot teacher rows."""
    N, c = cfg.N, cfg.chunk
    rows = set(np.linspace(0, N - 1, N_SAMPLES // 2).astype(np.int64).tolist())
    for b in (c, (N // c // 2) * c, N - c):
        rows.update({b - 1, b})
    rows.update({0, N - 1})
    if cfg.spike_frac > 0:
        spiky = torch.nonzero(lg[:, 0] > lg[:, 1] + 10).flatten()[:8].cpu().numpy()
        rows.update(int(r) for r in spiky)
    return np.array(sorted(r for r in rows if 0 <= r < N), dtype=np.int64)


@pytest.mark.parametrize("name", ["llama3b", "gptoss32k", "long64k", "ext256k"])
def test_full_size_sampled_parity(name):
    ensure_lib()
    cfg = workloads.CONFIGS[name]
    N, H, V, K, T = cfg.N, cfg.H, cfg.V, cfg.K, cfg.T
    dev = torch.device("cuda")
    inp = workloads.make_inputs(cfg, seed=0, device=dev)
    h, W, idx, lg = inp["hidden"], inp["W"], inp["topk_idx"], inp["topk_logit"]
    gh = torch.empty((N, H), dtype=torch.float32, device=dev)
    gW = torch.empty((V, H), dtype=torch.float32, device=dev)
    ws = kd.alloc_workspace(N, H, V, K, cfg.chunk, device=dev)
    lse = torch.empty((N,), dtype=torch.float32, device=dev)
    zg = torch.empty((N, K), dtype=torch.float32, device=dev)
    found = torch.full((N, K), -1, dtype=torch.int32, device=dev)
    loss_rows = torch.empty((N,), dtype=torch.float64, device=dev)
    loss = kd.kd_topk_kl_debug(h, W, idx, lg, T, cfg.chunk, gh, gW, ws, lse=lse, zg=zg,
                               found_idx=found, loss_rows=loss_rows)
    torch.cuda.synchronize()
    del ws

    # gathered ids: bit-exact on every row
    assert torch.equal(found, idx), "a cached id was gathered from the wrong column"

    # the loss is the mean of the per-token terms (double sum, fp32 result)
    mean_rows = float(loss_rows.sum().item()) / N
    assert abs(loss - mean_rows) <= 1e-6 * abs(mean_rows), (loss, mean_rows)
    assert torch.isfinite(gh).all() and torch.isfinite(gW).all()

    # sampled tokens against the oracle
    rows = _sample_rows(cfg, lg)
    rt = torch.from_numpy(rows).to(dev)
    W_cpu = W.cpu()
    want = oracle.rows_forward(h[rt].cpu(), W_cpu, idx[rt].cpu(), lg[rt].cpu(), T, N_total=N)
    np.testing.assert_allclose(lse[rt].cpu().numpy(), want["lse"], rtol=0, atol=LSE_ATOL)
    zscale = max(np.abs(want["zg"]).max(), 1e-6)
    assert np.abs(zg[rt].cpu().numpy() - want["zg"]).max() <= ZG_RTOL * zscale
    np.testing.assert_allclose(loss_rows[rt].cpu().numpy(), want["loss_rows"],
                               rtol=LOSS_RTOL, atol=1e-6)
    err = rel_l2(gh[rt].cpu().numpy(), want["grad_hidden"])
    assert err <= GRAD_REL_L2, err

    # grad_W: its vocabulary rows sum to zero, relative to the size of one
    # row-sum's terms (|dZ| summed over v is at most 2/(T N) per token)
    col = gW.double().sum(dim=0)
    scale = (h.double().abs().sum(dim=0) * (2.0 / (T * N)))
    assert float((col.abs() / scale).max()) <= 1e-3

    # grad_W: <grad_W, W> = <grad_hidden, hidden>
    a = float((gW.double() * W.double()).sum())
    b = float((gh.double() * h.double()).sum())
    mag = float((gh.double() * h.double()).abs().sum())
    assert abs(a - b) <= 1e-3 * mag, (a, b, mag)
    # and the identity is not vacuous: its value is a sizeable part of the scale
    assert abs(b) >= 1e-2 * mag


def test_full_vocab_head_grad_W_rows():
    """256 tokens of the GPT-OSS-like head (H=2880, V=201,088, chunk 2048):
    every output against the oracle, grad_W on sampled vocabulary rows
    (teacher-hit rows, the last rows of the ragged last vocab tile, random
    rows)."""
    ensure_lib()
    base = workloads.CONFIGS["gptoss32k"]
    inp = workloads.make_inputs(base, seed=4, n_rows=256)
    got = run_debug(to_device(inp), base.T, base.chunk)
    want = oracle.fused_topk_kl(inp["hidden"], inp["W"], inp["topk_idx"], inp["topk_logit"],
                                base.T)
    assert_parity(got, want, inp["topk_idx"].numpy(), check_grads=False)
    assert rel_l2(got["grad_hidden"], want["grad_hidden"]) <= GRAD_REL_L2
    idx = inp["topk_idx"].numpy()
    rng = np.random.default_rng(0)
    V = base.V
    vrows = np.unique(np.concatenate([idx[:8, 0], idx[100:104, 3], np.arange(V - 4, V),
                                      np.arange(V - 260, V - 256),
                                      rng.integers(0, V, size=24)]))
    err = rel_l2(got["grad_W"][vrows], want["grad_W"][vrows])
    assert err <= GRAD_REL_L2, err
    assert rel_l2(got["grad_W"], want["grad_W"]) <= GRAD_REL_L2
