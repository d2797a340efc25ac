"""The masked / accumulating entry point against the float64 oracle (GPU).

``kd_topk_kl_fwd_bwd_masked`` takes a per-token mask (the mean runs over the
valid tokens, masked tokens get zero gradient rows) and an accumulate flag
(gradients are added into the given tensors).  Cases span several chunks
with ragged tails, so masked rows fall in every chunk and tile position.
"""
import numpy as np
import pytest
import torch

import chunked_top_kl_gemm_b300 as kd
import oracle
import workloads
from tests.gpu_util import GRAD_REL_L2, LOSS_RTOL, ensure_lib, rel_l2, to_device

pytestmark = pytest.mark.gpu

CASES = {
    "ragged": workloads.custom("m_ragged", N=300, H=200, V=1000, K=7, T=0.7, chunk=128),
    "mid": workloads.custom("m_mid", N=640, H=576, V=8192, K=100, T=1.0, chunk=256,
                            hidden_rms_norm=True, teacher="zipf"),
    "spiky_T2": workloads.custom("m_spiky", N=256, H=128, V=2048, K=32, T=2.0, chunk=128,
                                 hidden_rms_norm=True, teacher="zipf", spike_frac=0.1),
}


def _mask(N, frac, seed):
    g = torch.Generator().manual_seed(seed)
    m = (torch.rand(N, generator=g) < frac).to(torch.uint8)
    return m


def _run(inp, mask, T, chunk, gh=None, gW=None, accumulate=False):
    h, W, idx, lg = inp["hidden"], inp["W"], inp["topk_idx"], inp["topk_logit"]
    N, H = h.shape
    V, K = W.shape[0], idx.shape[1]
    if gh is None:
        gh = torch.full((N, H), float("nan"), dtype=torch.float32, device="cuda")
    if gW is None:
        gW = torch.full((V, H), float("nan"), dtype=torch.float32, device="cuda")
    ws = kd.alloc_workspace(N, H, V, K, chunk, device="cuda")
    loss = kd.kd_topk_kl_fwd_bwd_masked(h, W, idx, lg, mask, T, chunk, gh, gW, ws,
                                        accumulate=accumulate)
    torch.cuda.synchronize()
    return loss, gh, gW


@pytest.mark.parametrize("name", list(CASES))
@pytest.mark.parametrize("frac", [0.7, 0.05])
def test_masked_parity_with_oracle(name, frac):
    ensure_lib()
    cfg = CASES[name]
    inp = workloads.make_inputs(cfg, seed=21)
    mask = _mask(cfg.N, frac, seed=3)
    mask[0] = 1
    want = oracle.fused_topk_kl(inp["hidden"], inp["W"], inp["topk_idx"], inp["topk_logit"],
                                cfg.T, mask=mask.numpy())
    loss, gh, gW = _run(to_device(inp), mask.cuda(), cfg.T, cfg.chunk)
    assert abs(loss - want["loss"]) <= LOSS_RTOL * abs(want["loss"]), (loss, want["loss"])
    gh = gh.cpu().numpy()
    keep = mask.numpy() != 0
    assert np.all(gh[~keep] == 0.0)
    assert rel_l2(gh, want["grad_hidden"]) <= GRAD_REL_L2
    assert rel_l2(gW.cpu().numpy(), want["grad_W"]) <= GRAD_REL_L2


def test_all_ones_mask_equals_unmasked_call_bitwise():
    ensure_lib()
    cfg = CASES["ragged"]
    inp = to_device(workloads.make_inputs(cfg, seed=5))
    ref_loss, ref_gh, ref_gW = kd.fwd_bwd(inp["hidden"], inp["W"], inp["topk_idx"],
                                          inp["topk_logit"], cfg.T, cfg.chunk)
    ones = torch.ones(cfg.N, dtype=torch.uint8, device="cuda")
    loss, gh, gW = _run(inp, ones, cfg.T, cfg.chunk)
    assert loss == ref_loss
    assert torch.equal(gh, ref_gh) and torch.equal(gW, ref_gW)
    # a NULL mask through the masked entry point is the unmasked call too
    loss2, gh2, gW2 = _run(inp, None, cfg.T, cfg.chunk)
    assert loss2 == ref_loss and torch.equal(gh2, ref_gh) and torch.equal(gW2, ref_gW)


def test_no_valid_token_gives_zeros():
    ensure_lib()
    cfg = CASES["ragged"]
    inp = to_device(workloads.make_inputs(cfg, seed=6))
    zeros = torch.zeros(cfg.N, dtype=torch.uint8, device="cuda")
    loss, gh, gW = _run(inp, zeros, cfg.T, cfg.chunk)
    assert loss == 0.0
    assert int(torch.count_nonzero(gh)) == 0 and int(torch.count_nonzero(gW)) == 0


def test_accumulate_adds_into_the_gradients():
    ensure_lib()
    cfg = CASES["mid"]
    inp = to_device(workloads.make_inputs(cfg, seed=8))
    mask = _mask(cfg.N, 0.6, seed=4).cuda()
    loss_a, gh_a, gW_a = _run(inp, mask, cfg.T, cfg.chunk)
    g = torch.Generator(device="cuda").manual_seed(1)
    gh0 = torch.randn(gh_a.shape, generator=g, device="cuda") * 1e-4
    gW0 = torch.randn(gW_a.shape, generator=g, device="cuda") * 1e-4
    gh = gh0.clone()
    gW = gW0.clone()
    loss_b, gh, gW = _run(inp, mask, cfg.T, cfg.chunk, gh=gh, gW=gW, accumulate=True)
    assert loss_b == loss_a
    # grad_hidden rows are written once per call: old + new, exactly
    assert torch.equal(gh, gh0 + gh_a)
    # grad_W is reduce-added chunk by chunk on top of the old values
    assert rel_l2(gW.cpu().numpy(), (gW0 + gW_a).cpu().numpy()) <= 1e-5
    # two accumulating calls on zeros give twice one call
    gh2 = torch.zeros_like(gh)
    gW2 = torch.zeros_like(gW)
    for _ in range(2):
        _run(inp, mask, cfg.T, cfg.chunk, gh=gh2, gW=gW2, accumulate=True)
    assert torch.allclose(gh2, 2 * gh_a, rtol=1e-6, atol=0)
    assert rel_l2(gW2.cpu().numpy(), (2 * gW_a).cpu().numpy()) <= 1e-5


def test_python_wrapper_forwards_mask_and_accumulate():
    ensure_lib()
    cfg = CASES["spiky_T2"]
    inp = to_device(workloads.make_inputs(cfg, seed=9))
    mask = _mask(cfg.N, 0.5, seed=2).to(torch.bool).cuda()
    loss, gh, gW = kd.fwd_bwd(inp["hidden"], inp["W"], inp["topk_idx"], inp["topk_logit"],
                              cfg.T, cfg.chunk, token_mask=mask)
    torch.cuda.synchronize()
    want = oracle.fused_topk_kl(inp["hidden"].cpu(), inp["W"].cpu(), inp["topk_idx"].cpu(),
                                inp["topk_logit"].cpu(), cfg.T, mask=mask.cpu().numpy())
    assert abs(loss - want["loss"]) <= LOSS_RTOL * abs(want["loss"])
    with pytest.raises(ValueError):
        kd.fwd_bwd(inp["hidden"], inp["W"], inp["topk_idx"], inp["topk_logit"], cfg.T,
                   cfg.chunk, accumulate=True)
