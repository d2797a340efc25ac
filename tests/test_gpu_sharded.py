"""Shards of a batch normalised by the whole batch (GPU).

``kd_topk_kl_fwd_bwd_sharded`` scales a shard's loss and gradients by the
batch's token count, so that shards add up: the losses sum to the batch
loss, the grad_W shares sum to the batch's grad_W (accumulated here on one
device, as a micro-batched step would; a data-parallel step would all-reduce
them), and each shard's grad_hidden rows are final.  Checked against the
single call on the whole batch and against the oracle.
"""
import numpy as np
import pytest
import torch

import chunked_top_kl_gemm_b300 as kd
import oracle
import workloads
from tests.gpu_util import GRAD_REL_L2, LOSS_RTOL, ensure_lib, rel_l2, to_device

pytestmark = pytest.mark.gpu

CFG = workloads.custom("shard", N=700, H=136, V=1032, K=9, T=1.3, chunk=128)
SHARDS = [(0, 250), (250, 600), (600, 700)]


def _ws(N, H, V, K, chunk, flags=0):
    return torch.empty(kd.kd_topk_kl_workspace_size_flags(N, H, V, K, chunk, flags),
                       dtype=torch.uint8, device="cuda")


def _run_shards(inp, mask, n_norm, extra=0):
    N, H = inp["hidden"].shape
    V, K = inp["W"].shape[0], inp["topk_idx"].shape[1]
    # the first shard overwrites grad_W, the others add to it; KD_FLAG_ACCUMULATE
    # also adds into grad_hidden, whose rows differ per shard: start at zero
    gh = torch.zeros((N, H), dtype=torch.float32, device="cuda")
    gW = torch.full((V, H), float("nan"), dtype=torch.float32, device="cuda")
    total = 0.0
    for i, (r0, r1) in enumerate(SHARDS):
        flags = (kd.KD_FLAG_ACCUMULATE if i > 0 else 0) | extra
        ws = _ws(r1 - r0, H, V, K, CFG.chunk, flags)
        m = None if mask is None else mask[r0:r1]
        total += kd.kd_topk_kl_fwd_bwd_sharded(
            inp["hidden"][r0:r1], inp["W"], inp["topk_idx"][r0:r1], inp["topk_logit"][r0:r1], m,
            CFG.T, CFG.chunk, flags, n_norm, gh[r0:r1], gW, ws)
    torch.cuda.synchronize()
    return total, gh.cpu().numpy(), gW.cpu().numpy()


def _run_whole(inp, mask, extra=0):
    N, H = inp["hidden"].shape
    V, K = inp["W"].shape[0], inp["topk_idx"].shape[1]
    gh = torch.empty((N, H), dtype=torch.float32, device="cuda")
    gW = torch.empty((V, H), dtype=torch.float32, device="cuda")
    loss = kd.kd_topk_kl_fwd_bwd_flags(inp["hidden"], inp["W"], inp["topk_idx"],
                                       inp["topk_logit"], mask, CFG.T, CFG.chunk, extra, gh, gW,
                                       _ws(N, H, V, K, CFG.chunk, extra))
    torch.cuda.synchronize()
    return loss, gh.cpu().numpy(), gW.cpu().numpy()


@pytest.mark.parametrize("masked", [False, True])
def test_shards_add_up_to_the_batch(masked):
    ensure_lib()
    inp_cpu = workloads.make_inputs(CFG, seed=17)
    inp = to_device(inp_cpu)
    mask_cpu = None
    if masked:
        g = torch.Generator().manual_seed(3)
        mask_cpu = (torch.rand(CFG.N, generator=g) < 0.7).to(torch.uint8)
    mask = None if mask_cpu is None else mask_cpu.cuda()
    n_norm = CFG.N if mask_cpu is None else int(mask_cpu.sum())
    loss, gh, gW = _run_shards(inp, mask, n_norm)
    ref_loss, ref_gh, ref_gW = _run_whole(inp, mask)
    assert abs(loss - ref_loss) <= 1e-6 * abs(ref_loss), (loss, ref_loss)
    assert rel_l2(gh, ref_gh) <= 1e-6
    assert rel_l2(gW, ref_gW) <= 1e-5
    want = oracle.fused_topk_kl(inp_cpu["hidden"], inp_cpu["W"], inp_cpu["topk_idx"],
                                inp_cpu["topk_logit"], CFG.T, mask=mask_cpu)
    assert abs(loss - want["loss"]) <= LOSS_RTOL * abs(want["loss"])
    assert rel_l2(gh, want["grad_hidden"]) <= GRAD_REL_L2
    assert rel_l2(gW, want["grad_W"]) <= GRAD_REL_L2


def test_whole_batch_as_one_shard_is_the_plain_call():
    ensure_lib()
    inp = to_device(workloads.make_inputs(CFG, seed=18))
    N, H, V, K = CFG.N, CFG.H, CFG.V, CFG.K
    gh = torch.empty((N, H), dtype=torch.float32, device="cuda")
    gW = torch.empty((V, H), dtype=torch.float32, device="cuda")
    loss = kd.kd_topk_kl_fwd_bwd_sharded(inp["hidden"], inp["W"], inp["topk_idx"],
                                         inp["topk_logit"], None, CFG.T, CFG.chunk, 0, N, gh, gW,
                                         _ws(N, H, V, K, CFG.chunk))
    torch.cuda.synchronize()
    ref_loss, ref_gh, ref_gW = _run_whole(inp, None)
    assert loss == ref_loss
    assert np.array_equal(gh.cpu().numpy(), ref_gh)
    assert np.array_equal(gW.cpu().numpy(), ref_gW)


def test_normaliser_below_one_is_rejected():
    ensure_lib()
    inp = to_device(workloads.make_inputs(CFG, seed=19))
    N, H, V, K = CFG.N, CFG.H, CFG.V, CFG.K
    gh = torch.empty((N, H), dtype=torch.float32, device="cuda")
    gW = torch.empty((V, H), dtype=torch.float32, device="cuda")
    with pytest.raises(kd.KdError) as ei:
        kd.kd_topk_kl_fwd_bwd_sharded(inp["hidden"], inp["W"], inp["topk_idx"],
                                      inp["topk_logit"], None, CFG.T, CFG.chunk, 0, 0, gh, gW,
                                      _ws(N, H, V, K, CFG.chunk))
    assert ei.value.name == "KD_ERR_INVALID_ARG"


@pytest.mark.parametrize("extra", ["store_logits", "min_scratch"])
def test_shards_add_up_with_other_flags(extra):
    # the stored-logits backward and the per-chunk grad_W form take the same
    # normaliser
    ensure_lib()
    flag = {"store_logits": kd.KD_FLAG_STORE_LOGITS, "min_scratch": kd.KD_FLAG_MIN_SCRATCH}[extra]
    inp = to_device(workloads.make_inputs(CFG, seed=20))
    loss, gh, gW = _run_shards(inp, None, CFG.N, extra=flag)
    ref_loss, ref_gh, ref_gW = _run_whole(inp, None, extra=flag)
    assert abs(loss - ref_loss) <= 1e-6 * abs(ref_loss), (loss, ref_loss)
    assert rel_l2(gh, ref_gh) <= 1e-6
    assert rel_l2(gW, ref_gW) <= 1e-5
