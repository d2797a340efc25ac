"""The store-logits backward (KD_FLAG_STORE_LOGITS) against the recompute path (GPU).

With the flag, the forward GEMM also writes each chunk's fp32 logits and
the backward forms dZ from them elementwise instead of recomputing the
GEMM.  The stored logits are the values the recompute produces and dZ is
rounded the same way, so loss and gradients must equal the recompute
path's bit for bit -- with and without a token mask, and when accumulating.
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
    "ragged": workloads.custom("z_ragged", N=300, H=200, V=1000, K=7, T=0.7, chunk=128),
    "mid": workloads.custom("z_mid", N=640, H=576, V=8192, K=100, T=1.0, chunk=256,
                            hidden_rms_norm=True, teacher="zipf"),
    "spiky_T2": workloads.custom("z_spiky", N=256, H=128, V=2048, K=32, T=2.0, chunk=128,
                                 hidden_rms_norm=True, teacher="zipf", spike_frac=0.1),
    "kv": workloads.custom("z_kv", N=130, H=72, V=136, K=136, T=1.5, chunk=128),
}


def _run(inp, T, chunk, flags, mask=None, gh=None, gW=None):
    h, W, idx, lg = inp["hidden"], inp["W"], inp["topk_idx"], inp["topk_logit"]
    N, H = h.shape
    V, K = W.shape[0], idx.shape[1]
    gh = torch.full((N, H), float("nan"), device="cuda") if gh is None else gh
    gW = torch.full((V, H), float("nan"), device="cuda") if gW is None else gW
    nbytes = kd.kd_topk_kl_workspace_size_flags(N, H, V, K, chunk, flags)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    loss = kd.kd_topk_kl_fwd_bwd_flags(h, W, idx, lg, mask, T, chunk, flags, gh, gW, ws)
    torch.cuda.synchronize()
    return loss, gh, gW


@pytest.mark.parametrize("name", list(CASES))
@pytest.mark.parametrize("masked", [False, True])
def test_store_logits_equals_recompute_bitwise(name, masked):
    ensure_lib()
    cfg = CASES[name]
    inp = to_device(workloads.make_inputs(cfg, seed=31))
    mask = None
    if masked:
        g = torch.Generator().manual_seed(7)
        mask = (torch.rand(cfg.N, generator=g) < 0.6).to(torch.uint8).cuda()
    a = _run(inp, cfg.T, cfg.chunk, 0, mask)
    b = _run(inp, cfg.T, cfg.chunk, kd.KD_FLAG_STORE_LOGITS, mask)
    assert a[0] == b[0]
    assert torch.equal(a[1], b[1]) and torch.equal(a[2], b[2])


def test_store_logits_with_accumulate_and_repeated_ids():
    ensure_lib()
    cfg = workloads.custom("z_dup", N=200, H=64, V=512, K=6, T=1.0, chunk=128)
    inp = workloads.make_inputs(cfg, seed=5)
    idx = inp["topk_idx"].clone()
    idx[::3, 1] = idx[::3, 0]            # repeated ids: the masses subtract one by one
    inp["topk_idx"] = idx
    inp = to_device(inp)
    g = torch.Generator(device="cuda").manual_seed(2)
    gh0 = torch.randn((cfg.N, cfg.H), generator=g, device="cuda") * 1e-3
    gW0 = torch.randn((cfg.V, cfg.H), generator=g, device="cuda") * 1e-3
    acc = kd.KD_FLAG_ACCUMULATE
    a = _run(inp, cfg.T, cfg.chunk, acc, gh=gh0.clone(), gW=gW0.clone())
    b = _run(inp, cfg.T, cfg.chunk, acc | kd.KD_FLAG_STORE_LOGITS, gh=gh0.clone(),
             gW=gW0.clone())
    assert a[0] == b[0] and torch.equal(a[1], b[1]) and torch.equal(a[2], b[2])
    want = oracle.fused_topk_kl(inp["hidden"].cpu(), inp["W"].cpu(), idx, inp["topk_logit"].cpu(),
                                cfg.T)
    assert abs(b[0] - want["loss"]) <= LOSS_RTOL * abs(want["loss"])
    assert rel_l2((b[2] - gW0).cpu().numpy(), want["grad_W"]) <= GRAD_REL_L2


def test_store_logits_full_vocabulary_two_chunks():
    """Two 2048-row chunks of the GPT-OSS-like head (V = 201,088): the same
    launch shapes as the benchmark's store-logits mode."""
    ensure_lib()
    cfg = workloads.CONFIGS["gptoss32k"]
    inp = workloads.make_inputs(cfg, seed=3, device="cuda", n_rows=4096)
    a = _run(inp, cfg.T, cfg.chunk, 0)
    b = _run(inp, cfg.T, cfg.chunk, kd.KD_FLAG_STORE_LOGITS)
    assert a[0] == b[0]
    assert torch.equal(a[1], b[1]) and torch.equal(a[2], b[2])


def test_chunk_of_more_than_65535_rows():
    """One 70,016-row chunk: the elementwise dZ kernel covers more rows than a
    grid's y dimension could hold.  Equal to the recompute, and to the oracle
    on sampled tokens."""
    ensure_lib()
    cfg = workloads.custom("z_big", N=70000, H=64, V=512, K=8, T=1.0, chunk=70000)
    inp_cpu = workloads.make_inputs(cfg, seed=13)
    inp = to_device(inp_cpu)
    a = _run(inp, cfg.T, cfg.chunk, 0)
    b = _run(inp, cfg.T, cfg.chunk, kd.KD_FLAG_STORE_LOGITS)
    assert a[0] == b[0]
    assert torch.equal(a[1], b[1]) and torch.equal(a[2], b[2])
    rows = np.array([0, 1, 65534, 65535, 65536, 69998, 69999])
    want = oracle.rows_forward(inp_cpu["hidden"][rows], inp_cpu["W"], inp_cpu["topk_idx"][rows],
                               inp_cpu["topk_logit"][rows], cfg.T, N_total=cfg.N)
    assert rel_l2(b[1].cpu().numpy()[rows], want["grad_hidden"]) <= GRAD_REL_L2


def test_full_logits_grid_past_int32_elements():
    """One chunk of all N tokens with stored logits holds the whole [N, V]
    grid: 12,288 x 200,704 = 2.47e9 elements, past what a 32-bit element
    offset reaches.  Bitwise equal to the recompute at the same chunk; the
    loss bitwise equal to the 2048-row chunked plan (its per-token terms do
    not depend on the chunking) and the gradients equal up to fp32
    summation order; grad_hidden rows against the oracle."""
    ensure_lib()
    cfg = workloads.custom("z_grid", N=12288, H=64, V=200704, K=16, T=1.0, chunk=12288,
                           hidden_rms_norm=True, teacher="zipf")
    assert cfg.N * cfg.V > 2**31
    inp_cpu = workloads.make_inputs(cfg, seed=17)
    inp = to_device(inp_cpu)
    b = _run(inp, cfg.T, cfg.N, kd.KD_FLAG_STORE_LOGITS)
    a = _run(inp, cfg.T, cfg.N, 0)
    assert a[0] == b[0]
    assert torch.equal(a[1], b[1]) and torch.equal(a[2], b[2])
    del a
    c = _run(inp, cfg.T, 2048, 0)
    assert c[0] == b[0]
    assert rel_l2(b[1].cpu().numpy(), c[1].cpu().numpy()) <= 1e-4
    assert rel_l2(b[2].cpu().numpy(), c[2].cpu().numpy()) <= 1e-4
    rows = np.array([0, 1, 6143, 6144, 10922, 12286, 12287])
    want = oracle.rows_forward(inp_cpu["hidden"][rows], inp_cpu["W"], inp_cpu["topk_idx"][rows],
                               inp_cpu["topk_logit"][rows], cfg.T, N_total=cfg.N)
    assert rel_l2(b[1].cpu().numpy()[rows], want["grad_hidden"]) <= GRAD_REL_L2


def test_workspace_grows_by_the_chunk_logits():
    ensure_lib()
    N, H, V, K, chunk = 32768, 2880, 201088, 100, 2048
    base = kd.kd_topk_kl_workspace_size_flags(N, H, V, K, chunk, 0)
    assert base == kd.kd_topk_kl_workspace_size(N, H, V, K, chunk)
    stored = kd.kd_topk_kl_workspace_size_flags(N, H, V, K, chunk, kd.KD_FLAG_STORE_LOGITS)
    assert 4 * chunk * V <= stored - base < 4 * chunk * V + 512
    assert kd.kd_topk_kl_workspace_size_flags(N, H, V, K, chunk, 8) == 0
