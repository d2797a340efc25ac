"""Seeded random shapes against the float64 oracle (GPU).

Each case draws N, H, V, K, chunk and T at random (small enough for the
oracle to finish in well under a second), and one of the call's modes: the
default plan, the per-chunk grad_W plan, the stored-logits backward, a token
mask, accumulation into non-zero gradients, two token shards normalised by
the whole batch (the second adding into the first's grad_W).  The shapes land on every kind of
boundary the kernels have: chunks that are not multiples of the 256-row tile
(so a chunk's recompute and the next chunk's forward share tiles' row ranges
differently), odd chunk counts (a lone last chunk in its grad_W pair),
vocabularies and hidden sizes that end inside a tile or a k-block.
"""
import numpy as np
import pytest
import torch

import chunked_top_kl_gemm_b300 as kd
import oracle
import workloads
from tests.gpu_util import GRAD_REL_L2, LOSS_RTOL, ensure_lib, rel_l2, to_device

pytestmark = pytest.mark.gpu

MODES = ["default", "min_scratch", "store_logits", "masked", "accumulate", "sharded"]


def _case(i):
    rng = np.random.default_rng(1000 + i)
    N = int(rng.integers(1, 1500))
    H = int(rng.integers(1, 81)) * 8
    V = int(rng.integers(1, 626)) * 8
    K = int(rng.integers(1, min(V, 64) + 1))
    chunk = int(rng.integers(1, 700))
    T = float(np.round(rng.uniform(0.3, 3.0), 3))
    mode = MODES[i % len(MODES)]
    cfg = workloads.custom(f"rand{i}", N=N, H=H, V=V, K=K, T=T, chunk=chunk,
                           hidden_rms_norm=bool(i % 2), teacher="zipf" if i % 3 == 0 else "exp_gaps")
    return cfg, mode


@pytest.mark.parametrize("i", range(36))
def test_random_shape_against_oracle(i):
    ensure_lib()
    cfg, mode = _case(i)
    inp_cpu = workloads.make_inputs(cfg, seed=2000 + i)
    inp = to_device(inp_cpu)
    N, H, V, K = cfg.N, cfg.H, cfg.V, cfg.K
    mask_cpu = None
    flags = {"min_scratch": kd.KD_FLAG_MIN_SCRATCH, "store_logits": kd.KD_FLAG_STORE_LOGITS,
             "accumulate": kd.KD_FLAG_ACCUMULATE}.get(mode, 0)
    if mode == "masked":
        g = torch.Generator().manual_seed(i)
        mask_cpu = (torch.rand(N, generator=g) < 0.6).to(torch.uint8)
        mask_cpu[0] = 1
    g0 = torch.Generator(device="cuda").manual_seed(i)
    gh0 = torch.randn((N, H), generator=g0, device="cuda") * 1e-4 if mode == "accumulate" \
        else torch.zeros((N, H), device="cuda")
    gW0 = torch.randn((V, H), generator=g0, device="cuda") * 1e-4 if mode == "accumulate" \
        else torch.zeros((V, H), device="cuda")
    gh, gW = gh0.clone(), gW0.clone()
    if mode == "sharded":
        # a random cut; the shards' rows of grad_hidden start at zero (the
        # accumulate flag of the second shard adds into them too)
        cut = int(np.random.default_rng(i).integers(1, N)) if N > 1 else 1
        loss = 0.0
        for k, (r0, r1) in enumerate(((0, cut), (cut, N))):
            if r1 <= r0:
                continue
            f = kd.KD_FLAG_ACCUMULATE if r0 > 0 else 0
            ws = torch.empty(kd.kd_topk_kl_workspace_size_flags(r1 - r0, H, V, K, cfg.chunk, f),
                             dtype=torch.uint8, device="cuda")
            loss += kd.kd_topk_kl_fwd_bwd_sharded(
                inp["hidden"][r0:r1], inp["W"], inp["topk_idx"][r0:r1],
                inp["topk_logit"][r0:r1], None, cfg.T, cfg.chunk, f, N, gh[r0:r1], gW, ws)
    else:
        ws = torch.empty(kd.kd_topk_kl_workspace_size_flags(N, H, V, K, cfg.chunk, flags),
                         dtype=torch.uint8, device="cuda")
        loss = kd.kd_topk_kl_fwd_bwd_flags(inp["hidden"], inp["W"], inp["topk_idx"],
                                           inp["topk_logit"],
                                           None if mask_cpu is None else mask_cpu.cuda(), cfg.T,
                                           cfg.chunk, flags, gh, gW, ws)
    torch.cuda.synchronize()
    want = oracle.fused_topk_kl(inp_cpu["hidden"], inp_cpu["W"], inp_cpu["topk_idx"],
                                inp_cpu["topk_logit"], cfg.T, mask=mask_cpu)
    got_gh = (gh - gh0).cpu().numpy()
    got_gW = (gW - gW0).cpu().numpy()
    assert np.isfinite(got_gh).all() and np.isfinite(got_gW).all()
    assert abs(loss - want["loss"]) <= LOSS_RTOL * abs(want["loss"]) + 1e-6, (cfg, mode, loss)
    # accumulation subtracts the start values back out: compare what was added
    # with the tolerance of the plain call plus the start values' rounding
    tol = GRAD_REL_L2 if mode != "accumulate" else 2 * GRAD_REL_L2
    e1, e2 = rel_l2(got_gh, want["grad_hidden"]), rel_l2(got_gW, want["grad_W"])
    assert e1 <= tol and e2 <= tol, (cfg, mode, e1, e2)
