"""The asynchronous entry point and CUDA-graph capture (GPU).

``kd_topk_kl_fwd_bwd_async`` enqueues the same launches as the blocking
entry points and leaves the loss and a status code in device memory, so a
training step can keep the host out of the loop or be captured in a CUDA
graph.  Checked here:

* it gives bit for bit the blocking call's loss and gradients (plain,
  masked, accumulating, stored logits, per-chunk grad_W, masked per-chunk);
* a captured graph replayed on new inputs written into the same buffers
  matches a blocking call on those inputs, and the float64 oracle;
* an accumulating masked graph replayed twice adds two steps' gradients;
* an out-of-range id shows up in the device status word, and the context
  stays usable;
* the per-kernel profiler does not time the asynchronous call.
"""
import numpy as np
import pytest
import torch

import chunked_top_kl_gemm_b300 as kd
import oracle
import workloads
from tests.gpu_util import GRAD_REL_L2, LOSS_RTOL, ensure_lib, rel_l2, to_device

pytestmark = pytest.mark.gpu

MID = workloads.custom("as_mid", N=640, H=576, V=8192, K=100, T=1.0, chunk=256,
                       hidden_rms_norm=True, teacher="zipf")
RAGGED = workloads.custom("as_ragged", N=300, H=200, V=1000, K=7, T=0.7, chunk=128)


def _bufs(cfg, flags=0, dev="cuda"):
    N, H, V, K = cfg.N, cfg.H, cfg.V, cfg.K
    return {
        "gh": torch.zeros((N, H), dtype=torch.float32, device=dev),
        "gW": torch.zeros((V, H), dtype=torch.float32, device=dev),
        "ws": torch.empty(kd.kd_topk_kl_workspace_size_flags(N, H, V, K, cfg.chunk, flags),
                          dtype=torch.uint8, device=dev),
        "loss": torch.full((1,), float("nan"), dtype=torch.float32, device=dev),
        "status": torch.full((1,), -1, dtype=torch.int32, device=dev),
    }


def _blocking(inp, cfg, mask, flags, b):
    return kd.kd_topk_kl_fwd_bwd_flags(inp["hidden"], inp["W"], inp["topk_idx"],
                                       inp["topk_logit"], mask, cfg.T, cfg.chunk, flags,
                                       b["gh"], b["gW"], b["ws"])


def _async(inp, cfg, mask, flags, b, stream=None):
    kd.kd_topk_kl_fwd_bwd_async(inp["hidden"], inp["W"], inp["topk_idx"], inp["topk_logit"],
                                mask, cfg.T, cfg.chunk, flags, b["loss"], b["status"],
                                b["gh"], b["gW"], b["ws"], stream=stream)


def _mask(N, frac, seed):
    g = torch.Generator().manual_seed(seed)
    m = (torch.rand(N, generator=g) < frac).to(torch.uint8)
    m[0] = 1
    return m.cuda()


@pytest.mark.parametrize("mode", ["plain", "masked", "accumulate", "store_logits", "min_scratch",
                                  "masked_min_scratch"])
@pytest.mark.parametrize("cfg", [MID, RAGGED], ids=["mid", "ragged"])
def test_async_equals_blocking_bitwise(cfg, mode):
    ensure_lib()
    inp = to_device(workloads.make_inputs(cfg, seed=31))
    mask = _mask(cfg.N, 0.6, seed=5) if mode.startswith("masked") else None
    flags = {"accumulate": kd.KD_FLAG_ACCUMULATE,
             "store_logits": kd.KD_FLAG_STORE_LOGITS,
             "min_scratch": kd.KD_FLAG_MIN_SCRATCH,
             "masked_min_scratch": kd.KD_FLAG_MIN_SCRATCH}.get(mode, 0)
    a, b = _bufs(cfg, flags), _bufs(cfg, flags)
    if mode == "accumulate":
        g = torch.Generator(device="cuda").manual_seed(2)
        for t in ("gh", "gW"):
            a[t].copy_(torch.randn(a[t].shape, generator=g, device="cuda") * 1e-4)
            b[t].copy_(a[t])
    want = _blocking(inp, cfg, mask, flags, a)
    _async(inp, cfg, mask, flags, b)
    torch.cuda.synchronize()
    assert int(b["status"].item()) == kd.KD_OK
    got = float(b["loss"].item())
    assert got == want, (got, want)
    assert torch.equal(b["gh"], a["gh"]) and torch.equal(b["gW"], a["gW"])


def _capture(fn):
    """Warm up on a side stream, then capture ``fn`` into a CUDA graph."""
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        fn()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        fn()
    return graph


def test_graph_replay_on_new_inputs_matches_blocking_and_oracle():
    ensure_lib()
    cfg = RAGGED
    static = to_device(workloads.make_inputs(cfg, seed=40))
    b = _bufs(cfg)
    graph = _capture(lambda: _async(static, cfg, None, 0, b))
    for seed in (41, 42, 43):
        fresh = workloads.make_inputs(cfg, seed=seed)
        for k in static:
            static[k].copy_(fresh[k])
        b["status"].fill_(-1)
        graph.replay()
        torch.cuda.synchronize()
        kd.check_status(b["status"])
        ref = _bufs(cfg)
        want = _blocking(static, cfg, None, 0, ref)
        assert float(b["loss"].item()) == want
        assert torch.equal(b["gh"], ref["gh"]) and torch.equal(b["gW"], ref["gW"])
        if seed == 41:
            o = oracle.fused_topk_kl(fresh["hidden"], fresh["W"], fresh["topk_idx"],
                                     fresh["topk_logit"], cfg.T)
            assert abs(want - o["loss"]) <= LOSS_RTOL * abs(o["loss"])
            assert rel_l2(b["gh"].cpu().numpy(), o["grad_hidden"]) <= GRAD_REL_L2
            assert rel_l2(b["gW"].cpu().numpy(), o["grad_W"]) <= GRAD_REL_L2


def test_graph_masked_accumulate_replayed_twice():
    ensure_lib()
    cfg = MID
    inp = to_device(workloads.make_inputs(cfg, seed=44))
    mask = _mask(cfg.N, 0.5, seed=6)
    flags = kd.KD_FLAG_ACCUMULATE
    one = _bufs(cfg, flags)
    loss1 = _blocking(inp, cfg, mask, flags, one)        # one step onto zeros
    b = _bufs(cfg, flags)
    graph = _capture(lambda: _async(inp, cfg, mask, flags, b))   # warm-up adds one step
    b["gh"].zero_()
    b["gW"].zero_()
    graph.replay()
    graph.replay()
    torch.cuda.synchronize()
    kd.check_status(b["status"])
    assert float(b["loss"].item()) == loss1
    assert torch.equal(b["gh"], 2 * one["gh"])           # x + x is exact
    assert rel_l2(b["gW"].cpu().numpy(), (2 * one["gW"]).cpu().numpy()) <= 1e-5
    keep = mask.cpu().numpy() != 0
    assert np.all(b["gh"].cpu().numpy()[~keep] == 0.0)


def test_out_of_range_id_sets_the_status_word():
    ensure_lib()
    cfg = RAGGED
    inp = to_device(workloads.make_inputs(cfg, seed=45))
    bad = {k: v.clone() for k, v in inp.items()}
    bad["topk_idx"][7, 3] = cfg.V
    b = _bufs(cfg)
    _async(bad, cfg, None, 0, b)                          # enqueues without error
    torch.cuda.synchronize()
    assert int(b["status"].item()) == kd.KD_ERR_INDEX
    with pytest.raises(kd.KdError):
        kd.check_status(b["status"])
    _async(inp, cfg, None, 0, b)                          # the context is still usable
    torch.cuda.synchronize()
    assert int(b["status"].item()) == kd.KD_OK


def test_profiler_skips_the_async_call():
    ensure_lib()
    cfg = RAGGED
    inp = to_device(workloads.make_inputs(cfg, seed=46))
    b = _bufs(cfg)
    kd.kd_profile_enable(True)
    try:
        before = kd.kd_profile_read()
        _async(inp, cfg, None, 0, b)
        torch.cuda.synchronize()
        after = kd.kd_profile_read()
        assert after == before
        _blocking(inp, cfg, None, 0, b)
        timed = kd.kd_profile_read()
        assert timed["gemm_fwd_lse_gather"][1] > before["gemm_fwd_lse_gather"][1]
    finally:
        kd.kd_profile_enable(False)
