"""CUDA path against the float64 oracle, element by element (small sizes).

Every case spans several tiles and ends in ragged tails: chunks that do not
divide N, vocabularies that are not multiples of the 256-wide vocab tile or
of the 128-row grad_W tile, hidden sizes that are not multiples of the 64
k-block or the 192-wide gradient tile.  Inputs come from ``workloads``
(seeded, CPU generator), the same bf16 values reach both sides.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests.gpu_util import assert_parity, ensure_lib, rel_l2, run_debug, to_device

pytestmark = pytest.mark.gpu


def _case(cfg, seed=0):
    ensure_lib()
    inp = workloads.make_inputs(cfg, seed=seed)
    want = oracle.fused_topk_kl(inp["hidden"], inp["W"], inp["topk_idx"],
                                inp["topk_logit"], cfg.T)
    got = run_debug(to_device(inp), cfg.T, cfg.chunk)
    return inp, got, want


CASES = {
    "tiny": workloads.CONFIGS["tiny"],
    # 3 chunks (last one 44 rows), V with a 232-wide last vocab tile and a
    # 104-row last grad_W tile, H with an 8-wide last k-block
    "ragged": workloads.custom("ragged", N=300, H=200, V=1000, K=7, T=0.7, chunk=128),
    # near-one-hot teachers (top logit +20 on 10% of tokens) at T = 2
    "spiky_T2": workloads.custom("spiky", N=256, H=128, V=2048, K=32, T=2.0, chunk=128,
                                 hidden_rms_norm=True, teacher="zipf", spike_frac=0.1),
    # K = 1: the loss is the cross-entropy of z/T at the cached id
    "k1": workloads.custom("k1", N=200, H=64, V=520, K=1, T=1.0, chunk=128),
    # K = V: every vocabulary column of every row is a hit
    "k_eq_v": workloads.custom("kv", N=130, H=72, V=136, K=136, T=1.5, chunk=128),
    # one token
    "n1": workloads.custom("n1", N=1, H=64, V=264, K=5, T=1.0, chunk=1),
    # larger head, several vocab and hidden tiles, chunk of 256 rows
    "mid": workloads.custom("mid", N=640, H=576, V=8192, K=100, T=1.0, chunk=256,
                            hidden_rms_norm=True, teacher="zipf"),
    # grad_W reduces over pairs of chunks: 4 chunks, the second pair's second
    # chunk ragged (50 rows); 5 chunks, the last (1 row) alone in its pair
    "pairs_ragged_second": workloads.custom("pr2", N=434, H=136, V=1032, K=9, T=1.0,
                                            chunk=128),
    "pairs_lone_last": workloads.custom("pr1", N=513, H=136, V=1032, K=9, T=0.8, chunk=128),
}


# Degenerate and extreme sizes: H below one 64-deep k-block, a vocabulary
# below one 256-wide tile (the pair multiplies 32 columns), teacher ids that
# cover half the vocabulary (about 128 hits per row and vocab tile), the
# largest K the library accepts, and extreme temperatures.
EDGE = {
    "h8_v8": workloads.custom("h8v8", N=33, H=8, V=8, K=3, T=1.0, chunk=128),
    "h24_v40_k_eq_v": workloads.custom("h24", N=200, H=24, V=40, K=40, T=0.5, chunk=64),
    "dense_hits": workloads.custom("dense", N=130, H=64, V=4096, K=2048, T=1.0, chunk=128),
    "k_max": workloads.custom("kmax", N=64, H=72, V=16384, K=8192, T=1.3, chunk=64),
    # temperature extremes: a sharp student softmax (z/T spans ~20) and a
    # nearly uniform one
    "cold_T0.1": workloads.custom("cold", N=300, H=256, V=4096, K=32, T=0.1, chunk=128,
                                  hidden_rms_norm=True, teacher="zipf"),
    "hot_T20": workloads.custom("hot", N=300, H=256, V=4096, K=32, T=20.0, chunk=128),
}
CASES.update(EDGE)


@pytest.mark.parametrize("name", list(CASES))
def test_parity(name):
    inp, got, want = _case(CASES[name])
    assert_parity(got, want, inp["topk_idx"].numpy())


def test_repeated_ids_scatter_add():
    cfg = workloads.custom("dup", N=160, H=64, V=512, K=6, T=1.0, chunk=128)
    ensure_lib()
    inp = workloads.make_inputs(cfg, seed=5)
    idx = inp["topk_idx"].clone()
    idx[::3, 1] = idx[::3, 0]            # every third row repeats its first id
    inp["topk_idx"] = idx
    want = oracle.fused_topk_kl(inp["hidden"], inp["W"], idx, inp["topk_logit"], cfg.T)
    got = run_debug(to_device(inp), cfg.T, cfg.chunk)
    assert abs(got["loss"] - want["loss"]) <= 1e-3 * abs(want["loss"])
    for key in ("grad_hidden", "grad_W"):
        assert rel_l2(got[key], want[key]) <= 2e-2, key
    assert np.array_equal(got["found"], idx.numpy())


def test_chunk_size_does_not_change_the_result():
    cfg = workloads.custom("chunks", N=520, H=136, V=1024, K=12, T=1.0, chunk=128)
    ensure_lib()
    inp = to_device(workloads.make_inputs(cfg, seed=7))
    outs = [run_debug(inp, cfg.T, c) for c in (1, 200, 256, 520, 4096)]
    for o in outs[1:]:
        assert abs(o["loss"] - outs[0]["loss"]) <= 1e-5 * abs(outs[0]["loss"])
        np.testing.assert_array_equal(o["found"], outs[0]["found"])
        np.testing.assert_allclose(o["lse"], outs[0]["lse"], rtol=0, atol=1e-5)
        np.testing.assert_allclose(o["grad_hidden"], outs[0]["grad_hidden"], rtol=0,
                                   atol=1e-6 * np.abs(outs[0]["grad_hidden"]).max())
        assert rel_l2(o["grad_W"], outs[0]["grad_W"]) < 1e-5


def test_bitwise_deterministic():
    cfg = CASES["ragged"]
    ensure_lib()
    inp = to_device(workloads.make_inputs(cfg, seed=1))
    a = run_debug(inp, cfg.T, cfg.chunk)
    b = run_debug(inp, cfg.T, cfg.chunk)
    assert a["loss"] == b["loss"]
    for key in ("grad_hidden", "grad_W", "lse", "zg"):
        assert np.array_equal(a[key], b[key]), key


def test_spec_entry_point_matches_debug_entry_point():
    import chunked_top_kl_gemm_b300 as kd
    cfg = CASES["tiny"]
    ensure_lib()
    inp = to_device(workloads.make_inputs(cfg, seed=2))
    ref = run_debug(inp, cfg.T, cfg.chunk)
    N, H, V = cfg.N, cfg.H, cfg.V
    gh = torch.empty((N, H), dtype=torch.float32, device="cuda")
    gW = torch.empty((V, H), dtype=torch.float32, device="cuda")
    torch.cuda.synchronize()
    loss = kd.kd_topk_kl_fwd_bwd(inp["hidden"], inp["W"], inp["topk_idx"], inp["topk_logit"],
                                 cfg.T, cfg.chunk, gh, gW)
    assert loss == ref["loss"]
    assert np.array_equal(gh.cpu().numpy(), ref["grad_hidden"])
    assert np.array_equal(gW.cpu().numpy(), ref["grad_W"])
    loss2, gh2, gW2 = kd.fwd_bwd(inp["hidden"], inp["W"], inp["topk_idx"], inp["topk_logit"],
                                 cfg.T, cfg.chunk)
    torch.cuda.synchronize()
    assert loss2 == ref["loss"]
    assert np.array_equal(gW2.cpu().numpy(), ref["grad_W"])


@pytest.mark.parametrize("name", ["ragged", "pairs_ragged_second", "pairs_lone_last", "mid"])
def test_grad_W_over_chunk_pairs_matches_per_chunk(name):
    # default plan: grad_W reduces over two chunks' dZ at once; with
    # KD_FLAG_MIN_SCRATCH it is formed per chunk.  The loss and grad_hidden
    # do not depend on that (bitwise equal), grad_W only through the fp32
    # accumulation order; both match the oracle.
    import chunked_top_kl_gemm_b300 as kd
    cfg = CASES[name]
    ensure_lib()
    inp_cpu = workloads.make_inputs(cfg, seed=9)
    inp = to_device(inp_cpu)
    N, H, V, K = cfg.N, cfg.H, cfg.V, cfg.K
    res = {}
    for flags in (0, kd.KD_FLAG_MIN_SCRATCH):
        ws = torch.empty(kd.kd_topk_kl_workspace_size_flags(N, H, V, K, cfg.chunk, flags),
                         dtype=torch.uint8, device="cuda")
        gh = torch.full((N, H), float("nan"), dtype=torch.float32, device="cuda")
        gW = torch.full((V, H), float("nan"), dtype=torch.float32, device="cuda")
        loss = kd.kd_topk_kl_fwd_bwd_flags(inp["hidden"], inp["W"], inp["topk_idx"],
                                           inp["topk_logit"], None, cfg.T, cfg.chunk, flags,
                                           gh, gW, ws)
        torch.cuda.synchronize()
        res[flags] = (loss, gh.cpu().numpy(), gW.cpu().numpy(), ws.numel())
    a, b = res[0], res[kd.KD_FLAG_MIN_SCRATCH]
    if -(-N // cfg.chunk) >= 2:
        assert a[3] > b[3]                      # two chunks' dZ instead of one
    assert a[0] == b[0]
    assert np.array_equal(a[1], b[1])
    assert rel_l2(a[2], b[2]) < 1e-5
    want = oracle.fused_topk_kl(inp_cpu["hidden"], inp_cpu["W"], inp_cpu["topk_idx"],
                                inp_cpu["topk_logit"], cfg.T)
    for r in (a, b):
        assert abs(r[0] - want["loss"]) <= 1e-3 * abs(want["loss"])
        assert rel_l2(r[1], want["grad_hidden"]) <= 2e-2
        assert rel_l2(r[2], want["grad_W"]) <= 2e-2
