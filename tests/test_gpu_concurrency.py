"""Concurrent calls (GPU): two streams, and several host threads.

Each call owns its workspace, its status word (inside the workspace) and its
output buffers; the library keeps no other state a call writes, apart from
per-device launch caches that every caller fills with the same values.  So
calls that overlap on the GPU (two streams) or in the host code (threads;
ctypes releases the GIL for the duration of a foreign call) must give bitwise
the results of the same calls run one after another.
"""
import threading

import pytest
import torch

import chunked_top_kl_gemm_b300 as kd
import workloads
from tests.gpu_util import ensure_lib, to_device

pytestmark = pytest.mark.gpu

CASES = [
    workloads.custom("cc_ragged", N=300, H=200, V=1000, K=7, T=0.7, chunk=128),
    workloads.custom("cc_mid", N=640, H=576, V=8192, K=100, T=1.0, chunk=256,
                     hidden_rms_norm=True, teacher="zipf"),
    workloads.custom("cc_pairs", N=513, H=136, V=1032, K=9, T=0.8, chunk=128),
]


def _problem(cfg, seed):
    inp = to_device(workloads.make_inputs(cfg, seed=seed))
    N, H, V, K = cfg.N, cfg.H, cfg.V, cfg.K
    return {
        "cfg": cfg, "inp": inp,
        "gh": torch.empty((N, H), dtype=torch.float32, device="cuda"),
        "gW": torch.empty((V, H), dtype=torch.float32, device="cuda"),
        "ws": kd.alloc_workspace(N, H, V, K, cfg.chunk, device="cuda"),
        "loss_out": torch.zeros(1, dtype=torch.float32, device="cuda"),
        "status_out": torch.zeros(1, dtype=torch.int32, device="cuda"),
    }


def _blocking(p, stream=None):
    i, c = p["inp"], p["cfg"]
    return kd.kd_topk_kl_fwd_bwd_ex(i["hidden"], i["W"], i["topk_idx"], i["topk_logit"], c.T,
                                    c.chunk, p["gh"], p["gW"], p["ws"], stream=stream)


def _enqueue(p, stream):
    i, c = p["inp"], p["cfg"]
    kd.kd_topk_kl_fwd_bwd_async(i["hidden"], i["W"], i["topk_idx"], i["topk_logit"], None, c.T,
                                c.chunk, 0, p["loss_out"], p["status_out"], p["gh"], p["gW"],
                                p["ws"], stream=stream)


def _reference(cfg, seed):
    p = _problem(cfg, seed)
    loss = _blocking(p)
    torch.cuda.synchronize()
    return loss, p["gh"].clone(), p["gW"].clone()


def test_calls_on_two_streams_equal_sequential_calls():
    ensure_lib()
    refs = [_reference(c, 40 + k) for k, c in enumerate(CASES[:2])]
    probs = [_problem(c, 40 + k) for k, c in enumerate(CASES[:2])]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    torch.cuda.synchronize()
    for _ in range(2):                       # twice: the second pair overlaps the first's tail
        for p, s in zip(probs, streams):
            _enqueue(p, s)
    torch.cuda.synchronize()
    for p, (loss, gh, gW) in zip(probs, refs):
        assert int(p["status_out"].item()) == kd.KD_OK
        assert float(p["loss_out"].item()) == loss
        assert torch.equal(p["gh"], gh) and torch.equal(p["gW"], gW)


def test_calls_from_several_host_threads_equal_sequential_calls():
    ensure_lib()
    jobs = [(CASES[k % len(CASES)], 60 + k) for k in range(6)]
    refs = [_reference(c, s) for c, s in jobs]
    probs = [_problem(c, s) for c, s in jobs]
    streams = [torch.cuda.Stream() for _ in jobs]
    torch.cuda.synchronize()
    losses = [None] * len(jobs)
    errors = []
    start = threading.Barrier(len(jobs))

    def work(k):
        try:
            start.wait()
            with torch.cuda.stream(streams[k]):
                for _ in range(3):
                    losses[k] = _blocking(probs[k], stream=streams[k])
        except Exception as e:  # reported below, in the main thread
            errors.append(e)

    threads = [threading.Thread(target=work, args=(k,)) for k in range(len(jobs))]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=300)
    assert not any(t.is_alive() for t in threads)
    assert not errors, errors
    torch.cuda.synchronize()
    for k, (loss, gh, gW) in enumerate(refs):
        assert losses[k] == loss
        assert torch.equal(probs[k]["gh"], gh) and torch.equal(probs[k]["gW"], gW)
